"""The C ABI without a GPU: the library loads, exports every symbol the public
header declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest
import torch

import swiglu_gemm_transformer_gb300 as sg
from swiglu_gemm_transformer_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "swiglu.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return sg.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(swiglu_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for must in ("swiglu_fused", "swiglu_fused_interleaved", "swiglu_pack_interleaved",
                 "swiglu_device_status", "swiglu_status_string"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), f"{name} declared in swiglu.h but not exported"
        assert name in sg.EXPORTS, f"{name} has no binding in the Python package"


def test_status_and_variant_strings(lib):
    assert sg.status_string(sg.OK) == "ok"
    assert "timed out" in sg.status_string(sg.ERR_TIMEOUT)
    assert sg.variant_name(sg.VARIANT_1SM_N128) == "1sm_n128"
    assert sg.variant_name(sg.VARIANT_2SM_N128) == "2sm_n128"
    assert sg.variant_name(99) == "?"


def test_host_side_variant_choice(lib):
    # 0.5B shape, M <= 128: 76 tiles of 64 columns, two CTAs each along K, fill 152 SMs
    assert lib.swiglu_select_variant(64, 4864, 896, 0) == sg.VARIANT_1SM_N64_SK2
    assert lib.swiglu_select_variant(128, 4864, 896, 1) == sg.VARIANT_1SM_N64_SK2
    # M = 256: 2 x 76 one-CTA tiles of 64 columns are one wave
    assert lib.swiglu_select_variant(256, 4864, 896, 0) == sg.VARIANT_1SM_N64
    # 7B shape, M = 128: 148 column blocks of 128 nearly fill 152 SMs
    assert lib.swiglu_select_variant(128, 18944, 3584, 0) == sg.VARIANT_1SM_N128
    assert lib.swiglu_select_variant(8192, 4864, 896, 0) == sg.VARIANT_2SM_N128


def test_host_side_weight_kernel_choice(lib):
    # no GPU here: planning assumes GB300's 152 SMs
    # 0.5B, M <= 128: 76 column blocks of 64, split along K over CTA pairs
    assert lib.swiglu_select_weight_kernel(64, 4864) == 0
    assert lib.swiglu_select_weight_kernel(128, 4864) == 0
    # 7B, M = 128: too many 64-column tiles for one wave -> the wide kernel
    assert lib.swiglu_select_weight_kernel(128, 18944) == 1
    # M > 128: two row blocks per CTA when that grid still fills a wave
    assert lib.swiglu_select_weight_kernel(256, 18944) == 2   # 1 x 148 CTAs
    assert lib.swiglu_select_weight_kernel(2048, 4864) == 2   # 8 x 38 CTAs
    # ... else one (0.5B M = 512: 2 x 38 two-block CTAs would idle half the GPU)
    assert lib.swiglu_select_weight_kernel(512, 4864) == 1
    assert lib.swiglu_select_weight_kernel(129, 64) == 1
    assert lib.swiglu_select_weight_kernel(-1, 64) == -1
    assert sg.WEIGHT_KERNELS[lib.swiglu_select_weight_kernel(256, 18944)] == "wide_mb2"


# Fake, never-dereferenced device addresses: validation is pure host arithmetic.
A_, W1_, W2_, Y_ = 0x10000000, 0x20000000, 0x30000000, 0x40000000


@pytest.mark.parametrize("args,want", [
    ((A_, W1_, W2_, Y_, -1, 64, 64), sg.ERR_INVALID_ARG),
    ((A_, W1_, W2_, Y_, 64, -8, 64), sg.ERR_INVALID_ARG),
    ((A_, W1_, W2_, None, 64, 64, 64), sg.ERR_INVALID_ARG),
    ((None, W1_, W2_, Y_, 64, 64, 64), sg.ERR_INVALID_ARG),
    ((A_, None, W2_, Y_, 64, 64, 64), sg.ERR_INVALID_ARG),
    ((A_, W1_, None, Y_, 64, 64, 64), sg.ERR_INVALID_ARG),
    ((A_ + 8, W1_, W2_, Y_, 64, 64, 64), sg.ERR_MISALIGNED),
    ((A_, W1_, W2_, Y_ + 2, 64, 64, 64), sg.ERR_MISALIGNED),
    ((A_, W1_, W2_, Y_, 64, 60, 64), sg.ERR_MISALIGNED),      # row pitch 120 B
    ((A_, W1_, W2_, Y_, 64, 64, 36), sg.ERR_MISALIGNED),
    ((A_, W1_, W2_, A_ + 64, 64, 64, 64), sg.ERR_INVALID_ARG),  # Y overlaps A
    ((A_, W1_, W2_, W2_, 64, 64, 64), sg.ERR_INVALID_ARG),      # Y overlaps W2
    ((A_, W1_, W2_, Y_, 1 << 31, 64, 64), sg.ERR_UNSUPPORTED),
    ((A_, W1_, W2_, Y_, 0, 64, 64), sg.OK),                     # empty: nothing to do
    ((A_, W1_, W2_, Y_, 64, 0, 64), sg.OK),
])
def test_fused_argument_validation(lib, args, want):
    assert lib.swiglu_fused(*args, None) == want


def test_bad_variant_rejected(lib):
    assert lib.swiglu_fused_ex(A_, W1_, W2_, Y_, 64, 64, 64, 77, None) == sg.ERR_INVALID_ARG
    assert lib.swiglu_fused_interleaved_ex(A_, W1_, Y_, 64, 64, 64, -1, None) == sg.ERR_INVALID_ARG
    # the swapped-operand kernel takes at most 128 rows
    assert lib.swiglu_fused_ex(A_, W1_, W2_, Y_, 129, 64, 64, sg.VARIANT_2SM_SWAP, None) == sg.ERR_UNSUPPORTED
    for retired in (5, 6, 7, 8):   # numbers of withdrawn variants stay unused
        assert lib.swiglu_fused_ex(A_, W1_, W2_, Y_, 64, 64, 64, retired, None) == sg.ERR_INVALID_ARG
        assert lib.swiglu_fused_interleaved_ex(A_, W1_, Y_, 64, 64, 64, retired, None) == sg.ERR_INVALID_ARG
        assert sg.variant_name(retired) == "?"


def test_interleaved_and_pack_validation(lib):
    assert lib.swiglu_fused_interleaved(A_, None, Y_, 64, 64, 64, None) == sg.ERR_INVALID_ARG
    assert lib.swiglu_fused_interleaved(A_, W1_, W1_ + 16, 64, 64, 64, None) == sg.ERR_INVALID_ARG
    assert lib.swiglu_pack_interleaved(W1_, W2_, None, 64, 64, None) == sg.ERR_INVALID_ARG
    assert lib.swiglu_pack_interleaved(W1_, W2_, Y_ + 4, 64, 64, None) == sg.ERR_MISALIGNED
    assert lib.swiglu_pack_interleaved(W1_, W2_, Y_, 64, 12, None) == sg.ERR_MISALIGNED
    assert lib.swiglu_pack_interleaved(W1_, W2_, W1_, 64, 64, None) == sg.ERR_INVALID_ARG
    assert lib.swiglu_pack_interleaved(W1_, W2_, Y_, 0, 64, None) == sg.OK


def test_pair_schedule_setter_validates(lib):
    assert lib.swiglu_set_pair_schedule(2) == sg.ERR_INVALID_ARG
    assert lib.swiglu_set_pair_schedule(-1) == sg.ERR_INVALID_ARG
    assert lib.swiglu_set_pair_schedule(0) == sg.OK
    assert lib.swiglu_set_pair_schedule(1) == sg.OK


def test_timeout_setters_validate(lib):
    assert lib.swiglu_set_wait_timeout_ns(10) == sg.ERR_INVALID_ARG
    assert lib.swiglu_set_wait_timeout_ns(2_000_000_000) == sg.OK
    assert lib.swiglu_selftest_wait_timeout(0, None) == sg.ERR_INVALID_ARG
    assert lib.swiglu_selftest_wait_timeout(2_000_000, None) == sg.ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_call_without_a_device_reports_cuda_error(lib):
    rc = lib.swiglu_fused(A_, W1_, W2_, Y_, 64, 64, 64, None)
    assert rc in (sg.ERR_CUDA, sg.ERR_UNSUPPORTED)
    detail = ctypes.c_uint32(7)
    assert lib.swiglu_device_status(None, ctypes.byref(detail)) in (sg.ERR_CUDA, sg.ERR_UNSUPPORTED)
    assert detail.value == 0


def test_python_binding_refuses_cpu_tensors(lib):
    A = torch.zeros(8, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        sg.swiglu_fused(A, A, A)


def test_fp8_argument_validation(lib):
    s = 0x50000000
    assert lib.swiglu_fused_fp8(A_, W1_, W2_, None, s, s, Y_, 64, 64, 64, None) == sg.ERR_INVALID_ARG
    assert lib.swiglu_fused_fp8(A_, W1_, W2_, s, s, s, Y_, 64, 64, 40, None) == sg.ERR_MISALIGNED
    assert lib.swiglu_fused_fp8(A_, W1_, W2_, s + 2, s, s, Y_, 64, 64, 64, None) == sg.ERR_MISALIGNED
    assert lib.swiglu_fused_fp8(A_, W1_, W2_, s, s, s, A_, 64, 64, 64, None) == sg.ERR_INVALID_ARG
    assert lib.swiglu_fused_fp8(A_, W1_, W2_, s, s, s, Y_, 0, 64, 64, None) == sg.OK
    assert lib.swiglu_fused_interleaved_fp8(A_, None, s, s, s, Y_, 64, 64, 64, None) == sg.ERR_INVALID_ARG
    assert lib.swiglu_pack_interleaved_fp8(W1_, W2_, Y_, 64, 24, None) == sg.ERR_MISALIGNED
    assert lib.swiglu_pack_interleaved_fp8(W1_, W2_, W1_, 64, 64, None) == sg.ERR_INVALID_ARG
    assert lib.swiglu_pack_interleaved_fp8(W1_, W2_, Y_, 0, 64, None) == sg.OK


def test_linear_and_mlp_validation(lib):
    ws = 0x60000000
    assert lib.swiglu_linear(A_, W1_, None, Y_, -1, 64, 64, None, 0, None) == sg.ERR_INVALID_ARG
    assert lib.swiglu_linear(A_, W1_, None, Y_, 64, 60, 64, None, 0, None) == sg.ERR_MISALIGNED
    assert lib.swiglu_linear(A_, W1_, None, A_ + 32, 64, 64, 64, None, 0, None) == sg.ERR_INVALID_ARG
    assert lib.swiglu_linear(A_, W1_, Y_ + 64, Y_, 64, 64, 64, None, 0, None) == sg.ERR_INVALID_ARG
    assert lib.swiglu_linear(A_, W1_, None, Y_, 0, 64, 64, None, 0, None) == sg.OK
    assert lib.swiglu_mlp(A_, W1_, W2_, W1_, None, Y_, 64, 64, 64, None, 0, None) == sg.ERR_INVALID_ARG
    assert lib.swiglu_mlp(A_, W1_, W2_, W1_, None, Y_, 64, 64, 64, ws, 100, None) == sg.ERR_INVALID_ARG
    assert lib.swiglu_mlp(A_, W1_, W2_, W1_, None, Y_, 64, 64, 64, Y_, 1 << 20, None) == sg.ERR_INVALID_ARG


def test_workspace_sizes(lib):
    # 0.5B down projection, M = 128: 14 tiles of 128 x 64, split K over clusters of
    # 8 CTAs whose partial sums meet in distributed shared memory: no workspace
    assert lib.swiglu_linear_workspace_size(128, 896, 4864) == 0
    assert lib.swiglu_mlp_workspace_size(128, 896, 4864) == 128 * 4864 * 2
    # 7B, M = 512: 112 tiles of 128 x 128 do not fit clusters in one wave ->
    # CTA pairs, K split into slices whose FP32 partial sums go to the workspace
    n = lib.swiglu_linear_workspace_size(512, 3584, 18944)
    assert n > 0 and n % (512 * 3584 * 4) == 0
    assert lib.swiglu_mlp_workspace_size(512, 3584, 18944) == 512 * 18944 * 2 + n
    assert lib.swiglu_linear_workspace_size(8192, 896, 4864) == 0      # enough tiles: no split
    assert lib.swiglu_linear_workspace_size(0, 896, 4864) == 0
