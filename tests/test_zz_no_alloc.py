"""The no-allocation MLP entry point, for callers that cannot allocate device
memory (a plugin handed only its tensors, a runtime whose memory is planned
before it runs).

swiglu_mlp_noalloc keeps Y in a fixed scratch area inside the library instead
of a caller-provided workspace.  Called through the C ABI on two calls in a
row with different shapes and data (the scratch area keeps the previous
call's contents), its result must meet the MLP block's acceptance rule
against the oracle's MLP block (the rule of the other MLP tests, with the
per-element slack for BF16 rounding of the intermediate Y), and must match
that of swiglu_mlp (the existing entry point, given a workspace that torch
allocates) within the same rule.  A size whose Y does not fit must be
rejected.

The file name makes pytest collect it last, so that a run stopping at the
first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import oracle
import swiglu_inputs as si

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def sg():
    import __graft_entry__
    __graft_entry__.build()
    import swiglu_gemm_transformer_gb300 as m
    m.lib()
    return m


def _case(M, H, F, seed, with_r):
    A, W1, W2 = si.make_bf16(M, F, H, seed)
    W3 = si.make_bf16(1, H, F, seed + 100)[1]
    R = None
    if with_r:
        R = torch.randn(M, H, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
    return (A, W1, W2, W3, R)


def _noalloc_c_abi(sg, A, W1, W2, W3, R):
    M, H = A.shape
    F = W1.shape[1]
    Z = torch.empty(M, H, dtype=torch.bfloat16, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = sg.lib().swiglu_mlp_noalloc(A.data_ptr(), W1.data_ptr(), W2.data_ptr(), W3.data_ptr(),
                                     R.data_ptr() if R is not None else None, Z.data_ptr(),
                                     M, H, F, stream)
    assert rc == sg.OK, sg.status_string(rc)
    return Z


def test_noalloc_matches_oracle_and_mlp_on_two_calls_in_a_row(sg):
    cases = [(128, 896, 4864, 11, True), (200, 264, 520, 12, False)]
    results = []
    for M, H, F, seed, with_r in cases:      # two calls back to back, no sync between
        host = _case(M, H, F, seed, with_r)
        dev = tuple(t.to(DEV) if t is not None else None for t in host)
        results.append((_noalloc_c_abi(sg, *dev), host, dev))
    rc, detail = sg.swiglu_device_status()
    assert rc == sg.OK, (sg.status_string(rc), detail)
    for Z, (A, W1, W2, W3, R), dev in results:
        z = Z.double().cpu().numpy()
        bits = [si.bits_u16(t) for t in (A, W1, W2, W3)]
        ref = oracle.mlp_bf16(*bits, si.bits_u16(R) if R is not None else None)
        slack = oracle.mlp_rounding_slack(*bits)
        oracle.assert_parity(z, ref, "noalloc vs oracle", sig_slack=slack)
        want = sg.swiglu_mlp(*dev)                       # the existing entry point
        torch.cuda.synchronize()
        oracle.assert_parity(z, want.double().cpu().numpy(), "noalloc vs swiglu_mlp",
                             sig_slack=2 * slack)


def test_noalloc_rejects_y_beyond_the_scratch(sg):
    limit = sg.lib().swiglu_mlp_noalloc_scratch_bytes()
    assert limit == 32 << 20
    H, F = 64, 4096
    M = limit // (F * 2) + 1                 # Y = M*F*2 bytes, just over the limit
    # rejected before any pointer is used or anything is enqueued
    rc = sg.lib().swiglu_mlp_noalloc(16, 16, 16, 16, None, 16, M, H, F, None)
    assert rc == sg.ERR_UNSUPPORTED
