"""GPU parity of the FP8 E4M3 path against the oracle on dequantised values.

Operands are per-tensor-scaled E4M3 codes (scale = amax/448); the oracle
evaluates Y = SiLU(A W1) (.) (A W2) on code*scale in double.  The GPU takes the
weights K-major ([N,K]); the oracle takes the same codes as [K,N].  The
acceptance rule is the BF16 one: FP8 inputs are exact values to both sides,
the only differences are FP32 accumulation and the BF16 rounding of Y.
"""
import numpy as np
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


def _scales(s):
    return [torch.tensor([v], dtype=torch.float32, device=DEV) for v in s]


def _run(sg, form, q, s):
    Aq, W1q, W2q = q
    Ad = Aq.to(DEV)
    W1t, W2t = W1q.t().contiguous().to(DEV), W2q.t().contiguous().to(DEV)
    sA, s1, s2 = _scales(s)
    if form == "separate":
        Y = sg.swiglu_fused_fp8(Ad, W1t, W2t, sA, s1, s2)
    else:
        Wft = sg.swiglu_pack_interleaved_fp8(W1t, W2t)
        Y = sg.swiglu_fused_interleaved_fp8(Ad, Wft, sA, s1, s2)
    rc, detail = sg.swiglu_device_status()
    assert rc == sg.OK, f"device status {sg.status_string(rc)} detail {detail}"
    return Y


def _ref(q, s, rows=None):
    Aq, W1q, W2q = q
    return oracle.swiglu_e4m3(si.bits_u8(Aq), si.bits_u8(W1q), si.bits_u8(W2q), *s, rows=rows)


@pytest.mark.parametrize("form", ["separate", "interleaved"])
@pytest.mark.parametrize("shape", [(1, 8, 16), (7, 72, 128), (200, 264, 272), (257, 392, 528),
                                   (512, 1000, 256)], ids=lambda s: "x".join(map(str, s)))
def test_fp8_small_shapes(sg, form, shape):
    M, N, K = shape
    q, s = si.make_e4m3(M, N, K, seed=M + N + K)
    Y = _run(sg, form, q, s)
    oracle.assert_parity(Y.float().cpu().numpy(), _ref(q, s), f"fp8 {form} {shape}")


@pytest.mark.parametrize("M", [512, 4096])
def test_fp8_qwen7b_shapes(sg, M):
    K, N = 3584, 18944
    q, s = si.make_e4m3(M, N, K, seed=4)
    rows = si.sample_rows(M, 128, 48, seed=4)
    for form in ("separate", "interleaved"):
        Y = _run(sg, form, q, s)
        y = Y.float().cpu().numpy()[rows]
        oracle.assert_parity(y, _ref(q, s, rows=rows), f"fp8 7b M={M} {form}")
        del Y
    torch.cuda.empty_cache()


def test_fp8_pack_is_bit_exact(sg):
    for N, K in [(8, 16), (264, 272), (4864, 896)]:
        q, _ = si.make_e4m3(1, N, K, seed=N)
        _, W1q, W2q = q
        Wft = sg.swiglu_pack_interleaved_fp8(W1q.t().contiguous().to(DEV),
                                             W2q.t().contiguous().to(DEV))
        torch.cuda.synchronize()
        want = oracle.pack_interleaved(si.bits_u8(W1q), si.bits_u8(W2q)).T
        assert np.array_equal(si.bits_u8(Wft.cpu()), want)


def test_fp8_scales_are_applied(sg):
    M, N, K = 130, 136, 256
    q, s = si.make_e4m3(M, N, K, seed=21)
    s2 = (s[0], s[1], 2.0 * s[2])   # doubling the up scale doubles Y
    Y1 = _run(sg, "separate", q, s)
    Y2 = _run(sg, "separate", q, s2)
    oracle.assert_parity(Y2.float().cpu().numpy(), _ref(q, s2), "fp8 scaled")
    assert torch.equal(Y2.float(), 2.0 * Y1.float())


@pytest.mark.parametrize("form", ["separate", "interleaved"])
def test_fp8_schedules_agree(sg, form):
    """The FP8 pair kernel on more tiles than pairs fit (3 x 31 tiles of 256 x
    128, ragged in M, N and K): the dynamic and static tile schedules give the
    same Y bit for bit, and both match the oracle."""
    M, N, K = 600, 3904, 208
    q, s = si.make_e4m3(M, N, K, seed=31)
    out = {}
    try:
        for dyn in (1, 0):
            sg.swiglu_set_pair_schedule(dyn)
            out[dyn] = _run(sg, form, q, s)
    finally:
        sg.swiglu_set_pair_schedule(1)
    assert torch.equal(out[0].view(torch.int16), out[1].view(torch.int16))
    rows = si.sample_rows(M, 128, 32, seed=31)
    oracle.assert_parity(out[1].float().cpu().numpy()[rows], _ref(q, s, rows=rows),
                         f"fp8 {form}, dynamic schedule")
