"""GPU parity of the A producer (RMSNorm + per-tensor E4M3 quantisation) and
of the weight quantiser against the oracle, and of the composed FP8 path
(producer, then the fused FP8 projection).

The codes are integers decided by floating point.  The oracle decides on the
exact quotient a / s (OCP 8-bit floating point: round to nearest even of the
value); the kernels decide in binary32.  So codes must be bit-identical except
where binary32 arithmetic may fall on the other side of a midpoint: an element
may take the other of the two codes around a / s only when a / s (oracle,
double) lies within a relative distance delta of their midpoint, with delta
the FP32 error bound of the kernel's arithmetic.

* Plain quantisation of BF16 values: the kernel's quotient is one correctly
  rounded binary32 division of the same a and s, so delta = u = 2^-24, and the
  scale (max|x| / 448, one correctly rounded division) must be bit-identical.
  With BF16 inputs and a BF16 maximum, many quotients lie within u of a
  midpoint, where binary32 sees an exact tie; those elements may take either
  neighbour.
* After RMSNorm the kernel's binary32 value of a also differs from the
  oracle's by rounding: the sum of K squares over K/32 sequential terms per
  lane plus a 5-level shuffle tree (relative error <= (K/32 + 5) u), halved
  by the square root, plus about ten correctly rounded operations on each
  side (division, square root, reciprocal, products, the scale's division by
  448): delta = (K/32 + 32) u covers it with room.  The scale must agree
  within the same relative bound.
"""
import numpy as np
import pytest
import torch

import oracle
import swiglu_inputs as si

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
U = 2.0 ** -24


@pytest.fixture(scope="module")
def sg():
    import __graft_entry__
    __graft_entry__.build()
    import swiglu_gemm_transformer_gb300 as m
    m.lib()
    return m


_DEC = None


def _decode(q):
    global _DEC
    if _DEC is None:
        _DEC = np.array([oracle.e4m3_to_f64(c) for c in range(256)])
    return _DEC[q]


def assert_codes(q_gpu, s_gpu, a_ref, K, what, plain=False):
    """q_gpu: uint8 codes, s_gpu: float scale; a_ref: oracle values (double).
    plain: quantisation of BF16 values without normalisation (the kernel's
    quotient is one correctly rounded binary32 division, its scale one
    correctly rounded binary32 division of the exact maximum)."""
    s_ref, q_ref = oracle.quant_e4m3(a_ref)
    delta = U if plain else (K / 32 + 32) * U
    if s_ref == 0.0:
        assert s_gpu == 0.0 and not q_gpu.any(), what
        return
    if plain:
        assert s_gpu == s_ref, f"{what}: scale {s_gpu} vs {s_ref}"
    else:
        assert abs(s_gpu - s_ref) <= delta * s_ref, f"{what}: scale {s_gpu} vs {s_ref}"
    bad = q_gpu != q_ref
    n_bad = int(bad.sum())
    if n_bad == 0:
        return
    v = a_ref[bad] / s_ref
    lo, hi = _decode(q_ref[bad]), _decode(q_gpu[bad])
    mid = (lo + hi) / 2
    neighbours = np.abs(lo - hi) <= np.maximum(np.abs(lo), np.abs(hi)) / 4 + 2 ** -9
    near_mid = np.abs(v - mid) <= delta * np.abs(v) + 1e-300
    ok = neighbours & near_mid & (np.sign(lo) * np.sign(hi) >= 0)
    assert ok.all(), (f"{what}: {int((~ok).sum())} of {q_gpu.size} codes differ away from a midpoint; "
                      f"first at {np.argwhere(bad)[~ok][0]}: v={v[~ok][0]!r} gpu={hi[~ok][0]} ref={lo[~ok][0]}")
    # Every value is a BF16 input times one FP32 factor, so far more values
    # sit within rounding of an exact midpoint than a continuous distribution
    # would put there; the per-element rule above is the criterion, this only
    # catches a wholesale shift.
    assert n_bad <= max(4, 0.02 * q_gpu.size), f"{what}: {n_bad} near-midpoint flips is too many"


def _produce(sg, X, gamma, eps):
    Xd = X.to(DEV)
    gd = gamma.to(DEV) if gamma is not None else None
    Aq, sA = sg.swiglu_rmsnorm_quant_fp8(Xd, gd, eps)
    rc, detail = sg.swiglu_device_status()
    assert rc == sg.OK, (sg.status_string(rc), detail)
    return si.bits_u8(Aq.cpu()), float(sA.item())


@pytest.mark.parametrize("shape", [(1, 16), (7, 112), (200, 896), (333, 3584), (64, 4864), (9, 8192)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("with_gamma", [True, False], ids=["gamma", "nogamma"])
@pytest.mark.parametrize("eps", [1e-6, 0.0])
def test_rmsnorm_quant_small(sg, shape, with_gamma, eps):
    M, K = shape
    X, gamma = si.make_producer_inputs(M, K, seed=M * 7 + K)
    g = gamma if with_gamma else None
    q, s = _produce(sg, X, g, eps)
    a = oracle.rmsnorm_bf16(si.bits_u16(X), si.bits_u16(g) if g is not None else None, eps)
    assert_codes(q, s, a, K, f"rmsnorm_quant {shape}")


@pytest.mark.parametrize("M", [512, 4096])
def test_rmsnorm_quant_full_size(sg, M):
    """The FP8 configuration's A: K = 3584, every element checked."""
    K = 3584
    X, gamma = si.make_producer_inputs(M, K, seed=4)
    q, s = _produce(sg, X, gamma, 1e-6)
    a = oracle.rmsnorm_bf16(si.bits_u16(X), si.bits_u16(gamma), 1e-6)
    assert_codes(q, s, a, K, f"rmsnorm_quant M={M}")


@pytest.mark.parametrize("shape", [(16, 16), (264, 144), (18944, 3584)], ids=lambda s: "x".join(map(str, s)))
def test_weight_quant(sg, shape):
    N, K = shape
    _, W1, _ = si.make_bf16(1, N, K, seed=N + K)
    Wt = W1.t().contiguous()                  # K-major [N,K], the FP8 entry points' layout
    q, s = sg.swiglu_quant_fp8(Wt.to(DEV))
    assert_codes(si.bits_u8(q.cpu()), float(s.item()), Wt.double().numpy(), K, f"quant {shape}", plain=True)


def test_edge_cases(sg):
    K = 64
    # all zeros: scale 0, codes 0
    q, s = _produce(sg, torch.zeros(5, K, dtype=torch.bfloat16), None, 0.0)
    assert s == 0.0 and not q.any()
    # one zero row with eps = 0 among normal rows: that row's codes are +0
    X, gamma = si.make_producer_inputs(6, K, seed=3)
    X[2] = 0
    q, s = _produce(sg, X, gamma, 0.0)
    assert not q[2].any()
    assert_codes(q, s, oracle.rmsnorm_bf16(si.bits_u16(X), si.bits_u16(gamma), 0.0), K, "zero row")
    # an outlier row: with eps > 0 every row normalises to rms ~ 1, and the
    # largest |a| in the tensor gets code +-448
    X = torch.randn(8, K, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    X[3, 5] = 3000.0
    q, s = _produce(sg, X, None, 1e-6)
    a = oracle.rmsnorm_bf16(si.bits_u16(X), None, 1e-6)
    assert_codes(q, s, a, K, "outlier")
    assert q[3, 5] == 0x7E
    # M = 0 writes the scale 0 and nothing else
    sA = torch.full((1,), 5.0, device=DEV)
    Aq = torch.empty(0, K, dtype=torch.float8_e4m3fn, device=DEV)
    sg.swiglu_rmsnorm_quant_fp8(torch.empty(0, K, dtype=torch.bfloat16, device=DEV), None, 1e-6, Aq, sA)
    assert float(sA.item()) == 0.0


def test_argument_errors(sg):
    lib = sg.lib()
    X = torch.zeros(4, 48, dtype=torch.bfloat16, device=DEV)
    Aq = torch.empty(4, 48, dtype=torch.float8_e4m3fn, device=DEV)
    s = torch.empty(1, device=DEV)
    st = None
    assert lib.swiglu_rmsnorm_quant_fp8(X.data_ptr(), None, 1e-6, Aq.data_ptr(), s.data_ptr(), 4, 40, st) == sg.ERR_UNSUPPORTED
    assert lib.swiglu_rmsnorm_quant_fp8(X.data_ptr(), None, -1.0, Aq.data_ptr(), s.data_ptr(), 4, 48, st) == sg.ERR_INVALID_ARG
    assert lib.swiglu_rmsnorm_quant_fp8(X.data_ptr(), None, float("nan"), Aq.data_ptr(), s.data_ptr(), 4, 48, st) == sg.ERR_INVALID_ARG
    assert lib.swiglu_rmsnorm_quant_fp8(X.data_ptr() + 2, None, 1e-6, Aq.data_ptr(), s.data_ptr(), 4, 32, st) == sg.ERR_MISALIGNED
    assert lib.swiglu_rmsnorm_quant_fp8(X.data_ptr(), X.data_ptr() + 8, 1e-6, Aq.data_ptr(), s.data_ptr(), 4, 32, st) == sg.ERR_MISALIGNED
    assert lib.swiglu_rmsnorm_quant_fp8(X.data_ptr(), None, 1e-6, Aq.data_ptr(), s.data_ptr(), -1, 48, st) == sg.ERR_INVALID_ARG
    assert lib.swiglu_quant_fp8(X.data_ptr(), Aq.data_ptr(), s.data_ptr(), 4, 0, st) == sg.ERR_INVALID_ARG
    torch.cuda.synchronize()


@pytest.mark.parametrize("form", ["separate", "interleaved"])
@pytest.mark.parametrize("shape", [(200, 264, 272), (512, 18944, 3584)], ids=lambda s: "x".join(map(str, s)))
def test_composed_fp8_path(sg, form, shape):
    """Producer on the GPU, then the fused FP8 projection, against the oracle's
    own producer and FP8 definition.  The weights are quantised on both sides
    and the GPU's codes checked against the oracle's; the projection then
    takes the oracle's weight codes and scales as its inputs, so that a valid
    near-midpoint flip in a weight code (binary32 ties, see the module
    docstring) does not move a whole column of Y away from the reference."""
    M, N, K = shape
    X, gamma = si.make_producer_inputs(M, K, seed=40 + M)
    _, W1, W2 = si.make_bf16(1, N, K, seed=41 + N)
    Xd, gd = X.to(DEV), gamma.to(DEV)
    W1t, W2t = W1.t().contiguous().to(DEV), W2.t().contiguous().to(DEV)
    Aq, sA = sg.swiglu_rmsnorm_quant_fp8(Xd, gd, 1e-6)
    W1q, s1 = sg.swiglu_quant_fp8(W1t)
    W2q, s2 = sg.swiglu_quant_fp8(W2t)
    rc, detail = sg.swiglu_device_status()
    assert rc == sg.OK, (sg.status_string(rc), detail)

    rows = si.sample_rows(M, 128, 64, seed=5) if M > 256 else np.arange(M)
    sAo, Aqo = oracle.rmsnorm_quant_e4m3(si.bits_u16(X), si.bits_u16(gamma), 1e-6)
    s1o, W1qo = oracle.quant_e4m3(W1.double().numpy())
    s2o, W2qo = oracle.quant_e4m3(W2.double().numpy())
    # The codes: equal to the oracle's except near-midpoint flips (validated here).
    a_gpu = si.bits_u8(Aq.cpu())
    assert_codes(a_gpu, float(sA.item()), oracle.rmsnorm_bf16(si.bits_u16(X), si.bits_u16(gamma), 1e-6), K, "A")
    assert_codes(si.bits_u8(W1q.cpu()).T, float(s1.item()), W1.double().numpy(), K, "W1", plain=True)
    assert_codes(si.bits_u8(W2q.cpu()).T, float(s2.item()), W2.double().numpy(), K, "W2", plain=True)
    # The projection on the GPU's A codes and the oracle's weight codes.
    to_dev = lambda q: torch.from_numpy(np.ascontiguousarray(q.T)).view(torch.float8_e4m3fn).to(DEV)
    W1o, W2o = to_dev(W1qo), to_dev(W2qo)
    s1d = torch.tensor([s1o], dtype=torch.float32, device=DEV)
    s2d = torch.tensor([s2o], dtype=torch.float32, device=DEV)
    if form == "separate":
        Y = sg.swiglu_fused_fp8(Aq, W1o, W2o, sA, s1d, s2d)
    else:
        Y = sg.swiglu_fused_interleaved_fp8(Aq, sg.swiglu_pack_interleaved_fp8(W1o, W2o), sA, s1d, s2d)
    rc, detail = sg.swiglu_device_status()
    assert rc == sg.OK, (sg.status_string(rc), detail)
    # Y: element by element on every row whose A codes both sides chose alike
    # (a flipped code is a valid rounding, but it moves its whole row of Y by
    # one code step's worth).
    ref = oracle.swiglu_e4m3(Aqo, W1qo, W2qo, sAo, s1o, s2o, rows=rows)
    got = Y.double().cpu().numpy()[rows]
    same_rows = (a_gpu[rows] == Aqo[rows]).all(axis=1)
    assert same_rows.mean() > 0.9
    oracle.assert_parity(got[same_rows], ref[same_rows], f"rmsnorm+quant+fp8 {form} {shape}")
