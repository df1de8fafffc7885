"""Pins for the oracle's MLP pieces: BF16 rounding, the linear product with a
residual, and the MLP block Z = BF16(SiLU(A W1) (.) (A W2)) W3 + R (the down
projection that follows the fused projection in the MLP the page discusses,
section "Definizione del Problema")."""
import numpy as np
import pytest
import torch

import oracle
import swiglu_inputs as si


def _bits(x):
    return si.bits_u16(torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16))


def test_bf16_rounding_matches_torch_on_floats():
    rng = np.random.default_rng(0)
    u = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    # add ties (low 16 bits exactly 0x8000), subnormals, extremes
    ties = (rng.integers(0, 2 ** 16, size=500, dtype=np.uint64).astype(np.uint32) << 16 | 0x8000).view(np.float32)
    extra = np.array([0.0, -0.0, 1e-45, -1e-45, 1.17e-38, 3.3e38, -3.39e38, 1.0, -1.0, 65504.0],
                     dtype=np.float32)
    f = np.concatenate([f, ties[np.isfinite(ties)], extra])
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f64_to_bf16(float(x)) for x in f], dtype=np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(f[i]), hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_bf16_rounding_exact_on_doubles():
    # 1 + 2^-8 + 2^-30 is just above the midpoint of 1 and 1 + 2^-7: rounds up.
    # (Rounding through float first would lose 2^-30 and tie down to 1.0.)
    assert oracle.f64_to_bf16(1.0 + 2 ** -8 + 2 ** -30) == 0x3F81
    assert oracle.f64_to_bf16(1.0 + 2 ** -8) == 0x3F80          # tie to even (down)
    assert oracle.f64_to_bf16(1.0 + 3 * 2 ** -8) == 0x3F82      # tie to even (up)
    assert oracle.f64_to_bf16(2.0 ** 128) == 0x7F80              # overflow
    assert oracle.f64_to_bf16(-(2.0 ** -133)) == 0x8001          # smallest subnormal
    assert oracle.f64_to_bf16(2.0 ** -134) == 0x0000             # tie to even at zero
    assert oracle.f64_to_bf16(3 * 2.0 ** -134) == 0x0002         # tie to even (up)


def test_rounding_slack_flags_only_values_near_a_midpoint():
    # g = 40.x, u = 1: y = SiLU(g) = g to double precision.  BF16 values in
    # [32, 64) are 2^-2 apart, so 40.125 is a rounding midpoint.  With K = 1,
    # Gabs = |g| and Uabs = 1 the modelled error of y is about 1.5e-3: a value
    # 2^-14 off the midpoint is flagged (slack = spacing + dy), values 2^-6
    # off it or exactly representable are not.
    g = np.array([40.125 + 2 ** -14, 40.25, 40.125 + 2 ** -6, 40.0])
    s = oracle.bf16_rounding_slack(g, g, np.ones(4), np.abs(g), np.ones(4), 1)
    assert 0.25 < s[0] < 0.26
    assert s[1] == 0 and s[2] == 0 and s[3] == 0
    # y = 0 exactly with u = 0 and Uabs = 0: nothing can move, slack 0
    assert oracle.bf16_rounding_slack(np.zeros(1), np.ones(1), np.zeros(1), np.ones(1),
                                      np.zeros(1), 1)[0] == 0.0


def _other_bf16_neighbour(y, yb):
    """The BF16 value next to yb on the side of y (y exact, yb = BF16(y))."""
    ab = np.abs(yb)
    m, e = np.frexp(ab)
    above = np.ldexp(1.0, e - 8)
    below = np.where(m == 0.5, above / 2, above)
    up = np.abs(y) > ab
    return np.sign(y) * np.where(up, ab + above, ab - below)


def test_mlp_rounding_slack_covers_neighbour_roundings():
    # Z computed with every flagged Y element rounded to its other BF16
    # neighbour stays within the slack of the oracle's Z; rows are independent.
    M, H, F = 9, 64, 96
    A, W1, W2 = si.make_bf16(M, F, H, seed=13)
    W3 = si.make_bf16(1, H, F, seed=14)[1]
    a, w1, w2, w3 = (si.bits_u16(t) for t in (A, W1, W2, W3))
    Z, Yb = oracle.mlp_bf16(a, w1, w2, w3, with_y=True)
    G, U, Y = oracle.swiglu_bf16(a, w1, w2, with_gate_up=True)
    Ga, Ua, _ = oracle.swiglu_bf16(a & 0x7FFF, w1 & 0x7FFF, w2 & 0x7FFF, with_gate_up=True)
    s = oracle.bf16_rounding_slack(Y, G, U, Ga, Ua, H)
    assert 0 < np.count_nonzero(s) < s.size // 4
    yb = oracle.bf16_bits_to_f64(Yb)
    flipped = np.where(s > 0, _other_bf16_neighbour(Y, yb), yb)
    Z_other = flipped @ oracle.bf16_bits_to_f64(w3)
    B = oracle.mlp_rounding_slack(a, w1, w2, w3)
    assert np.all(np.abs(Z_other - Z) <= B + 1e-12 * np.abs(Z))
    assert np.array_equal(oracle.mlp_rounding_slack(a, w1, w2, w3, rows=[8, 2]), B[[8, 2]])


@pytest.mark.parametrize("with_r", [False, True])
def test_linear_against_numpy(with_r):
    M, N, K = 37, 72, 56
    X, W, _ = si.make_bf16(M, N, K, seed=7)
    R = si.make_bf16(M, N, 8, seed=8)[0][:, :8].repeat(1, N // 8) if with_r else None
    Rb = si.bits_u16(R.contiguous()) if with_r else None
    Z = oracle.linear_bf16(si.bits_u16(X), si.bits_u16(W), Rb)
    want = X.double().numpy() @ W.double().numpy()
    if with_r:
        want = want + R.double().numpy()
    np.testing.assert_allclose(Z, want, rtol=1e-12, atol=1e-12)


def test_linear_identity_weight_and_rows():
    X = _bits(np.arange(12, dtype=np.float32).reshape(3, 4) - 5)
    I = _bits(np.eye(4, dtype=np.float32))
    R = _bits(np.full((3, 4), 0.5, dtype=np.float32))
    Z = oracle.linear_bf16(X, I, R)
    assert np.array_equal(Z, np.arange(12, dtype=np.float64).reshape(3, 4) - 5 + 0.5)
    assert np.array_equal(oracle.linear_bf16(X, I, R, rows=[2, 0]), Z[[2, 0]])


def test_mlp_is_rounded_swiglu_then_linear():
    M, H, F = 21, 40, 56
    A, W1, W2 = si.make_bf16(M, F, H, seed=3)
    W3 = si.make_bf16(1, H, F, seed=4)[1]          # [F, H]
    R = si.make_bf16(M, H, 8, seed=5)[0][:, :8].repeat(1, H // 8).contiguous()
    a, w1, w2, w3, r = (si.bits_u16(t) for t in (A, W1, W2, W3, R))
    Z, Y = oracle.mlp_bf16(a, w1, w2, w3, r, with_y=True)
    y_exact = oracle.swiglu_bf16(a, w1, w2)
    assert np.array_equal(Y, np.array([[oracle.f64_to_bf16(v) for v in row] for row in y_exact],
                                      dtype=np.uint16))
    assert np.array_equal(Z, oracle.linear_bf16(Y, w3, r))
    # rows are independent
    assert np.array_equal(oracle.mlp_bf16(a, w1, w2, w3, r, rows=[20, 3]), Z[[20, 3]])
    # without the residual
    assert np.array_equal(oracle.mlp_bf16(a, w1, w2, w3), oracle.linear_bf16(Y, w3))
