"""Pins for the producer part of the oracle: RMSNorm of A and its per-tensor
FP8 E4M3 quantisation (the step that feeds the FP8 form of the projection).

The page names FP8 quantisation as the next step in tensor-core density (page
"Riepilogo Tecnico: Sovrapposizione delle Attivazioni a Livello di Tile per
l'Inferenza Efficiente di LLM", section "Definizione del Problema") but defines
neither step, so the oracle follows the standard definitions (RMSNorm of Zhang
and Sennrich 2019; OCP E4M3 with round-to-nearest-even).  What pins it, other
than itself:

* hand-worked cases (``tests/golden/producer_cases.json``);
* the E4M3 encoder against the code table (every finite code round-trips),
  exact midpoints between neighbouring codes (ties to the even code), values
  beyond 448 (saturation), and torch's float8_e4m3fn conversion (a library
  routine) on random float32 values in range;
* RMSNorm closed forms: a constant row normalises to +-gamma, a one-hot row
  to sqrt(K) gamma_j, mean(a^2) = 1 for gamma = 1 and eps = 0, invariance under
  scaling x by a power of two, linearity in gamma, rows independent, and a
  zero row with eps = 0 (0/0) normalises to zeros, the reading the oracle and
  the kernels share;
* quantisation: the largest |a| maps to code +-448, every code is the nearest
  one (the error is at most half the local spacing), the rounding decision is
  taken on the exact quotient (values a hair off a midpoint, closer than
  binary32 resolves, still round to their own side), an all-zero input gives
  scale 0 and zero codes.

``producer_pin_failures(lib)`` runs them against a loaded oracle library; the
planted-mistake tests run it against mutated copies of the oracle.
"""
import ctypes
import json
import math
import os

import numpy as np
import torch

import oracle
import swiglu_inputs as si

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "producer_cases.json")


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def _bits(x):
    return si.bits_u16(torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16))


def _enc(lib, x):
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    q = np.empty(a.shape, dtype=np.uint8)
    lib.oracle_f64_to_e4m3_n(_ptr(a), a.size, _ptr(q))
    return q


def _dec(lib, codes):
    return np.array([lib.oracle_e4m3_to_f64(int(c)) for c in np.ravel(codes)]).reshape(np.shape(codes))


def _rms(lib, X, gamma, eps):
    X = np.ascontiguousarray(X)
    M, K = X.shape
    g = None if gamma is None else np.ascontiguousarray(gamma)
    A = np.empty((M, K))
    rc = lib.oracle_rmsnorm_bf16(_ptr(X), _ptr(g) if g is not None else None, float(eps), M, K, _ptr(A))
    assert rc == 0
    return A


def _quant(lib, a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    q = np.empty(a.shape, dtype=np.uint8)
    s = np.zeros(1, dtype=np.float32)
    assert lib.oracle_quant_e4m3(_ptr(a), a.size, _ptr(s), _ptr(q)) == 0
    return float(s[0]), q


def _finite_codes():
    c = np.arange(256, dtype=np.uint8)
    return c[(c & 0x7F) != 0x7F]


def producer_pin_failures(lib):
    """Names of the pins the given oracle library fails (empty = all pass)."""
    bad = []
    # -- hand-worked cases
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        X = _bits(c["X"])
        g = None if c["gamma"] is None else _bits(c["gamma"])
        A = _rms(lib, X, g, c["eps"])
        if not np.allclose(A, np.array(c["A"]), rtol=1e-14, atol=1e-15):
            bad.append(f"golden A: {c['name']}")
        s, q = _quant(lib, A)
        if s != float(np.float32(c["scale_exact"])):
            bad.append(f"golden scale: {c['name']}")
        if not np.array_equal(q, np.array(c["codes"], dtype=np.uint8)):
            bad.append(f"golden codes: {c['name']}")

    # -- E4M3 encoder
    codes = _finite_codes()
    vals = _dec(lib, codes)
    if not np.array_equal(_enc(lib, vals), codes):
        bad.append("encode(decode(code)) != code")
    pos = np.sort(vals[(vals > 0)])
    lo, hi = pos[:-1], pos[1:]
    mid = (lo + hi) / 2
    q_mid = _dec(lib, _enc(lib, mid))
    lo_even = (_enc(lib, lo) & 1) == 0
    if not np.array_equal(q_mid, np.where(lo_even, lo, hi)):
        bad.append("midpoints do not round to the even code")
    if not np.array_equal(_dec(lib, _enc(lib, mid * (1 + 1e-12))), hi):
        bad.append("just above a midpoint does not round up")
    if not np.array_equal(_dec(lib, _enc(lib, mid * (1 - 1e-12))), lo):
        bad.append("just below a midpoint does not round down")
    if not np.array_equal(_enc(lib, [449.0, 464.0, 1e6, -500.0]), np.array([0x7E, 0x7E, 0x7E, 0xFE], np.uint8)):
        bad.append("no saturation at 448")
    rng = np.random.default_rng(5)
    f = (rng.standard_normal(6000) * np.exp(rng.uniform(-9, 5.5, 6000))).astype(np.float32)
    f = f[np.abs(f) < 440]
    want = torch.from_numpy(f.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    if not np.array_equal(_enc(lib, f.astype(np.float64)), want):
        bad.append("encoder disagrees with torch float8_e4m3fn")

    # -- RMSNorm closed forms
    K = 24
    const = _bits(np.full((2, K), [[1.5], [-0.75]]))
    if not np.allclose(_rms(lib, const, None, 0.0), np.full((2, K), [[1.0], [-1.0]]), rtol=1e-15):
        bad.append("constant row does not normalise to sign")
    onehot = np.zeros((1, K), np.float32)
    onehot[0, 7] = 5.0
    A1 = _rms(lib, _bits(onehot), None, 0.0)
    if not (math.isclose(A1[0, 7], math.sqrt(K), rel_tol=1e-14) and np.count_nonzero(A1) == 1):
        bad.append("one-hot row is not sqrt(K)")
    Xr, _, _ = si.make_bf16(11, 8, K, seed=21)
    xb = si.bits_u16(Xr)
    A = _rms(lib, xb, None, 0.0)
    if not np.allclose((A * A).mean(axis=1), 1.0, rtol=1e-13):
        bad.append("mean of squares is not 1")
    A4 = _rms(lib, si.bits_u16(Xr * 4), None, 0.0)
    if not np.allclose(A4, A, rtol=1e-14, atol=0):
        bad.append("not invariant under scaling x")
    gam = torch.linspace(-2, 2, K).to(torch.bfloat16)
    Ag = _rms(lib, xb, si.bits_u16(gam), 0.0)
    Ag2 = _rms(lib, xb, si.bits_u16(gam * 2), 0.0)
    if not (np.allclose(Ag2, 2 * Ag, rtol=1e-15, atol=0)
            and np.allclose(Ag, A * gam.double().numpy(), rtol=1e-14, atol=1e-15)):
        bad.append("gamma is not a per-column factor")
    z = _rms(lib, _bits(np.zeros((2, K))), None, 0.0)
    if not (np.all(z == 0) and not np.signbit(z).any()):
        bad.append("zero row with eps = 0 does not normalise to +0")
    perm = np.random.default_rng(2).permutation(11)
    if not np.array_equal(_rms(lib, np.ascontiguousarray(xb[perm]), None, 1e-3), _rms(lib, xb, None, 1e-3)[perm]):
        bad.append("rows not independent")

    # -- quantisation
    a = np.random.default_rng(9).standard_normal((17, 40)) * 3
    s, q = _quant(lib, a)
    if s != float(np.float32(np.abs(a).max() / 448)):
        bad.append("scale is not amax/448")
    imax = np.unravel_index(np.abs(a).argmax(), a.shape)
    if q[imax] & 0x7F != 0x7E:
        bad.append("amax element is not +-448")
    v = a / s
    dq = _dec(lib, q)
    allv = np.sort(np.concatenate([-vals, vals]))
    idx = np.clip(np.searchsorted(allv, v), 1, allv.size - 1)
    gap = allv[idx] - allv[idx - 1]
    if not np.all(np.abs(dq - v) <= gap / 2 + 1e-12 * np.abs(v)):
        bad.append("a code is not the nearest")
    # The decision is taken on the exact quotient (OCP FP8: round to nearest
    # even of the value itself).  With max|a| = 448 the scale is exactly 1;
    # 1.0625 is the midpoint of codes 1.0 (0x38) and 1.125 (0x39), 1.1875 that
    # of 1.125 and 1.25 (0x3A).  A hair above the first rounds up and a hair
    # below the second rounds down, although binary32 would see both as exact
    # midpoints and round them to the even codes 0x38 and 0xBA.
    _, qt = _quant(lib, [448.0, 1.0625 * (1 + 2.0 ** -30), -1.1875 * (1 - 2.0 ** -30)])
    if not np.array_equal(qt, np.array([0x7E, 0x39, 0xB9], np.uint8)):
        bad.append("quantisation decision not taken on the exact quotient")
    s0, q0 = _quant(lib, np.zeros(10))
    if s0 != 0.0 or q0.any():
        bad.append("zero input does not give scale 0")
    return bad


def test_producer_pins():
    assert producer_pin_failures(oracle._load()) == []


def test_wrappers_agree_with_the_c_functions():
    X, _, _ = si.make_bf16(6, 8, 48, seed=4)
    xb = si.bits_u16(X)
    gam = si.bits_u16(torch.linspace(0.5, 1.5, 48).to(torch.bfloat16))
    s, q = oracle.rmsnorm_quant_e4m3(xb, gam, 1e-6)
    s2, q2 = oracle.quant_e4m3(oracle.rmsnorm_bf16(xb, gam, 1e-6))
    assert s == s2 and np.array_equal(q, q2) and q.shape == (6, 48)
