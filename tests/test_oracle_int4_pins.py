"""Pins for the weight-only INT4 part of the oracle.

The page names INT4 (section "Definizione del Problema") but fixes no format;
the oracle's reading: signed 4-bit two's complement codes packed two per byte
along N (even column in the low nibble), one BF16 scale per column and per
group of G rows along K, and the weight the product uses is BF16(q * s).
What pins it, other than itself:

* hand-worked cases (``tests/golden/int4_cases.json``): nibble order, sign
  extension, group broadcast, and a product that BF16 must round (one case
  rounds up, one is an exact tie that goes to the even value);
* the code table against numpy's own two's-complement view of a nibble;
* group scales: multiplying one group's scales by 2 doubles exactly that
  group's rows, and nothing else;
* the product: with scales of one significant bit the dequantised weights are
  exact, and the SwiGLU result equals the BF16 definition on those weights
  computed by numpy in float64;
* planted mistakes (in test_oracle_mutants.py) each fail one
  of these.

``int4_pin_failures(lib)`` runs them against a loaded oracle library.
"""
import ctypes
import json
import os

import numpy as np
import torch

import oracle
import swiglu_inputs as si

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "int4_cases.json")


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def _bf16_bits(x):
    return si.bits_u16(torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def _deq(lib, Wq, S, G):
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    S = np.ascontiguousarray(S)
    K, half = Wq.shape
    W = np.empty((K, 2 * half))
    assert lib.oracle_dequant_int4(_ptr(Wq), _ptr(S), K, 2 * half, G, _ptr(W)) == 0
    return W


def _y(lib, A, W1q, S1, W2q, S2, G):
    A = np.ascontiguousarray(A)
    M, K = A.shape
    N = 2 * W1q.shape[1]
    Y = np.empty((M, N))
    assert lib.oracle_swiglu_w4(_ptr(A), _ptr(np.ascontiguousarray(W1q)), _ptr(np.ascontiguousarray(S1)),
                                _ptr(np.ascontiguousarray(W2q)), _ptr(np.ascontiguousarray(S2)),
                                M, N, K, G, None, M, _ptr(Y)) == 0
    return Y


def int4_pin_failures(lib):
    bad = []
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        W = _deq(lib, np.array(c["Wq"], dtype=np.uint8), _bf16_bits(c["S"]), c["G"])
        if not np.array_equal(W, np.array(c["W"])):
            bad.append(f"golden: {c['name']}")
    want = (np.arange(16, dtype=np.uint8) << 4).view(np.int8) >> 4   # arithmetic shift sign-extends
    got = np.array([lib.oracle_int4_value(i) for i in range(16)])
    if not np.array_equal(got, want.astype(np.float64)):
        bad.append("code table")
    rng = np.random.default_rng(3)
    K, N, G = 8, 6, 4
    Wq = rng.integers(0, 256, size=(K, N // 2), dtype=np.uint8)
    S = _bf16_bits(2.0 ** rng.integers(-6, -2, size=(K // G, N)))  # one significant bit: exact products
    W = _deq(lib, Wq, S, G)
    S2 = S.copy()
    S2[1] = _bf16_bits(2.0 * torch.from_numpy(S[1].view(np.int16)).view(torch.bfloat16).float().numpy())
    W2 = _deq(lib, Wq, S2, G)
    if not (np.array_equal(W2[:G], W[:G]) and np.array_equal(W2[G:], 2 * W[G:])):
        bad.append("group scale is not per group of G rows")
    q = np.stack([(Wq & 0xF), (Wq >> 4)], axis=2).reshape(K, N).astype(np.int8)
    q = np.where(q >= 8, q - 16, q).astype(np.float64)
    sc = torch.from_numpy(S.view(np.int16)).view(torch.bfloat16).double().numpy()
    if not np.array_equal(W, q * np.repeat(sc, G, axis=0)):
        bad.append("dequantised weights differ from q * s")
    A = _bf16_bits(rng.standard_normal((5, K)))
    Wq2 = rng.integers(0, 256, size=(K, N // 2), dtype=np.uint8)
    Y = _y(lib, A, Wq, S, Wq2, S, G)
    a = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).double().numpy()
    with np.errstate(all="ignore"):  # a planted mistake may produce non-finite weights
        g, u = a @ W, a @ _deq(lib, Wq2, S, G)
        ok = np.allclose(Y, g / (1 + np.exp(-g)) * u, rtol=1e-12, atol=1e-12)
    if not ok:
        bad.append("SwiGLU on the dequantised weights")
    return bad


def test_int4_pins():
    assert int4_pin_failures(oracle._load()) == []


def test_int4_recipe_round_trips():
    """The input recipe's codes and scales reproduce its FP32 draws within half
    a quantisation step (a check of the inputs, not of the method)."""
    _, W1, _ = si.draw_fp32(1, 64, 256, seed=9)
    Wq, S = si.quantize_int4(W1, G=128)
    W = oracle.dequant_int4(si.bits_u8(Wq) if Wq.dtype != torch.uint8 else Wq.numpy(), si.bits_u16(S), 128)
    step = np.repeat(S.float().numpy(), 128, axis=0)
    assert np.all(np.abs(W - W1.double().numpy()) <= 0.5 * step + 2.0 ** -8 * np.abs(W) + 1e-30)


# ---- the K-major arrangement of the codes (swiglu_pack_w4_kmajor's layout) -------------------

def _kmajor(lib, Wq):
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    K, half = Wq.shape
    Wk = np.zeros((2 * half, K // 2), dtype=np.uint8)
    assert lib.oracle_pack_w4_kmajor(_ptr(Wq), K, 2 * half, _ptr(Wk)) == 0
    return Wk


def kmajor_pin_failures(lib):
    """The K-major packer against what pins it:

    * hand-worked (K = 8, N = 2): column 0 holds codes 1..8 down K, column 1
      codes 15..8; word 0 of a column is nibbles (k0 k2 k4 k6 k1 k3 k5 k7) from
      the low end, so column 0's bytes are 0x31 0x75 0x42 0x86 and column 1's
      0xDF 0x9B 0xCE 0x8A (worked by hand from the layout's statement);
    * read back the way the kernel reads it: (word >> 4i) & 0x000F000F is the
      pair (8j + 2i, 8j + 2i + 1) in its low and high 16 bits, for every
      column, word and i (random codes, an odd number of column pairs);
    * every code appears exactly once (the multiset of nibbles is unchanged).
    """
    bad = []
    c0 = np.arange(1, 9, dtype=np.uint8)
    c1 = (15 - np.arange(8)).astype(np.uint8)
    want = np.array([[0x31, 0x75, 0x42, 0x86], [0xDF, 0x9B, 0xCE, 0x8A]], dtype=np.uint8)
    if not np.array_equal(_kmajor(lib, (c0 | (c1 << 4)).reshape(8, 1)), want):
        bad.append("hand-worked K-major case")
    rng = np.random.default_rng(11)
    K, N = 64, 10
    Wq = rng.integers(0, 256, size=(K, N // 2), dtype=np.uint8)
    code = np.stack([Wq & 0xF, Wq >> 4], axis=2).reshape(K, N)  # code[k, n]
    words = _kmajor(lib, Wq).view("<u4")  # [N, K/8]
    ok = True
    for n in range(N):
        for j in range(K // 8):
            for i in range(4):
                pair = (int(words[n, j]) >> (4 * i)) & 0x000F000F
                ok &= bool(pair & 0xF == code[8 * j + 2 * i, n])
                ok &= bool(pair >> 16 == code[8 * j + 2 * i + 1, n])
    if not ok:
        bad.append("pairs (k, k + 1) in K order")
    Wq = rng.integers(0, 256, size=(24, 7), dtype=np.uint8)
    nib = lambda a: np.sort(np.concatenate([(a & 0xF).ravel(), (a >> 4).ravel()]))
    if not np.array_equal(nib(Wq), nib(_kmajor(lib, Wq))):
        bad.append("not a permutation of the codes")
    return bad


def test_kmajor_pack_pins():
    assert kmajor_pin_failures(oracle._load()) == []
