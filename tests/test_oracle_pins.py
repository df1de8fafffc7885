"""Pins for the CPU oracle: each check ties it to something other than itself.

The oracle implements Y = SiLU(A x W1) (.) (A x W2) (page "Riepilogo Tecnico:
Sovrapposizione delle Attivazioni a Livello di Tile per l'Inferenza Efficiente
di LLM", section "Definizione del Problema") and the interleaved W_fused form
(same page, section "Metodologia", item 2).  The pins below are: hand-worked
examples with closed forms, exact integer brute force, an independent float64
library product (numpy), decoding tables checked against torch's own dtype
conversions, algebraic identities of SiLU, and invariants of the definition.
A dropped term, a sign error in the exponent, a transposed operand, a swapped
gate/up pair or an off-by-one in the K loop each fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import swiglu_inputs as si

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _bf16_bits(x):
    return si.bits_u16(torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16))


def _golden(golden_dir):
    with open(os.path.join(golden_dir, "swiglu_2x2.json")) as f:
        return json.load(f)


# ---- hand-worked examples ------------------------------------------------

def test_golden_2x2_gate_up_exact(golden_dir):
    for case in _golden(golden_dir)["cases"]:
        A, W1, W2 = (_bf16_bits(case[k]) for k in ("A", "W1", "W2"))
        G, U, Y = oracle.swiglu_bf16(A, W1, W2, with_gate_up=True)
        assert np.array_equal(G, np.array(case["G"], dtype=np.float64)), case["name"]
        assert np.array_equal(U, np.array(case["U"], dtype=np.float64)), case["name"]


def test_golden_2x2_closed_forms(golden_dir):
    for case in _golden(golden_dir)["cases"]:
        A, W1, W2 = (_bf16_bits(case[k]) for k in ("A", "W1", "W2"))
        Y = oracle.swiglu_bf16(A, W1, W2)
        want = np.array([[eval(e, {"exp": math.exp}) for e in row]
                         for row in case["Y_closed_form"]], dtype=np.float64)
        np.testing.assert_allclose(Y, want, rtol=1e-14, atol=1e-300)
        np.testing.assert_allclose(Y, np.array(case["Y_decimal"]), rtol=0, atol=6e-11)


def test_golden_2x2_interleaved(golden_dir):
    for case in _golden(golden_dir)["cases"]:
        A, W1, W2 = (_bf16_bits(case[k]) for k in ("A", "W1", "W2"))
        Wf = oracle.pack_interleaved(W1, W2)
        assert np.array_equal(Wf, _bf16_bits(case["W_fused"])), case["name"]
        Y = oracle.swiglu_interleaved_bf16(A, Wf)
        np.testing.assert_allclose(Y, np.array(case["Y_decimal"]), rtol=0, atol=6e-11)


# ---- decoding tables against torch's conversions --------------------------

def test_bf16_decode_all_codes():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).float().double().numpy()
    lib = oracle._load()
    got = np.array([lib.oracle_bf16_to_f64(int(c)) for c in codes[::17]])
    want = ref[::17]
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # a few by value
    assert oracle.bf16_to_f64(0x3F80) == 1.0
    assert oracle.bf16_to_f64(0xC000) == -2.0
    assert oracle.bf16_to_f64(0x0001) == 2.0 ** -133


def test_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().double().numpy()
    got = np.array([oracle.e4m3_to_f64(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert oracle.e4m3_to_f64(0x7E) == 448.0
    assert oracle.e4m3_to_f64(0x38) == 1.0
    assert oracle.e4m3_to_f64(0x01) == 2.0 ** -9
    assert oracle.e4m3_to_f64(0x08) == 2.0 ** -6
    assert oracle.e4m3_to_f64(0xFE) == -448.0


# ---- SiLU -------------------------------------------------------------------

def test_silu_special_values_and_identity():
    assert oracle.silu(0.0) == 0.0
    # sigma(1) = e / (1 + e), a textbook constant
    assert oracle.silu(1.0) == pytest.approx(0.7310585786300049, rel=1e-15)
    # SiLU(x) -> x for large x, -> 0- for very negative x
    assert oracle.silu(40.0) == pytest.approx(40.0, rel=1e-15)
    assert -1e-15 < oracle.silu(-40.0) < 0.0
    assert oracle.silu(-1000.0) == 0.0 or oracle.silu(-1000.0) == -0.0
    # sigma(-x) = 1 - sigma(x)  =>  SiLU(-x) = SiLU(x) - x
    for x in np.linspace(-30, 30, 241):
        assert oracle.silu(-x) == pytest.approx(oracle.silu(x) - x, rel=1e-12, abs=1e-13)
    # derivative at 0 is 1/2: SiLU(h) / h -> sigma(0) = 1/2
    h = 1e-8
    assert oracle.silu(h) / h == pytest.approx(0.5, rel=1e-7)


# ---- exact brute force on small integers ----------------------------------

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_integer_brute_force_exact(seed):
    rng = np.random.default_rng(seed)
    M, N, K = (int(v) for v in rng.integers(1, 17, size=3))
    A = rng.integers(-8, 9, size=(M, K))
    W1 = rng.integers(-8, 9, size=(K, N))
    W2 = rng.integers(-8, 9, size=(K, N))
    G, U, Y = oracle.swiglu_bf16(_bf16_bits(A), _bf16_bits(W1), _bf16_bits(W2), with_gate_up=True)
    for m in range(M):
        for n in range(N):
            g = sum(int(A[m, k]) * int(W1[k, n]) for k in range(K))
            u = sum(int(A[m, k]) * int(W2[k, n]) for k in range(K))
            assert G[m, n] == g and U[m, n] == u
            if u == 0:
                assert Y[m, n] == 0.0
            else:
                # sigma from its limit forms, written independently of the oracle's x/(1+e^-x)
                sig = math.exp(g) / (1.0 + math.exp(g)) if g < 0 else 1.0 / (1.0 + math.exp(-g))
                assert Y[m, n] == pytest.approx(g * sig * u, rel=1e-14, abs=1e-300)


def test_exhaustive_1x1():
    # every small integer pair (a*w1, a*w2) on a 1x1x1 problem
    for a in range(-3, 4):
        for w1 in range(-3, 4):
            for w2 in range(-3, 4):
                Y = oracle.swiglu_bf16(_bf16_bits([[a]]), _bf16_bits([[w1]]), _bf16_bits([[w2]]))
                g, u = a * w1, a * w2
                want = g * u / (1.0 + math.exp(-g))
                assert Y[0, 0] == pytest.approx(want, rel=1e-15, abs=0.0)


# ---- an independent float64 library product --------------------------------

@pytest.mark.parametrize("shape", [(37, 53, 72), (5, 130, 264), (64, 24, 9)])
def test_against_numpy_float64(shape):
    M, N, K = shape
    A, W1, W2 = si.make_bf16(M, N, K, seed=11)
    a, w1, w2 = (t.double().numpy() for t in (A, W1, W2))
    g = a @ w1
    u = a @ w2
    want = g / (1.0 + np.exp(-g)) * u
    G, U, Y = oracle.swiglu_bf16(si.bits_u16(A), si.bits_u16(W1), si.bits_u16(W2), with_gate_up=True)
    scale_g = np.abs(a) @ np.abs(w1)
    scale_u = np.abs(a) @ np.abs(w2)
    assert np.all(np.abs(G - g) <= 1e-13 * scale_g + 1e-300)
    assert np.all(np.abs(U - u) <= 1e-13 * scale_u + 1e-300)
    np.testing.assert_allclose(Y, want, rtol=1e-9, atol=1e-12 * np.abs(want).max())


# ---- invariants of the definition -------------------------------------------

def _case(M=23, N=40, K=48, seed=5):
    A, W1, W2 = si.make_bf16(M, N, K, seed)
    return si.bits_u16(A), si.bits_u16(W1), si.bits_u16(W2)


def test_zero_operands_give_zero():
    A, W1, W2 = _case()
    z = np.zeros_like(W1)
    assert np.all(oracle.swiglu_bf16(A, W1, z) == 0.0)     # U = 0
    assert np.all(oracle.swiglu_bf16(A, z, W2) == 0.0)     # SiLU(0) = 0
    assert np.all(oracle.swiglu_bf16(np.zeros_like(A), W1, W2) == 0.0)


def test_scaling_up_weights_doubles_output_exactly():
    A, W1, W2 = _case()
    W2x2 = _bf16_bits(torch.from_numpy(W2.view(np.int16).copy()).view(torch.bfloat16).float() * 2)
    assert np.array_equal(oracle.swiglu_bf16(A, W1, W2x2), 2.0 * oracle.swiglu_bf16(A, W1, W2))


def test_gate_and_up_are_not_interchangeable():
    A, W1, W2 = _case()
    assert not np.allclose(oracle.swiglu_bf16(A, W1, W2), oracle.swiglu_bf16(A, W2, W1))


def test_rows_are_independent_and_sampling_matches():
    A, W1, W2 = _case(M=31)
    Y = oracle.swiglu_bf16(A, W1, W2)
    perm = np.random.default_rng(3).permutation(A.shape[0])
    assert np.array_equal(oracle.swiglu_bf16(A[perm], W1, W2), Y[perm])
    rows = [30, 0, 7, 7, 19]
    assert np.array_equal(oracle.swiglu_bf16(A, W1, W2, rows=rows), Y[rows])


def test_interleaved_form_equals_separate_form():
    A, W1, W2 = _case(M=17, N=72, K=40)
    Wf = oracle.pack_interleaved(W1, W2)
    assert np.array_equal(Wf[:, 0::2], W1) and np.array_equal(Wf[:, 1::2], W2)
    assert np.array_equal(oracle.swiglu_interleaved_bf16(A, Wf), oracle.swiglu_bf16(A, W1, W2))


def test_bad_row_index_is_rejected():
    A, W1, W2 = _case(M=4)
    with pytest.raises(ValueError):
        oracle.swiglu_bf16(A, W1, W2, rows=[4])


def test_k_zero_gives_zero():
    A = np.zeros((3, 0), dtype=np.uint16)
    W = np.zeros((0, 5), dtype=np.uint16)
    assert np.all(oracle.swiglu_bf16(A, W, W) == 0.0)


# ---- FP8 E4M3 ----------------------------------------------------------------

def test_e4m3_oracle_matches_bf16_oracle_on_same_values():
    (Aq, W1q, W2q), _ = si.make_e4m3(19, 48, 64, seed=4)
    # every E4M3 value is exact in BF16 (3 mantissa bits, exponent within range)
    to_bf = lambda q: si.bits_u16(q.float().to(torch.bfloat16))
    Yq = oracle.swiglu_e4m3(si.bits_u8(Aq), si.bits_u8(W1q), si.bits_u8(W2q), 1.0, 1.0, 1.0)
    Yb = oracle.swiglu_bf16(to_bf(Aq), to_bf(W1q), to_bf(W2q))
    assert np.array_equal(Yq, Yb)
    Y2 = oracle.swiglu_e4m3(si.bits_u8(Aq), si.bits_u8(W1q), si.bits_u8(W2q), 1.0, 1.0, 2.0)
    assert np.array_equal(Y2, 2.0 * Yq)


def test_e4m3_dequantised_definition():
    (Aq, W1q, W2q), (sA, s1, s2) = si.make_e4m3(9, 24, 32, seed=4)
    a = Aq.float().double().numpy() * sA
    w1 = W1q.float().double().numpy() * s1
    w2 = W2q.float().double().numpy() * s2
    g, u = a @ w1, a @ w2
    want = g / (1.0 + np.exp(-g)) * u
    got = oracle.swiglu_e4m3(si.bits_u8(Aq), si.bits_u8(W1q), si.bits_u8(W2q), sA, s1, s2)
    np.testing.assert_allclose(got, want, rtol=1e-9, atol=1e-12 * np.abs(want).max())


# ---- the acceptance check itself ------------------------------------------------

def test_parity_report_flags_errors():
    ref = np.linspace(-3, 3, 101)
    assert oracle.parity_report(ref, ref)["ok"]
    assert oracle.parity_report(ref * (1 + 5e-3), ref)["ok"]
    bad = ref.copy()
    bad[80] *= 1.02            # 2 % off on a significant element
    assert not oracle.parity_report(bad, ref)["ok"]
    nan = ref.copy()
    nan[3] = np.nan
    assert not oracle.parity_report(nan, ref)["ok"]


def test_parity_report_per_element_slack():
    ref = np.linspace(1, 2, 1000)
    y = ref.copy()
    y[:2] *= 1.011              # 2 of 1000 significant elements 1.1 % off, inside bound (1)
    assert not oracle.parity_report(y, ref)["ok"]
    slack = np.zeros_like(ref)
    slack[0] = 0.002            # explains the first element's excess only
    assert not oracle.parity_report(y, ref, sig_slack=slack)["ok"]
    slack[1] = 0.002
    assert oracle.parity_report(y, ref, sig_slack=slack)["ok"]
    # slack widens rule (2) only: bound (1) still holds every element
    far = ref.copy()
    far[500] *= 1.03
    assert not oracle.parity_report(far, ref, sig_slack=np.full_like(ref, 1.0))["ok"]
