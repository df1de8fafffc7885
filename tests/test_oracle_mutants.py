"""Planted-mistake checks: the oracle's pins must catch plausible bugs.

Each case below copies the oracle's C source, plants one mistake (a sign error
in the sigmoid, a dropped factor, a transposed operand, swapped gate/up roles,
an off-by-one in the K loop, a wrong exponent bias), builds the copy on the CPU
and runs the same kinds of pins as the pin suite against it.  The unmodified
source must pass them all and every mutant must fail at least one.  Nothing
here touches a GPU.
"""
import ctypes
import json
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
import swiglu_inputs as si

SRC = os.path.join(os.path.dirname(oracle.__file__), "swiglu_oracle.c")

MUTANTS = {
    "sigmoid_sign": ("return x / (1.0 + exp(-x));", "return x / (1.0 + exp(x));"),
    "drop_up_factor": ("Y[i * N + n] = oracle_silu(g[n]) * u[n];", "Y[i * N + n] = oracle_silu(g[n]);"),
    "transposed_w1": ("g[n] += ak * w1k[n];", "g[n] += ak * w1[n * K + k];"),
    "pack_swaps_roles": ("Wf[k * 2 * N + 2 * n] = W1[k * N + n];\n            Wf[k * 2 * N + 2 * n + 1] = W2[k * N + n];\n        }\n}\n\nvoid oracle_pack_interleaved_u8",
                         "Wf[k * 2 * N + 2 * n] = W2[k * N + n];\n            Wf[k * 2 * N + 2 * n + 1] = W1[k * N + n];\n        }\n}\n\nvoid oracle_pack_interleaved_u8"),
    "pair_step_swapped": ("oracle_silu(d[2 * n]) * d[2 * n + 1]", "oracle_silu(d[2 * n + 1]) * d[2 * n]"),
    "k_loop_short": ("for (int64_t k = 0; k < K; ++k) {\n        const double ak = a[k];", "for (int64_t k = 0; k + 1 < K; ++k) {\n        const double ak = a[k];"),
    "e4m3_bias": ("v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "bf16_shift": ("uint32_t w = (uint32_t)bits << 16;", "uint32_t w = (uint32_t)bits << 15;"),
}

# Planted mistakes in the MLP pieces, caught by the MLP pins below.
MLP_MUTANTS = {
    "round_truncates": ("double m = nearbyint(a / ulp);", "double m = floor(a / ulp);"),
    "round_via_float": ("double m = nearbyint(a / ulp);", "double m = nearbyint((double)(float)(a / ulp));"),
    "linear_drops_residual": ("Z[i * N + n] = z[n] + (R ? oracle_bf16_to_f64(R[m * N + n]) : 0.0);",
                              "Z[i * N + n] = z[n];"),
    "linear_transposed_w": ("const double *wk = w + k * N;\n                for (int64_t n = 0; n < N; ++n)\n                    z[n] += xk * wk[n];",
                            "for (int64_t n = 0; n < N; ++n)\n                    z[n] += xk * w[n * K + k];"),
    "mlp_skips_rounding": ("y[f] = oracle_bf16_to_f64(yb);", "y[f] = oracle_silu(g[f]) * u[f];"),
}


def _build(tmp_path, name, src_text):
    c = tmp_path / f"{name}.c"
    c.write_text(src_text)
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", str(so), str(c), "-lm"],
                   check=True)
    lib = ctypes.CDLL(str(so))
    p, i64, d = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double
    lib.oracle_swiglu_bf16.argtypes = [p, p, p, i64, i64, i64, p, i64, p, p, p]
    lib.oracle_swiglu_e4m3.argtypes = [p, p, p, d, d, d, i64, i64, i64, p, i64, p, p, p]
    lib.oracle_pack_interleaved_u16.argtypes = [p, p, p, i64, i64]
    lib.oracle_swiglu_interleaved_bf16.argtypes = [p, p, i64, i64, i64, p, i64, p]
    lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_f64.restype = d
    lib.oracle_f64_to_bf16.argtypes = [d]
    lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
    lib.oracle_linear_bf16.argtypes = [p, p, p, i64, i64, i64, p, i64, p]
    lib.oracle_mlp_bf16.argtypes = [p, p, p, p, p, i64, i64, i64, p, i64, p, p]
    return lib


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def _bits(x):
    return si.bits_u16(torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16))


def _y(lib, A, W1, W2):
    M, K = A.shape
    N = W1.shape[1]
    Y = np.empty((M, N))
    lib.oracle_swiglu_bf16(_ptr(A), _ptr(W1), _ptr(W2), M, N, K, None, M, None, None, _ptr(Y))
    return Y


def _y_inter(lib, A, W1, W2):
    M, K = A.shape
    N = W1.shape[1]
    Wf = np.empty((K, 2 * N), dtype=np.uint16)
    lib.oracle_pack_interleaved_u16(_ptr(W1), _ptr(W2), _ptr(Wf), K, N)
    Y = np.empty((M, N))
    lib.oracle_swiglu_interleaved_bf16(_ptr(A), _ptr(Wf), M, N, K, None, M, _ptr(Y))
    return Y


def _pins_pass(lib, golden_dir) -> bool:
    with open(os.path.join(golden_dir, "swiglu_2x2.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        A, W1, W2 = (_bits(case[k]) for k in ("A", "W1", "W2"))
        want = np.array(case["Y_decimal"])
        if not np.allclose(_y(lib, A, W1, W2), want, rtol=0, atol=6e-11):
            return False
        if not np.allclose(_y_inter(lib, A, W1, W2), want, rtol=0, atol=6e-11):
            return False
    A, W1, W2 = si.make_bf16(37, 53, 72, seed=11)
    a, w1, w2 = (t.double().numpy() for t in (A, W1, W2))
    g, u = a @ w1, a @ w2
    want = g / (1.0 + np.exp(-g)) * u
    got = _y(lib, si.bits_u16(A), si.bits_u16(W1), si.bits_u16(W2))
    if not np.allclose(got, want, rtol=1e-9, atol=1e-12 * np.abs(want).max()):
        return False
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().double().numpy()
    dec = np.array([lib.oracle_e4m3_to_f64(int(c)) for c in codes])
    ok = ~np.isnan(ref)
    if not np.array_equal(dec[ok], ref[ok]):
        return False
    return True


def test_unmodified_oracle_passes(tmp_path, golden_dir):
    lib = _build(tmp_path, "orig", open(SRC).read())
    assert _pins_pass(lib, golden_dir)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, golden_dir, name):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation site for {name} not found in the oracle source"
    lib = _build(tmp_path, name, src.replace(old, new, 1))
    assert not _pins_pass(lib, golden_dir), f"pins did not catch mutant {name}"


def _mlp_pins_pass(lib) -> bool:
    # (1) BF16 rounding against torch's float conversion, including exact ties
    rng = np.random.default_rng(1)
    f = rng.standard_normal(4000).astype(np.float32) * np.float32(3.0)
    ties = (rng.integers(0, 2 ** 15, size=200, dtype=np.uint64).astype(np.uint32) << 16 | 0x8000).view(np.float32)
    f = np.concatenate([f, ties[np.isfinite(ties)]])
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([lib.oracle_f64_to_bf16(float(x)) for x in f], dtype=np.uint16)
    if not np.array_equal(got, want):
        return False
    # a double just above a midpoint (not representable in float) rounds up
    if lib.oracle_f64_to_bf16(1.0 + 2 ** -8 + 2 ** -30) != 0x3F81:
        return False
    # (2) linear with a residual against numpy, non-square
    X, W, _ = si.make_bf16(13, 24, 40, seed=7)
    R = si.make_bf16(13, 24, 8, seed=8)[0][:, :8].repeat(1, 3).contiguous()
    x, w, r = si.bits_u16(X), si.bits_u16(W), si.bits_u16(R)
    Z = np.empty((13, 24))
    lib.oracle_linear_bf16(_ptr(x), _ptr(w), _ptr(r), 13, 24, 40, None, 13, _ptr(Z))
    if not np.allclose(Z, X.double().numpy() @ W.double().numpy() + R.double().numpy(),
                       rtol=1e-12, atol=1e-12):
        return False
    # (3) MLP: Y is the BF16 rounding of the SwiGLU output, Z is that Y times W3
    A, W1, W2 = si.make_bf16(9, 32, 24, seed=3)
    W3 = si.make_bf16(1, 24, 32, seed=4)[1]
    a, w1, w2, w3 = (si.bits_u16(t) for t in (A, W1, W2, W3))
    Zm = np.empty((9, 24))
    Yb = np.empty((9, 32), dtype=np.uint16)
    lib.oracle_mlp_bf16(_ptr(a), _ptr(w1), _ptr(w2), _ptr(w3), None, 9, 24, 32, None, 9, _ptr(Zm), _ptr(Yb))
    g = A.double().numpy() @ W1.double().numpy()
    u = A.double().numpy() @ W2.double().numpy()
    y = g / (1 + np.exp(-g)) * u
    y_torch = torch.from_numpy(y).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    if np.mean(Yb != y_torch) > 0.01:       # torch rounds through float: rare near-tie differences
        return False
    yd = torch.from_numpy(Yb.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    return bool(np.allclose(Zm, yd @ W3.double().numpy(), rtol=1e-12, atol=1e-12))


def test_unmodified_oracle_passes_mlp_pins(tmp_path):
    lib = _build(tmp_path, "orig_mlp", open(SRC).read())
    assert _mlp_pins_pass(lib)


@pytest.mark.parametrize("name", sorted(MLP_MUTANTS))
def test_planted_mlp_mistake_is_caught(tmp_path, name):
    src = open(SRC).read()
    old, new = MLP_MUTANTS[name]
    old = old.replace("\\n", "\n")
    new = new.replace("\\n", "\n")
    assert src.count(old) >= 1, f"mutation site for {name} not found in the oracle source"
    lib = _build(tmp_path, name, src.replace(old, new, 1))
    assert not _mlp_pins_pass(lib), f"pins did not catch mutant {name}"


# Planted mistakes in the producer (RMSNorm and E4M3 quantisation), caught by
# the producer pins of test_oracle_producer_pins.py.
PRODUCER_MUTANTS = {
    "eps_outside_sqrt": ("double rms = sqrt(ss / (double)K + eps);", "double rms = sqrt(ss / (double)K) + eps;"),
    "mean_over_k_minus_1": ("double rms = sqrt(ss / (double)K + eps);", "double rms = sqrt(ss / (double)(K - 1) + eps);"),
    "drops_gamma": ("double g = gamma ? oracle_bf16_to_f64(gamma[k]) : 1.0;", "double g = 1.0;"),
    "e4m3_truncates": ("double m = nearbyint(a / ulp); /* exact division by a power of two; ties to even */\n    double r = m * ulp;            /* a < 448",
                       "double m = floor(a / ulp); /* exact division by a power of two; ties to even */\n    double r = m * ulp;            /* a < 448"),
    "e4m3_ties_away": ("double m = nearbyint(a / ulp); /* exact division by a power of two; ties to even */\n    double r = m * ulp;            /* a < 448",
                       "double m = round(a / ulp); /* exact division by a power of two; ties to even */\n    double r = m * ulp;            /* a < 448"),
    "e4m3_no_saturation": ("if (a >= 448.0)\n        return (uint8_t)(sign | 0x7E);", ""),
    "e4m3_subnormal_spacing": ("if (q < -6)\n        q = -6;", "if (q < -7)\n        q = -7;"),
    "scale_not_448": ("float s = (float)(amax / 448.0);", "float s = (float)(amax / 240.0);"),
    "quant_drops_sign": ("q[i] = s > 0.0f ? oracle_f64_to_e4m3(a[i] / (double)s) : 0;",
                         "q[i] = s > 0.0f ? oracle_f64_to_e4m3(fabs(a[i]) / (double)s) : 0;"),
    "quant_decides_in_binary32": ("q[i] = s > 0.0f ? oracle_f64_to_e4m3(a[i] / (double)s) : 0;",
                                  "q[i] = s > 0.0f ? oracle_f64_to_e4m3((double)((float)a[i] / s)) : 0;"),
}


def _build_producer(tmp_path, name, src_text):
    lib = _build(tmp_path, name, src_text)
    p, i64, d = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double
    lib.oracle_f64_to_e4m3_n.argtypes = [p, i64, p]
    lib.oracle_f64_to_e4m3_n.restype = None
    lib.oracle_rmsnorm_bf16.argtypes = [p, p, d, i64, i64, p]
    lib.oracle_quant_e4m3.argtypes = [p, i64, p, p]
    return lib


def test_unmodified_oracle_passes_producer_pins(tmp_path):
    from test_oracle_producer_pins import producer_pin_failures
    lib = _build_producer(tmp_path, "orig_producer", open(SRC).read())
    assert producer_pin_failures(lib) == []


@pytest.mark.parametrize("name", sorted(PRODUCER_MUTANTS))
def test_planted_producer_mistake_is_caught(tmp_path, name):
    from test_oracle_producer_pins import producer_pin_failures
    src = open(SRC).read()
    old, new = PRODUCER_MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not unique in the oracle source"
    lib = _build_producer(tmp_path, name, src.replace(old, new, 1))
    try:
        failures = producer_pin_failures(lib)
    except AssertionError:      # the mutant broke a call outright
        failures = ["call failed"]
    assert failures, f"pins did not catch mutant {name}"


# Planted mistakes in the INT4 weight path, caught by the INT4 pins.
INT4_MUTANTS = {
    "nibble_order": ("uint8_t nib = (n & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);",
                     "uint8_t nib = (n & 1) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4);"),
    "no_sign_extension": ("return (double)(v < 8 ? v : v - 16);", "return (double)v;"),
    "group_by_modulo": ("oracle_bf16_to_f64(S[(k / G) * N + n]);", "oracle_bf16_to_f64(S[(k % G) * N + n]);"),
    "no_bf16_rounding": ("W[k * N + n] = oracle_bf16_to_f64(oracle_f64_to_bf16(p));", "W[k * N + n] = p;"),
}


def _build_int4(tmp_path, name, src_text):
    lib = _build(tmp_path, name, src_text)
    p, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.oracle_int4_value.argtypes = [ctypes.c_uint8]
    lib.oracle_int4_value.restype = ctypes.c_double
    lib.oracle_dequant_int4.argtypes = [p, p, i64, i64, i64, p]
    lib.oracle_swiglu_w4.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, i64, p]
    return lib


def test_unmodified_oracle_passes_int4_pins(tmp_path):
    from test_oracle_int4_pins import int4_pin_failures
    assert int4_pin_failures(_build_int4(tmp_path, "orig_int4", open(SRC).read())) == []


@pytest.mark.parametrize("name", sorted(INT4_MUTANTS))
def test_planted_int4_mistake_is_caught(tmp_path, name):
    from test_oracle_int4_pins import int4_pin_failures
    src = open(SRC).read()
    old, new = INT4_MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not unique in the oracle source"
    lib = _build_int4(tmp_path, name, src.replace(old, new, 1))
    try:
        failures = int4_pin_failures(lib)
    except AssertionError:
        failures = ["call failed"]
    assert failures, f"pins did not catch mutant {name}"


# Planted mistakes in the K-major INT4 arrangement, caught by its pins.
KMAJOR_MUTANTS = {
    "kmajor_natural_nibble_order": ("int64_t nib = (r % 2 == 0) ? r / 2 : 4 + r / 2;", "int64_t nib = r;"),
    "kmajor_column_nibble_swapped": ("(Wq[k * (N / 2) + n / 2] >> (4 * (n % 2))) & 0xF",
                                     "(Wq[k * (N / 2) + n / 2] >> (4 * (1 - n % 2))) & 0xF"),
    "kmajor_halves_swapped": ("Wk[at] |= (uint8_t)(code << (4 * (nib % 2)));",
                              "Wk[at] |= (uint8_t)(code << (4 * (1 - nib % 2)));"),
}


@pytest.mark.parametrize("name", sorted(KMAJOR_MUTANTS))
def test_planted_kmajor_mistake_is_caught(tmp_path, name):
    from test_oracle_int4_pins import kmajor_pin_failures
    src = open(SRC).read()
    old, new = KMAJOR_MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not unique in the oracle source"
    lib = _build(tmp_path, name, src.replace(old, new, 1))
    p, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.oracle_pack_w4_kmajor.argtypes = [p, i64, i64, p]
    lib.oracle_pack_w4_kmajor.restype = ctypes.c_int
    assert kmajor_pin_failures(lib), f"pins did not catch mutant {name}"


# Planted mistakes in the MXFP8 / NVFP4 weight paths, caught by the MX pins.
MX_MUTANTS = {
    "e8m0_bias": ("return ldexp(1.0, (int)e - 127);", "return ldexp(1.0, (int)e - 126);"),
    "mxfp8_block_16": ("* oracle_e8m0_to_f64(S[(k / 32) * N + n]);", "* oracle_e8m0_to_f64(S[(k / 16) * N + n]);"),
    "e2m1_table": ("{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}", "{0.0, 0.5, 1.0, 1.5, 2.0, 4.0, 3.0, 6.0}"),
    "nvfp4_nibble_order": ("uint8_t code = (n & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);",
                           "uint8_t code = (n & 1) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4);"),
    "nvfp4_drops_global": ("* oracle_e4m3_to_f64(S[(k / 16) * N + n]) * global;", "* oracle_e4m3_to_f64(S[(k / 16) * N + n]);"),
    "nvfp4_block_32": ("* oracle_e4m3_to_f64(S[(k / 16) * N + n]) * global;", "* oracle_e4m3_to_f64(S[(k / 32) * N + n]) * global;"),
}


def _build_mx(tmp_path, name, src_text):
    lib = _build(tmp_path, name, src_text)
    p, i64, d = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double
    lib.oracle_e2m1_to_f64.argtypes = [ctypes.c_uint8]
    lib.oracle_e2m1_to_f64.restype = d
    lib.oracle_e8m0_to_f64.argtypes = [ctypes.c_uint8]
    lib.oracle_e8m0_to_f64.restype = d
    lib.oracle_dequant_mxfp8.argtypes = [p, p, i64, i64, p]
    lib.oracle_dequant_nvfp4.argtypes = [p, p, d, i64, i64, p]
    lib.oracle_swiglu_mx.argtypes = [p, ctypes.c_int, p, p, d, p, p, d, i64, i64, i64, p, i64, p]
    return lib


def test_unmodified_oracle_passes_mx_pins(tmp_path):
    from test_oracle_mx_pins import mx_pin_failures
    assert mx_pin_failures(_build_mx(tmp_path, "orig_mx", open(SRC).read())) == []


@pytest.mark.parametrize("name", sorted(MX_MUTANTS))
def test_planted_mx_mistake_is_caught(tmp_path, name):
    from test_oracle_mx_pins import mx_pin_failures
    src = open(SRC).read()
    old, new = MX_MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not unique in the oracle source"
    lib = _build_mx(tmp_path, name, src.replace(old, new, 1))
    try:
        failures = mx_pin_failures(lib)
    except AssertionError:
        failures = ["call failed"]
    assert failures, f"pins did not catch mutant {name}"
