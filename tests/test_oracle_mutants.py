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
