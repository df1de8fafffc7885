"""Pins for the weight-only MXFP8 and NVFP4 part of the oracle.

The GEMM page names the formats (benchmark paragraph) without defining them;
the oracle follows the OCP Microscaling specification (MXFP8: E4M3 codes, one
E8M0 scale per 32 K rows) and NVIDIA's NVFP4 (E2M1 codes, one E4M3 scale per 16
K rows, one FP32 scale per tensor).  What pins it, other than itself:

* hand-worked cases (``tests/golden/mx_cases.json``);
* the E2M1 table against the bit-field formula written out separately
  ((-1)^s * (e == 0 ? m/2 : (1 + m/2) 2^(e-1))), and E8M0 against ldexp;
* block broadcast: changing the scale of one block changes exactly its rows
  (32 for MXFP8, 16 for NVFP4), and the NVFP4 per-tensor scale is linear;
* the SwiGLU result on the decoded weights against numpy in float64.

``mx_pin_failures(lib)`` runs them against a loaded oracle library.
"""
import ctypes
import json
import math
import os

import numpy as np
import torch

import oracle
import swiglu_inputs as si

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "mx_cases.json")


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def _mx(lib, C, S):
    C, S = np.ascontiguousarray(C, np.uint8), np.ascontiguousarray(S, np.uint8)
    K, N = C.shape
    W = np.empty((K, N))
    assert lib.oracle_dequant_mxfp8(_ptr(C), _ptr(S), K, N, _ptr(W)) == 0
    return W


def _nv(lib, C, S, g):
    C, S = np.ascontiguousarray(C, np.uint8), np.ascontiguousarray(S, np.uint8)
    K, half = C.shape
    W = np.empty((K, 2 * half))
    assert lib.oracle_dequant_nvfp4(_ptr(C), _ptr(S), float(g), K, 2 * half, _ptr(W)) == 0
    return W


def mx_pin_failures(lib):
    bad = []
    with open(GOLDEN) as f:
        gold = json.load(f)
    c = gold["mxfp8"]
    C = np.tile(np.array(c["code_col"], np.uint8), (c["K"], 1))
    W = _mx(lib, C, np.array(c["scales"], np.uint8))
    if not np.array_equal(W, np.repeat(np.array(c["W_block"]), 32, axis=0)):
        bad.append("golden mxfp8")
    c = gold["nvfp4"]
    W = _nv(lib, np.full((c["K"], c["N"] // 2), c["byte"], np.uint8), np.array([c["scales"]], np.uint8), c["global"])
    if not np.array_equal(W, np.tile(np.array(c["W_row"]), (c["K"], 1))):
        bad.append("golden nvfp4")
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        want = (-1.0) ** s * (m / 2 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1))
        if lib.oracle_e2m1_to_f64(code) != want:
            bad.append(f"e2m1 code {code}")
            break
    for e in range(255):
        if lib.oracle_e8m0_to_f64(e) != math.ldexp(1.0, e - 127):
            bad.append(f"e8m0 {e}")
            break
    if not math.isnan(lib.oracle_e8m0_to_f64(255)):
        bad.append("e8m0 255 is not NaN")
    rng = np.random.default_rng(4)
    # MXFP8 block broadcast: rows 32..63 follow scale row 1 only
    C = rng.choice(np.array([0x30, 0x38, 0x40, 0xB8, 0xC4], np.uint8), size=(96, 4))
    S = np.full((3, 4), 127, np.uint8)
    W0 = _mx(lib, C, S)
    S[1] = 128
    W1 = _mx(lib, C, S)
    if not (np.array_equal(W1[32:64], 2 * W0[32:64]) and np.array_equal(W1[:32], W0[:32])
            and np.array_equal(W1[64:], W0[64:])):
        bad.append("mxfp8 block is not 32 rows")
    # NVFP4 block broadcast (16 rows) and global linearity
    Cn = rng.integers(0, 256, size=(48, 3), dtype=np.uint8)
    Sn = np.full((3, 6), 0x38, np.uint8)          # E4M3 1.0
    V0 = _nv(lib, Cn, Sn, 1.0)
    Sn[1] = 0x40                                    # E4M3 2.0
    V1 = _nv(lib, Cn, Sn, 1.0)
    if not (np.array_equal(V1[16:32], 2 * V0[16:32]) and np.array_equal(V1[:16], V0[:16])
            and np.array_equal(V1[32:], V0[32:])):
        bad.append("nvfp4 block is not 16 rows")
    if not np.array_equal(_nv(lib, Cn, Sn, 0.25), 0.25 * V1):
        bad.append("nvfp4 global scale is not a factor")
    lo = np.array([lib.oracle_e2m1_to_f64(int(b) & 15) for b in Cn[:, 0]])
    if not np.array_equal(V0[:, 0], lo):
        bad.append("nvfp4 even column is not the low nibble")
    # SwiGLU on decoded weights against numpy
    A = si.bits_u16(torch.from_numpy(rng.standard_normal((5, 96)).astype(np.float32)).to(torch.bfloat16))
    C2 = rng.choice(np.array([0x30, 0x34, 0xB0], np.uint8), size=(96, 4))
    Y = np.empty((5, 4))
    S3 = np.full((3, 4), 125, np.uint8)
    assert lib.oracle_swiglu_mx(_ptr(A), 0, _ptr(C), _ptr(S3), 1.0, _ptr(C2), _ptr(S3), 1.0,
                                5, 4, 96, None, 5, _ptr(Y)) == 0
    a = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).double().numpy()
    g, u = a @ _mx(lib, C, S3), a @ _mx(lib, C2, S3)
    if not np.allclose(Y, g / (1 + np.exp(-g)) * u, rtol=1e-12, atol=1e-12):
        bad.append("SwiGLU on decoded MXFP8 weights")
    return bad


def test_mx_pins():
    assert mx_pin_failures(oracle._load()) == []


def test_mx_recipes_round_trip():
    """The input recipes reproduce their FP32 draws within one element step
    (a check of the inputs, not of the method)."""
    _, W1, _ = si.draw_fp32(1, 64, 128, seed=12)
    C, S = si.quantize_mxfp8(W1)
    Wm = oracle.dequant_mxfp8(C.numpy(), S.numpy())
    assert np.all(np.abs(Wm - W1.double().numpy()) <= 2.0 ** -3 * np.abs(W1.double().numpy()) + 1e-6)
    Cn, Sn, g = si.quantize_nvfp4(W1)
    Wn = oracle.dequant_nvfp4(Cn.numpy(), Sn.numpy(), g)
    blk = np.repeat(np.abs(W1.double().numpy()).reshape(8, 16, 64).max(axis=1), 16, axis=0)
    assert np.all(np.abs(Wn - W1.double().numpy()) <= 0.26 * blk + 1e-6)
