"""CPU oracle for the fused SwiGLU projection Y = SiLU(A x W1) (.) (A x W2).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The product path never
does, and this package never imports the product.  The arithmetic lives in
``swiglu_oracle.c`` (plain C, double precision); this module builds it with gcc
and wraps it with ctypes over numpy arrays.

Source of the method: page "Riepilogo Tecnico: Sovrapposizione delle
Attivazioni a Livello di Tile per l'Inferenza Efficiente di LLM" (gist.science
paper 2607.02521), section "Definizione del Problema" (the formula) and section
"Metodologia", item 2 (the interleaved W_fused layout and the pair step).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "swiglu_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile swiglu_oracle.c into liboracle.so (gcc, OpenMP over rows)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        d = ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = d
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_f64.restype = d
        lib.oracle_silu.argtypes = [d]
        lib.oracle_silu.restype = d
        lib.oracle_swiglu_bf16.argtypes = [p, p, p, i64, i64, i64, p, i64, p, p, p]
        lib.oracle_swiglu_bf16.restype = ctypes.c_int
        lib.oracle_swiglu_e4m3.argtypes = [p, p, p, d, d, d, i64, i64, i64, p, i64, p, p, p]
        lib.oracle_swiglu_e4m3.restype = ctypes.c_int
        lib.oracle_pack_interleaved_u16.argtypes = [p, p, p, i64, i64]
        lib.oracle_pack_interleaved_u16.restype = None
        lib.oracle_pack_interleaved_u8.argtypes = [p, p, p, i64, i64]
        lib.oracle_pack_interleaved_u8.restype = None
        lib.oracle_swiglu_interleaved_bf16.argtypes = [p, p, i64, i64, i64, p, i64, p]
        lib.oracle_swiglu_interleaved_bf16.restype = ctypes.c_int
        lib.oracle_f64_to_bf16.argtypes = [d]
        lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
        lib.oracle_linear_bf16.argtypes = [p, p, p, i64, i64, i64, p, i64, p]
        lib.oracle_linear_bf16.restype = ctypes.c_int
        lib.oracle_mlp_bf16.argtypes = [p, p, p, p, p, i64, i64, i64, p, i64, p, p]
        lib.oracle_mlp_bf16.restype = ctypes.c_int
        lib.oracle_f64_to_e4m3.argtypes = [d]
        lib.oracle_f64_to_e4m3.restype = ctypes.c_uint8
        lib.oracle_f64_to_e4m3_n.argtypes = [p, i64, p]
        lib.oracle_f64_to_e4m3_n.restype = None
        lib.oracle_rmsnorm_bf16.argtypes = [p, p, d, i64, i64, p]
        lib.oracle_rmsnorm_bf16.restype = ctypes.c_int
        lib.oracle_quant_e4m3.argtypes = [p, i64, p, p]
        lib.oracle_quant_e4m3.restype = ctypes.c_int
        lib.oracle_int4_value.argtypes = [ctypes.c_uint8]
        lib.oracle_int4_value.restype = d
        lib.oracle_dequant_int4.argtypes = [p, p, i64, i64, i64, p]
        lib.oracle_dequant_int4.restype = ctypes.c_int
        lib.oracle_swiglu_w4.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, i64, p]
        lib.oracle_pack_w4_kmajor.argtypes = [p, i64, i64, p]
        lib.oracle_pack_w4_kmajor.restype = ctypes.c_int
        lib.oracle_swiglu_w4.restype = ctypes.c_int
        lib.oracle_e2m1_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_to_f64.restype = d
        lib.oracle_e8m0_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e8m0_to_f64.restype = d
        lib.oracle_dequant_mxfp8.argtypes = [p, p, i64, i64, p]
        lib.oracle_dequant_mxfp8.restype = ctypes.c_int
        lib.oracle_dequant_nvfp4.argtypes = [p, p, d, i64, i64, p]
        lib.oracle_dequant_nvfp4.restype = ctypes.c_int
        lib.oracle_swiglu_mx.argtypes = [p, ctypes.c_int, p, p, d, p, p, d, i64, i64, i64, p, i64, p]
        lib.oracle_swiglu_mx.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _u16(x) -> np.ndarray:
    """Raw BF16 bit patterns as a C-contiguous uint16 array."""
    a = np.ascontiguousarray(x)
    if a.dtype != np.uint16:
        raise TypeError(f"expected BF16 bit patterns as uint16, got {a.dtype}")
    return a


def _u8(x) -> np.ndarray:
    a = np.ascontiguousarray(x)
    if a.dtype != np.uint8:
        raise TypeError(f"expected E4M3 codes as uint8, got {a.dtype}")
    return a


def _rows(rows, M):
    if rows is None:
        return None, M
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return r, int(r.size)


def bf16_to_f64(bits: int) -> float:
    return _load().oracle_bf16_to_f64(int(bits))


def e4m3_to_f64(code: int) -> float:
    return _load().oracle_e4m3_to_f64(int(code))


def silu(x: float) -> float:
    return _load().oracle_silu(float(x))


def swiglu_bf16(A, W1, W2, rows=None, with_gate_up: bool = False):
    """Y[r, :] = SiLU(A[m_r] W1) * (A[m_r] W2) in double for BF16 inputs.

    A [M,K], W1/W2 [K,N] are uint16 arrays of BF16 bit patterns (row-major).
    ``rows`` selects rows of A (default: all).  Returns Y [nrows, N] float64,
    or (G, U, Y) when ``with_gate_up``.
    """
    A, W1, W2 = _u16(A), _u16(W1), _u16(W2)
    M, K = A.shape
    K2, N = W1.shape
    if K2 != K or W2.shape != (K, N):
        raise ValueError("shape mismatch")
    r, nr = _rows(rows, M)
    Y = np.empty((nr, N), dtype=np.float64)
    G = np.empty_like(Y) if with_gate_up else None
    U = np.empty_like(Y) if with_gate_up else None
    rc = _load().oracle_swiglu_bf16(
        _ptr(A), _ptr(W1), _ptr(W2), M, N, K,
        _ptr(r) if r is not None else None, nr,
        _ptr(G) if G is not None else None, _ptr(U) if U is not None else None, _ptr(Y))
    if rc != 0:
        raise ValueError("oracle_swiglu_bf16 failed (bad row index or out of memory)")
    return (G, U, Y) if with_gate_up else Y


def swiglu_e4m3(Aq, W1q, W2q, sA: float, sW1: float, sW2: float, rows=None,
                with_gate_up: bool = False):
    """The definition on dequantised FP8 E4M3 operands (value = code * scale)."""
    Aq, W1q, W2q = _u8(Aq), _u8(W1q), _u8(W2q)
    M, K = Aq.shape
    K2, N = W1q.shape
    if K2 != K or W2q.shape != (K, N):
        raise ValueError("shape mismatch")
    r, nr = _rows(rows, M)
    Y = np.empty((nr, N), dtype=np.float64)
    G = np.empty_like(Y) if with_gate_up else None
    U = np.empty_like(Y) if with_gate_up else None
    rc = _load().oracle_swiglu_e4m3(
        _ptr(Aq), _ptr(W1q), _ptr(W2q), float(sA), float(sW1), float(sW2), M, N, K,
        _ptr(r) if r is not None else None, nr,
        _ptr(G) if G is not None else None, _ptr(U) if U is not None else None, _ptr(Y))
    if rc != 0:
        raise ValueError("oracle_swiglu_e4m3 failed")
    return (G, U, Y) if with_gate_up else Y


def pack_interleaved(W1, W2) -> np.ndarray:
    """W_fused[k, 2n] = W1[k, n], W_fused[k, 2n+1] = W2[k, n] (uint16 or uint8 codes)."""
    W1 = np.ascontiguousarray(W1)
    W2 = np.ascontiguousarray(W2)
    if W1.shape != W2.shape or W1.dtype != W2.dtype:
        raise ValueError("W1 and W2 must match in shape and dtype")
    K, N = W1.shape
    Wf = np.empty((K, 2 * N), dtype=W1.dtype)
    if W1.dtype == np.uint16:
        _load().oracle_pack_interleaved_u16(_ptr(W1), _ptr(W2), _ptr(Wf), K, N)
    elif W1.dtype == np.uint8:
        _load().oracle_pack_interleaved_u8(_ptr(W1), _ptr(W2), _ptr(Wf), K, N)
    else:
        raise TypeError("expected uint16 (BF16) or uint8 (FP8) codes")
    return Wf


def swiglu_interleaved_bf16(A, Wf, rows=None) -> np.ndarray:
    """D = A x W_fused, then Y[m,n] = SiLU(D[m,2n]) * D[m,2n+1], in double."""
    A, Wf = _u16(A), _u16(Wf)
    M, K = A.shape
    K2, N2 = Wf.shape
    if K2 != K or N2 % 2:
        raise ValueError("shape mismatch")
    N = N2 // 2
    r, nr = _rows(rows, M)
    Y = np.empty((nr, N), dtype=np.float64)
    rc = _load().oracle_swiglu_interleaved_bf16(
        _ptr(A), _ptr(Wf), M, N, K, _ptr(r) if r is not None else None, nr, _ptr(Y))
    if rc != 0:
        raise ValueError("oracle_swiglu_interleaved_bf16 failed")
    return Y


def f64_to_bf16(x: float) -> int:
    """Round to the nearest BF16 (ties to even); returns the 16-bit pattern."""
    return int(_load().oracle_f64_to_bf16(float(x)))


def linear_bf16(X, W, R=None, rows=None) -> np.ndarray:
    """Z = X W (+ R) in double; X [M,K], W [K,N], R [M,N] as BF16 bit patterns."""
    X, W = _u16(X), _u16(W)
    M, K = X.shape
    K2, N = W.shape
    if K2 != K:
        raise ValueError("shape mismatch")
    if R is not None:
        R = _u16(R)
        if R.shape != (M, N):
            raise ValueError("R must be [M, N]")
    r, nr = _rows(rows, M)
    Z = np.empty((nr, N), dtype=np.float64)
    rc = _load().oracle_linear_bf16(_ptr(X), _ptr(W), _ptr(R) if R is not None else None,
                                    M, N, K, _ptr(r) if r is not None else None, nr, _ptr(Z))
    if rc != 0:
        raise ValueError("oracle_linear_bf16 failed")
    return Z


def mlp_bf16(A, W1, W2, W3, R=None, rows=None, with_y: bool = False):
    """The SwiGLU MLP block: Y = BF16(SiLU(A W1) * (A W2)), Z = Y W3 (+ R).

    A [M,H], W1/W2 [H,F], W3 [F,H], R [M,H] as BF16 bit patterns.  Returns Z
    [nrows,H] float64, or (Z, Ybits) with the rounded Y as uint16 patterns."""
    A, W1, W2, W3 = _u16(A), _u16(W1), _u16(W2), _u16(W3)
    M, H = A.shape
    H2, F = W1.shape
    if H2 != H or W2.shape != (H, F) or W3.shape != (F, H):
        raise ValueError("shape mismatch")
    if R is not None:
        R = _u16(R)
        if R.shape != (M, H):
            raise ValueError("R must be [M, H]")
    r, nr = _rows(rows, M)
    Z = np.empty((nr, H), dtype=np.float64)
    Y = np.empty((nr, F), dtype=np.uint16) if with_y else None
    rc = _load().oracle_mlp_bf16(_ptr(A), _ptr(W1), _ptr(W2), _ptr(W3),
                                 _ptr(R) if R is not None else None, M, H, F,
                                 _ptr(r) if r is not None else None, nr, _ptr(Z),
                                 _ptr(Y) if Y is not None else None)
    if rc != 0:
        raise ValueError("oracle_mlp_bf16 failed")
    return (Z, Y) if with_y else Z


from .check import parity_report, assert_parity, bf16_rounding_slack  # noqa: E402,F401


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Decode an array of BF16 bit patterns (exact)."""
    b = _u16(bits)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def mlp_rounding_slack(A, W1, W2, W3, rows=None) -> np.ndarray:
    """Per element of the MLP block's Z [nrows, H]: how far Z may move when
    every element of Y whose exact value lies within the kernel's FP32 error
    bound of a BF16 rounding midpoint rounds to the other neighbour:
    sum over f of slack(Y[m,f]) * |W3[f,h]| (``bf16_rounding_slack``).  G, U
    and Y come from the definition; the sums of absolute products from the
    definition on the inputs' absolute values (sign bits cleared)."""
    A, W1, W2, W3 = _u16(A), _u16(W1), _u16(W2), _u16(W3)
    G, U, Y = swiglu_bf16(A, W1, W2, rows=rows, with_gate_up=True)
    clear = lambda b: np.ascontiguousarray(b & np.uint16(0x7FFF))
    Ga, Ua, _ = swiglu_bf16(clear(A), clear(W1), clear(W2), rows=rows, with_gate_up=True)
    s = bf16_rounding_slack(Y, G, U, Ga, Ua, A.shape[1])
    return s @ np.abs(bf16_bits_to_f64(W3))


# ---- the producer: RMSNorm and per-tensor E4M3 quantisation ----------------

def f64_to_e4m3(x) -> np.ndarray:
    """Round each value to FP8 E4M3 (ties to even, saturating at +-448);
    returns the codes as uint8 with the input's shape."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    q = np.empty(a.shape, dtype=np.uint8)
    _load().oracle_f64_to_e4m3_n(_ptr(a), a.size, _ptr(q))
    return q


def rmsnorm_bf16(X, gamma=None, eps: float = 1e-6) -> np.ndarray:
    """a[m,k] = x[m,k] * gamma[k] / sqrt(mean_k x[m,k]^2 + eps), in double.
    X [M,K] and gamma [K] are BF16 bit patterns (gamma None = all ones)."""
    X = _u16(X)
    M, K = X.shape
    g = None if gamma is None else _u16(gamma)
    if g is not None and g.shape != (K,):
        raise ValueError("gamma must have K elements")
    A = np.empty((M, K), dtype=np.float64)
    rc = _load().oracle_rmsnorm_bf16(_ptr(X), _ptr(g) if g is not None else None, float(eps),
                                     M, K, _ptr(A))
    if rc != 0:
        raise ValueError("oracle_rmsnorm_bf16 failed (K = 0 or eps < 0)")
    return A


def quant_e4m3(a):
    """Per-tensor quantisation: returns (scale, codes) with scale =
    float32(max|a| / 448) and codes = E4M3(a / scale) (all zero if scale is 0)."""
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    q = np.empty(a.shape, dtype=np.uint8)
    s = np.zeros(1, dtype=np.float32)
    rc = _load().oracle_quant_e4m3(_ptr(a), a.size, _ptr(s), _ptr(q))
    if rc != 0:
        raise ValueError("oracle_quant_e4m3 failed (NaN input)")
    return float(s[0]), q


def rmsnorm_quant_e4m3(X, gamma=None, eps: float = 1e-6):
    """RMSNorm then per-tensor E4M3 quantisation: returns (scale, codes [M,K])."""
    return quant_e4m3(rmsnorm_bf16(X, gamma, eps))


# ---- weight-only INT4 -----------------------------------------------------

def int4_value(nibble: int) -> float:
    """Signed 4-bit two's complement value of a nibble."""
    return _load().oracle_int4_value(int(nibble))


def dequant_int4(Wq, S, G: int) -> np.ndarray:
    """W[k,n] = BF16(q[k,n] * S[k // G, n]) in double: Wq [K, N/2] bytes (column
    n in the low nibble when even, high when odd), S [K/G, N] BF16 bits."""
    Wq = _u8(Wq)
    S = _u16(S)
    K, half = Wq.shape
    N = 2 * half
    W = np.empty((K, N), dtype=np.float64)
    rc = _load().oracle_dequant_int4(_ptr(Wq), _ptr(S), K, N, int(G), _ptr(W))
    if rc != 0:
        raise ValueError("oracle_dequant_int4: K must be a multiple of G")
    return W


def pack_w4_kmajor(Wq) -> np.ndarray:
    """The K-major arrangement [N, K/2] of INT4 codes given as [K, N/2]."""
    Wq = _u8(Wq)
    K, half = Wq.shape
    Wk = np.empty((2 * half, K // 2), dtype=np.uint8)
    if _load().oracle_pack_w4_kmajor(_ptr(Wq), K, 2 * half, _ptr(Wk)) != 0:
        raise ValueError("oracle_pack_w4_kmajor: K must be a multiple of 8")
    return Wk


def swiglu_w4(A, W1q, S1, W2q, S2, G: int, rows=None) -> np.ndarray:
    """The definition with INT4 weights (dequantised as in dequant_int4)."""
    A, W1q, W2q, S1, S2 = _u16(A), _u8(W1q), _u8(W2q), _u16(S1), _u16(S2)
    M, K = A.shape
    N = 2 * W1q.shape[1]
    r, nr = _rows(rows, M)
    Y = np.empty((nr, N), dtype=np.float64)
    rc = _load().oracle_swiglu_w4(_ptr(A), _ptr(W1q), _ptr(S1), _ptr(W2q), _ptr(S2), M, N, K,
                                  int(G), _ptr(r) if r is not None else None, nr, _ptr(Y))
    if rc != 0:
        raise ValueError("oracle_swiglu_w4 failed")
    return Y


# ---- weight-only MXFP8 and NVFP4 -------------------------------------------

def e2m1_to_f64(code: int) -> float:
    return _load().oracle_e2m1_to_f64(int(code))


def e8m0_to_f64(e: int) -> float:
    return _load().oracle_e8m0_to_f64(int(e))


def dequant_mxfp8(C, S) -> np.ndarray:
    """W[k,n] = BF16(E4M3(C[k,n]) * 2^(S[k//32, n] - 127)); C [K,N], S [K/32,N] bytes."""
    C, S = _u8(C), _u8(S)
    K, N = C.shape
    W = np.empty((K, N), dtype=np.float64)
    if _load().oracle_dequant_mxfp8(_ptr(C), _ptr(S), K, N, _ptr(W)) != 0:
        raise ValueError("oracle_dequant_mxfp8: K must be a multiple of 32")
    return W


def dequant_nvfp4(C, S, global_scale: float) -> np.ndarray:
    """W[k,n] = E2M1(c[k,n]) * E4M3(S[k//16, n]) * global; C [K, N/2] packed (even
    column in the low nibble), S [K/16, N] E4M3 bytes."""
    C, S = _u8(C), _u8(S)
    K, half = C.shape
    W = np.empty((K, 2 * half), dtype=np.float64)
    if _load().oracle_dequant_nvfp4(_ptr(C), _ptr(S), float(global_scale), K, 2 * half, _ptr(W)) != 0:
        raise ValueError("oracle_dequant_nvfp4: K must be a multiple of 16")
    return W


def swiglu_mx(A, fmt: str, w1, w2, rows=None) -> np.ndarray:
    """The definition with block-scaled weights: fmt "mxfp8" with w = (C, S), or
    "nvfp4" with w = (C, S, global)."""
    A = _u16(A)
    M, K = A.shape
    f = 0 if fmt == "mxfp8" else 1
    C1, S1 = _u8(w1[0]), _u8(w1[1])
    C2, S2 = _u8(w2[0]), _u8(w2[1])
    g1 = float(w1[2]) if f else 1.0
    g2 = float(w2[2]) if f else 1.0
    N = C1.shape[1] * (2 if f else 1)
    r, nr = _rows(rows, M)
    Y = np.empty((nr, N), dtype=np.float64)
    rc = _load().oracle_swiglu_mx(_ptr(A), f, _ptr(C1), _ptr(S1), g1, _ptr(C2), _ptr(S2), g2,
                                  M, N, K, _ptr(r) if r is not None else None, nr, _ptr(Y))
    if rc != 0:
        raise ValueError("oracle_swiglu_mx failed")
    return Y
