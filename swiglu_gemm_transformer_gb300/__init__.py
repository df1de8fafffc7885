"""Python binding of the GB300 fused SwiGLU library (argument marshalling only).

Every function here forwards to the C ABI of ``libswiglu_gb300.so`` (declared
in ``include/swiglu.h``) with the same name; all arithmetic runs in the CUDA
kernels.  There is no CPU fallback: if the library is missing or a call fails
the function raises.

    Y = SiLU(A @ W1) * (A @ W2)   A: [M,K] bf16, W1/W2: [K,N] bf16, Y: [M,N] bf16

PyTorch supplies device memory and the current CUDA stream.
"""
from __future__ import annotations

import ctypes
import functools
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libswiglu_gb300.so")

OK, ERR_INVALID_ARG, ERR_MISALIGNED, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = range(6)
VARIANT_AUTO, VARIANT_1SM_N128, VARIANT_1SM_N64, VARIANT_2SM_N128, VARIANT_1SM_N32 = range(5)
VARIANT_1SM_N64_SK2 = 9   # 5-8 are retired numbers the library rejects
VARIANT_2SM_SWAP = 10
VARIANTS = {"auto": VARIANT_AUTO, "1sm_n128": VARIANT_1SM_N128, "1sm_n64": VARIANT_1SM_N64,
            "2sm_n128": VARIANT_2SM_N128, "1sm_n32": VARIANT_1SM_N32,
            "1sm_n64_sk2": VARIANT_1SM_N64_SK2, "2sm_swap": VARIANT_2SM_SWAP}

EXPORTS = {
    # name: (argtypes, restype)
    "swiglu_fused": ("pppp lll p", ctypes.c_int),
    "swiglu_fused_ex": ("pppp lll i p", ctypes.c_int),
    "swiglu_fused_interleaved": ("ppp lll p", ctypes.c_int),
    "swiglu_fused_interleaved_ex": ("ppp lll i p", ctypes.c_int),
    "swiglu_pack_interleaved": ("ppp ll p", ctypes.c_int),
    "swiglu_fused_fp8": ("ppp ppp p lll p", ctypes.c_int),
    "swiglu_fused_interleaved_fp8": ("pp ppp p lll p", ctypes.c_int),
    "swiglu_pack_interleaved_fp8": ("ppp ll p", ctypes.c_int),
    "swiglu_rmsnorm_quant_fp8": ("pp f pp ll p", ctypes.c_int),
    "swiglu_quant_fp8": ("ppp ll p", ctypes.c_int),
    "swiglu_fused_w4": ("ppppp p lll l p", ctypes.c_int),
    "swiglu_pack_w4_kmajor": ("pp ll p", ctypes.c_int),
    "swiglu_fused_w4_kmajor": ("ppppp p lll l p", ctypes.c_int),
    "swiglu_fused_mxfp8": ("ppppp p lll p", ctypes.c_int),
    "swiglu_fused_nvfp4": ("pppppppp lll p", ctypes.c_int),
    "swiglu_fused_nvfp4_kmajor": ("pppppppp lll p", ctypes.c_int),
    "swiglu_fused_mxfp8_kmajor": ("ppppp p lll p", ctypes.c_int),
    "swiglu_linear_workspace_size": ("lll", ctypes.c_uint64),
    "swiglu_linear": ("pppp lll pQ p", ctypes.c_int),
    "swiglu_mlp_workspace_size": ("lll", ctypes.c_uint64),
    "swiglu_mlp": ("ppppp p lll pQ p", ctypes.c_int),
    "swiglu_mlp_noalloc_scratch_bytes": ("", ctypes.c_uint64),
    "swiglu_mlp_noalloc": ("ppppp p lll p", ctypes.c_int),
    "swiglu_select_variant": ("lll i", ctypes.c_int),
    "swiglu_select_weight_kernel": ("ll", ctypes.c_int),
    "swiglu_set_weight_kernel": ("i", ctypes.c_int),
    "swiglu_set_pair_schedule": ("i", ctypes.c_int),
    "swiglu_variant_name": ("i", ctypes.c_char_p),
    "swiglu_status_string": ("i", ctypes.c_char_p),
    "swiglu_device_status": ("p P", ctypes.c_int),
    "swiglu_set_wait_timeout_ns": ("Q", ctypes.c_int),
    "swiglu_set_weights_read_only": ("i", ctypes.c_int),
    "swiglu_selftest_wait_timeout": ("I p", ctypes.c_int),
}
_CT = {"p": ctypes.c_void_p, "l": ctypes.c_int64, "f": ctypes.c_float, "i": ctypes.c_int32, "Q": ctypes.c_uint64,
       "I": ctypes.c_uint32, "P": ctypes.POINTER(ctypes.c_uint32)}

_lock = threading.Lock()
_lib = None


class SwigluError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} (status {status})")


def lib() -> ctypes.CDLL:
    """The loaded C library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        l = ctypes.CDLL(LIB_PATH)
        for name, (sig, res) in EXPORTS.items():
            f = getattr(l, name)
            f.argtypes = [_CT[c] for c in sig.replace(" ", "")]
            f.restype = res
        _lib = l
        return l


def status_string(status: int) -> str:
    try:
        return lib().swiglu_status_string(int(status)).decode()
    except Exception:  # library not loadable: still give a message
        return f"status {status}"


def variant_name(v: int) -> str:
    return lib().swiglu_variant_name(int(v)).decode()


def _check(fn: str, rc: int):
    if rc != OK:
        raise SwigluError(fn, rc)


def _stream(stream):
    import torch
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _on_tensor_device(fn):
    """Run an entry point with the tensors' CUDA device current (the library
    works on the current device: its launches, per-device state and the
    no-allocation scratch area); all tensor arguments must share one device."""
    @functools.wraps(fn)
    def call(*args, **kw):
        import torch
        ts = [a for a in list(args) + list(kw.values()) if isinstance(a, torch.Tensor)]
        devs = {t.device for t in ts}
        if len(devs) > 1:
            raise ValueError(f"{fn.__name__}: tensors on several devices: {sorted(map(str, devs))}")
        if ts and ts[0].is_cuda:
            with torch.cuda.device(ts[0].device):
                return fn(*args, **kw)
        return fn(*args, **kw)
    return call


def _need(t, name, dtype=None, ndim=2):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-D tensor")
    return t


@_on_tensor_device
def swiglu_fused(A, W1, W2, Y=None, *, variant: int = VARIANT_AUTO, stream=None):
    """Y = SiLU(A @ W1) * (A @ W2) with separate [K,N] weights; returns Y."""
    import torch
    bf = torch.bfloat16
    _need(A, "A", bf), _need(W1, "W1", bf), _need(W2, "W2", bf)
    M, K = A.shape
    if W1.shape[0] != K or W2.shape != W1.shape:
        raise ValueError(f"shape mismatch: A {tuple(A.shape)}, W1 {tuple(W1.shape)}, W2 {tuple(W2.shape)}")
    N = W1.shape[1]
    if Y is None:
        Y = torch.empty((M, N), dtype=bf, device=A.device)
    else:
        _need(Y, "Y", bf)
        if tuple(Y.shape) != (M, N):
            raise ValueError("Y must be [M, N]")
    rc = lib().swiglu_fused_ex(A.data_ptr(), W1.data_ptr(), W2.data_ptr(), Y.data_ptr(),
                               M, N, K, int(variant), _stream(stream))
    _check("swiglu_fused", rc)
    return Y


@_on_tensor_device
def swiglu_fused_interleaved(A, Wfused, Y=None, *, variant: int = VARIANT_AUTO, stream=None):
    """Y[m,n] = SiLU(D[m,2n]) * D[m,2n+1] with D = A @ Wfused, Wfused [K,2N]; returns Y."""
    import torch
    bf = torch.bfloat16
    _need(A, "A", bf), _need(Wfused, "Wfused", bf)
    M, K = A.shape
    if Wfused.shape[0] != K or Wfused.shape[1] % 2:
        raise ValueError(f"shape mismatch: A {tuple(A.shape)}, Wfused {tuple(Wfused.shape)}")
    N = Wfused.shape[1] // 2
    if Y is None:
        Y = torch.empty((M, N), dtype=bf, device=A.device)
    else:
        _need(Y, "Y", bf)
        if tuple(Y.shape) != (M, N):
            raise ValueError("Y must be [M, N]")
    rc = lib().swiglu_fused_interleaved_ex(A.data_ptr(), Wfused.data_ptr(), Y.data_ptr(),
                                           M, N, K, int(variant), _stream(stream))
    _check("swiglu_fused_interleaved", rc)
    return Y


@_on_tensor_device
def swiglu_pack_interleaved(W1, W2, Wfused=None, *, stream=None):
    """Wfused[k,2n] = W1[k,n], Wfused[k,2n+1] = W2[k,n]; returns Wfused [K,2N]."""
    import torch
    if W1.dtype != W2.dtype or W1.shape != W2.shape:
        raise ValueError("W1 and W2 must match in shape and dtype")
    _need(W1, "W1", torch.bfloat16), _need(W2, "W2", torch.bfloat16)
    K, N = W1.shape
    if Wfused is None:
        Wfused = torch.empty((K, 2 * N), dtype=W1.dtype, device=W1.device)
    else:
        _need(Wfused, "Wfused", W1.dtype)
        if tuple(Wfused.shape) != (K, 2 * N):
            raise ValueError("Wfused must be [K, 2N]")
    rc = lib().swiglu_pack_interleaved(W1.data_ptr(), W2.data_ptr(), Wfused.data_ptr(), K, N,
                                       _stream(stream))
    _check("swiglu_pack_interleaved", rc)
    return Wfused


def _fp8(t, name, ndim=2):
    import torch
    return _need(t, name, torch.float8_e4m3fn, ndim)


def _scale(s, name):
    import torch
    if not isinstance(s, torch.Tensor) or not s.is_cuda or s.dtype != torch.float32 or s.numel() != 1:
        raise TypeError(f"{name} must be a one-element float32 CUDA tensor")
    return s.data_ptr()


@_on_tensor_device
def swiglu_fused_fp8(Aq, W1t, W2t, sA, sW1, sW2, Y=None, *, stream=None):
    """Y = SiLU(sA*sW1 * Aq@W1t.T) * (sA*sW2 * Aq@W2t.T); Aq [M,K], W1t/W2t [N,K] E4M3."""
    import torch
    _fp8(Aq, "Aq"), _fp8(W1t, "W1t"), _fp8(W2t, "W2t")
    M, K = Aq.shape
    N = W1t.shape[0]
    if W1t.shape[1] != K or W2t.shape != W1t.shape:
        raise ValueError(f"shape mismatch: Aq {tuple(Aq.shape)}, W1t {tuple(W1t.shape)}, W2t {tuple(W2t.shape)}")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=Aq.device)
    else:
        _need(Y, "Y", torch.bfloat16)
        if tuple(Y.shape) != (M, N):
            raise ValueError("Y must be [M, N]")
    rc = lib().swiglu_fused_fp8(Aq.data_ptr(), W1t.data_ptr(), W2t.data_ptr(), _scale(sA, "sA"),
                                _scale(sW1, "sW1"), _scale(sW2, "sW2"), Y.data_ptr(), M, N, K,
                                _stream(stream))
    _check("swiglu_fused_fp8", rc)
    return Y


@_on_tensor_device
def swiglu_fused_interleaved_fp8(Aq, Wfused_t, sA, sW1, sW2, Y=None, *, stream=None):
    """FP8 interleaved form: Wfused_t [2N,K] (even rows gate, odd rows up)."""
    import torch
    _fp8(Aq, "Aq"), _fp8(Wfused_t, "Wfused_t")
    M, K = Aq.shape
    if Wfused_t.shape[1] != K or Wfused_t.shape[0] % 2:
        raise ValueError(f"shape mismatch: Aq {tuple(Aq.shape)}, Wfused_t {tuple(Wfused_t.shape)}")
    N = Wfused_t.shape[0] // 2
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=Aq.device)
    else:
        _need(Y, "Y", torch.bfloat16)
        if tuple(Y.shape) != (M, N):
            raise ValueError("Y must be [M, N]")
    rc = lib().swiglu_fused_interleaved_fp8(Aq.data_ptr(), Wfused_t.data_ptr(), _scale(sA, "sA"),
                                            _scale(sW1, "sW1"), _scale(sW2, "sW2"), Y.data_ptr(),
                                            M, N, K, _stream(stream))
    _check("swiglu_fused_interleaved_fp8", rc)
    return Y


@_on_tensor_device
def swiglu_pack_interleaved_fp8(W1t, W2t, Wfused_t=None, *, stream=None):
    """Wfused_t[2n,:] = W1t[n,:], Wfused_t[2n+1,:] = W2t[n,:] (E4M3, K-major)."""
    import torch
    _fp8(W1t, "W1t"), _fp8(W2t, "W2t")
    if W1t.shape != W2t.shape:
        raise ValueError("W1t and W2t must match in shape")
    N, K = W1t.shape
    if Wfused_t is None:
        Wfused_t = torch.empty((2 * N, K), dtype=W1t.dtype, device=W1t.device)
    else:
        _fp8(Wfused_t, "Wfused_t")
        if tuple(Wfused_t.shape) != (2 * N, K):
            raise ValueError("Wfused_t must be [2N, K]")
    rc = lib().swiglu_pack_interleaved_fp8(W1t.data_ptr(), W2t.data_ptr(), Wfused_t.data_ptr(),
                                           N, K, _stream(stream))
    _check("swiglu_pack_interleaved_fp8", rc)
    return Wfused_t


def _quant_outputs(X, Xq, s):
    import torch
    if Xq is None:
        Xq = torch.empty(X.shape, dtype=torch.float8_e4m3fn, device=X.device)
    else:
        _fp8(Xq, "Xq")
        if Xq.shape != X.shape:
            raise ValueError("the codes must have the shape of X")
    if s is None:
        s = torch.empty(1, dtype=torch.float32, device=X.device)
    return Xq, s


@_on_tensor_device
def swiglu_rmsnorm_quant_fp8(X, gamma=None, eps: float = 1e-6, Aq=None, sA=None, *, stream=None):
    """RMSNorm of the rows of X (BF16 [M,K], gamma BF16 [K] or None) then
    per-tensor E4M3 quantisation; returns (Aq, sA) for swiglu_fused_fp8."""
    import torch
    _need(X, "X", torch.bfloat16)
    M, K = X.shape
    if gamma is not None:
        _need(gamma, "gamma", torch.bfloat16, ndim=1)
        if gamma.numel() != K:
            raise ValueError("gamma must have K elements")
    Aq, sA = _quant_outputs(X, Aq, sA)
    rc = lib().swiglu_rmsnorm_quant_fp8(X.data_ptr(), gamma.data_ptr() if gamma is not None else None,
                                        float(eps), Aq.data_ptr(), _scale(sA, "sA"), M, K,
                                        _stream(stream))
    _check("swiglu_rmsnorm_quant_fp8", rc)
    return Aq, sA


@_on_tensor_device
def swiglu_quant_fp8(X, Xq=None, s=None, *, stream=None):
    """Per-tensor E4M3 quantisation of a BF16 [M,K] matrix; returns (Xq, s)."""
    import torch
    _need(X, "X", torch.bfloat16)
    M, K = X.shape
    Xq, s = _quant_outputs(X, Xq, s)
    rc = lib().swiglu_quant_fp8(X.data_ptr(), Xq.data_ptr(), _scale(s, "s"), M, K, _stream(stream))
    _check("swiglu_quant_fp8", rc)
    return Xq, s


@_on_tensor_device
def swiglu_fused_w4(A, W1q, S1, W2q, S2, Y=None, *, group: int = 128, stream=None):
    """Y = SiLU(A @ W1) * (A @ W2) with INT4 weights: W1q/W2q uint8 [K, N/2]
    (two codes per byte along N), S1/S2 BF16 [K/group, N]."""
    import torch
    _need(A, "A", torch.bfloat16)
    _need(W1q, "W1q", torch.uint8), _need(W2q, "W2q", torch.uint8)
    _need(S1, "S1", torch.bfloat16), _need(S2, "S2", torch.bfloat16)
    M, K = A.shape
    N = 2 * W1q.shape[1]
    if W1q.shape[0] != K or W2q.shape != W1q.shape or S1.shape != (K // group, N) or S2.shape != S1.shape:
        raise ValueError("shape mismatch")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    else:
        _need(Y, "Y", torch.bfloat16)
        if tuple(Y.shape) != (M, N):
            raise ValueError("Y must be [M, N]")
    rc = lib().swiglu_fused_w4(A.data_ptr(), W1q.data_ptr(), S1.data_ptr(), W2q.data_ptr(),
                               S2.data_ptr(), Y.data_ptr(), M, N, K, int(group), _stream(stream))
    _check("swiglu_fused_w4", rc)
    return Y


@_on_tensor_device
def swiglu_pack_w4_kmajor(Wq, Wk=None, *, stream=None):
    """INT4 codes [K, N/2] (swiglu_fused_w4's layout) -> the K-major layout
    [N, K/2] that swiglu_fused_w4_kmajor reads."""
    import torch
    _need(Wq, "Wq", torch.uint8)
    K, half = Wq.shape
    N = 2 * half
    if Wk is None:
        Wk = torch.empty((N, K // 2), dtype=torch.uint8, device=Wq.device)
    else:
        _need(Wk, "Wk", torch.uint8)
        if tuple(Wk.shape) != (N, K // 2):
            raise ValueError("Wk must be [N, K/2]")
    _check("swiglu_pack_w4_kmajor",
           lib().swiglu_pack_w4_kmajor(Wq.data_ptr(), Wk.data_ptr(), K, N, _stream(stream)))
    return Wk


@_on_tensor_device
def swiglu_fused_w4_kmajor(A, W1k, S1, W2k, S2, Y=None, *, group: int = 128, stream=None):
    """swiglu_fused_w4 with the codes in the K-major layout [N, K/2] of
    swiglu_pack_w4_kmajor (weights decoded into tensor memory)."""
    import torch
    _need(A, "A", torch.bfloat16)
    _need(W1k, "W1k", torch.uint8), _need(W2k, "W2k", torch.uint8)
    _need(S1, "S1", torch.bfloat16), _need(S2, "S2", torch.bfloat16)
    M, K = A.shape
    N = W1k.shape[0]
    if W1k.shape[1] * 2 != K or W2k.shape != W1k.shape or S1.shape != (K // group, N) or S2.shape != S1.shape:
        raise ValueError("shape mismatch")
    Y = _out(A, N, Y)
    rc = lib().swiglu_fused_w4_kmajor(A.data_ptr(), W1k.data_ptr(), S1.data_ptr(), W2k.data_ptr(),
                                      S2.data_ptr(), Y.data_ptr(), M, N, K, int(group), _stream(stream))
    _check("swiglu_fused_w4_kmajor", rc)
    return Y


def _out(A, N, Y):
    import torch
    M = A.shape[0]
    if Y is None:
        return torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _need(Y, "Y", torch.bfloat16)
    if tuple(Y.shape) != (M, N):
        raise ValueError("Y must be [M, N]")
    return Y


@_on_tensor_device
def swiglu_fused_mxfp8(A, C1, S1, C2, S2, Y=None, *, stream=None):
    """Y = SiLU(A @ W1) * (A @ W2), W = E4M3(C) * 2^(S - 127) per 32 K rows:
    C1/C2 uint8 [K,N], S1/S2 uint8 [K/32,N]."""
    import torch
    _need(A, "A", torch.bfloat16)
    for t, n in ((C1, "C1"), (C2, "C2"), (S1, "S1"), (S2, "S2")):
        _need(t, n, torch.uint8)
    M, K = A.shape
    N = C1.shape[1]
    if C1.shape != (K, N) or C2.shape != C1.shape or S1.shape != (K // 32, N) or S2.shape != S1.shape:
        raise ValueError("shape mismatch")
    Y = _out(A, N, Y)
    rc = lib().swiglu_fused_mxfp8(A.data_ptr(), C1.data_ptr(), S1.data_ptr(), C2.data_ptr(),
                                  S2.data_ptr(), Y.data_ptr(), M, N, K, _stream(stream))
    _check("swiglu_fused_mxfp8", rc)
    return Y


@_on_tensor_device
def swiglu_fused_mxfp8_kmajor(A, C1k, S1, C2k, S2, Y=None, *, stream=None):
    """swiglu_fused_mxfp8 with the codes K-major: C1k/C2k uint8 [N,K], the
    transposes of the [K,N] codes (weights decoded into tensor memory)."""
    import torch
    _need(A, "A", torch.bfloat16)
    for t, n in ((C1k, "C1k"), (C2k, "C2k"), (S1, "S1"), (S2, "S2")):
        _need(t, n, torch.uint8)
    M, K = A.shape
    N = C1k.shape[0]
    if C1k.shape != (N, K) or C2k.shape != C1k.shape or S1.shape != (K // 32, N) or S2.shape != S1.shape:
        raise ValueError("shape mismatch")
    Y = _out(A, N, Y)
    rc = lib().swiglu_fused_mxfp8_kmajor(A.data_ptr(), C1k.data_ptr(), S1.data_ptr(), C2k.data_ptr(),
                                         S2.data_ptr(), Y.data_ptr(), M, N, K, _stream(stream))
    _check("swiglu_fused_mxfp8_kmajor", rc)
    return Y


@_on_tensor_device
def swiglu_fused_nvfp4(A, C1, S1, g1, C2, S2, g2, Y=None, *, stream=None):
    """Y = SiLU(A @ W1) * (A @ W2), W = E2M1(C) * E4M3(S) * g per 16 K rows:
    C1/C2 uint8 [K,N/2] (two codes per byte), S1/S2 uint8 [K/16,N] E4M3,
    g1/g2 one-element float32 CUDA tensors."""
    import torch
    _need(A, "A", torch.bfloat16)
    for t, n in ((C1, "C1"), (C2, "C2"), (S1, "S1"), (S2, "S2")):
        _need(t, n, torch.uint8)
    M, K = A.shape
    N = 2 * C1.shape[1]
    if C1.shape[0] != K or C2.shape != C1.shape or S1.shape != (K // 16, N) or S2.shape != S1.shape:
        raise ValueError("shape mismatch")
    Y = _out(A, N, Y)
    rc = lib().swiglu_fused_nvfp4(A.data_ptr(), C1.data_ptr(), S1.data_ptr(), _scale(g1, "g1"),
                                  C2.data_ptr(), S2.data_ptr(), _scale(g2, "g2"), Y.data_ptr(),
                                  M, N, K, _stream(stream))
    _check("swiglu_fused_nvfp4", rc)
    return Y


@_on_tensor_device
def swiglu_fused_nvfp4_kmajor(A, C1k, S1, g1, C2k, S2, g2, Y=None, *, stream=None):
    """swiglu_fused_nvfp4 with the codes in the K-major layout [N, K/2] of
    swiglu_pack_w4_kmajor (weights decoded into tensor memory)."""
    import torch
    _need(A, "A", torch.bfloat16)
    for t, n in ((C1k, "C1k"), (C2k, "C2k"), (S1, "S1"), (S2, "S2")):
        _need(t, n, torch.uint8)
    M, K = A.shape
    N = C1k.shape[0]
    if C1k.shape[1] * 2 != K or C2k.shape != C1k.shape or S1.shape != (K // 16, N) or S2.shape != S1.shape:
        raise ValueError("shape mismatch")
    Y = _out(A, N, Y)
    rc = lib().swiglu_fused_nvfp4_kmajor(A.data_ptr(), C1k.data_ptr(), S1.data_ptr(), _scale(g1, "g1"),
                                         C2k.data_ptr(), S2.data_ptr(), _scale(g2, "g2"), Y.data_ptr(),
                                         M, N, K, _stream(stream))
    _check("swiglu_fused_nvfp4_kmajor", rc)
    return Y


def _workspace(nbytes, device, workspace):
    import torch
    if workspace is None:
        if nbytes == 0:
            return None, 0
        workspace = torch.empty(int(nbytes), dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


@_on_tensor_device
def swiglu_linear(X, W, R=None, Z=None, *, workspace=None, stream=None):
    """Z = X @ W (+ R); X [M,K], W [K,N], R [M,N] or None; BF16.

    ``workspace`` (a CUDA tensor) holds split-K partial sums for small M; when
    None, one of swiglu_linear_workspace_size() bytes is allocated here."""
    import torch
    bf = torch.bfloat16
    _need(X, "X", bf), _need(W, "W", bf)
    M, K = X.shape
    if W.shape[0] != K:
        raise ValueError(f"shape mismatch: X {tuple(X.shape)}, W {tuple(W.shape)}")
    N = W.shape[1]
    if R is not None:
        _need(R, "R", bf)
        if tuple(R.shape) != (M, N):
            raise ValueError("R must be [M, N]")
    if Z is None:
        Z = torch.empty((M, N), dtype=bf, device=X.device)
    else:
        _need(Z, "Z", bf)
        if tuple(Z.shape) != (M, N):
            raise ValueError("Z must be [M, N]")
    ws, nbytes = _workspace(lib().swiglu_linear_workspace_size(M, N, K), X.device, workspace)
    rc = lib().swiglu_linear(X.data_ptr(), W.data_ptr(), R.data_ptr() if R is not None else None,
                             Z.data_ptr(), M, N, K, ws.data_ptr() if ws is not None else None,
                             nbytes, _stream(stream))
    _check("swiglu_linear", rc)
    return Z


@_on_tensor_device
def swiglu_mlp(A, W1, W2, W3, R=None, Z=None, *, workspace=None, stream=None):
    """Z = BF16(SiLU(A @ W1) * (A @ W2)) @ W3 (+ R); A [M,H], W1/W2 [H,F], W3 [F,H]."""
    import torch
    bf = torch.bfloat16
    for t, n in ((A, "A"), (W1, "W1"), (W2, "W2"), (W3, "W3")):
        _need(t, n, bf)
    M, H = A.shape
    F = W1.shape[1]
    if W1.shape != (H, F) or W2.shape != (H, F) or W3.shape != (F, H):
        raise ValueError("shape mismatch: A [M,H], W1/W2 [H,F], W3 [F,H]")
    if R is not None:
        _need(R, "R", bf)
        if tuple(R.shape) != (M, H):
            raise ValueError("R must be [M, H]")
    if Z is None:
        Z = torch.empty((M, H), dtype=bf, device=A.device)
    ws, nbytes = _workspace(lib().swiglu_mlp_workspace_size(M, H, F), A.device, workspace)
    rc = lib().swiglu_mlp(A.data_ptr(), W1.data_ptr(), W2.data_ptr(), W3.data_ptr(),
                          R.data_ptr() if R is not None else None, Z.data_ptr(), M, H, F,
                          ws.data_ptr() if ws is not None else None, nbytes, _stream(stream))
    _check("swiglu_mlp", rc)
    return Z


@_on_tensor_device
def swiglu_mlp_noalloc(A, W1, W2, W3, R, Z, *, stream=None):
    """swiglu_mlp without any device allocation, for callers that may not
    allocate: Y lives in the library's fixed 32 MiB scratch area.  Z must be
    given; calls on one device whose GPU work overlaps must be serialised."""
    bf = __import__("torch").bfloat16
    for t, n in ((A, "A"), (W1, "W1"), (W2, "W2"), (W3, "W3"), (Z, "Z")):
        _need(t, n, bf)
    M, H = A.shape
    F = W1.shape[1]
    if W1.shape != (H, F) or W2.shape != (H, F) or W3.shape != (F, H) or tuple(Z.shape) != (M, H):
        raise ValueError("shape mismatch: A [M,H], W1/W2 [H,F], W3 [F,H], Z [M,H]")
    if R is not None:
        _need(R, "R", bf)
    rc = lib().swiglu_mlp_noalloc(A.data_ptr(), W1.data_ptr(), W2.data_ptr(), W3.data_ptr(),
                                  R.data_ptr() if R is not None else None, Z.data_ptr(), M, H, F,
                                  _stream(stream))
    _check("swiglu_mlp_noalloc", rc)
    return Z


def swiglu_select_variant(M: int, N: int, K: int, interleaved: bool = False) -> int:
    return lib().swiglu_select_variant(M, N, K, 1 if interleaved else 0)


WEIGHT_KERNELS = ("sk2", "wide", "wide_mb2")


def swiglu_select_weight_kernel(M: int, N: int) -> int:
    """0 split-K cluster kernel, 1 wide kernel, 2 wide kernel with two row
    blocks per CTA: the kernel the INT4/MXFP8/NVFP4 entry points run."""
    return lib().swiglu_select_weight_kernel(M, N)


def swiglu_set_weight_kernel(kernel: int):
    """Force the weight-format kernel (0 split-K, 1 wide, 2 wide with two row
    blocks per CTA) for later calls, or -1 for the library's choice."""
    _check("swiglu_set_weight_kernel", lib().swiglu_set_weight_kernel(int(kernel)))


def swiglu_set_pair_schedule(dynamic: int):
    """Tile schedule of the CTA-pair kernels when a call has more units than
    resident pairs: 1 dynamic (cluster launch control, the default), 0 static."""
    _check("swiglu_set_pair_schedule", lib().swiglu_set_pair_schedule(int(dynamic)))


def swiglu_device_status(stream=None):
    """Synchronise the stream; return (status, detail) and clear the device error word."""
    detail = ctypes.c_uint32(0)
    rc = lib().swiglu_device_status(_stream(stream), ctypes.byref(detail))
    return rc, detail.value


def swiglu_set_wait_timeout_ns(ns: int):
    _check("swiglu_set_wait_timeout_ns", lib().swiglu_set_wait_timeout_ns(int(ns)))


def swiglu_set_weights_read_only(on: bool):
    """Promise that no earlier work on a stream writes a later call's weights
    (model parameters): lets the kernels start streaming weights before the
    preceding kernel finishes."""
    _check("swiglu_set_weights_read_only", lib().swiglu_set_weights_read_only(1 if on else 0))


def swiglu_selftest_wait_timeout(timeout_us: int, stream=None):
    _check("swiglu_selftest_wait_timeout",
           lib().swiglu_selftest_wait_timeout(int(timeout_us), _stream(stream)))
