"""Seeded synthetic inputs for the fused SwiGLU projection.

This module is the one piece shared by the CUDA path's tests and benchmark and
by the oracle's checks.  It draws random numbers and converts them to the
storage types; it holds none of the method's arithmetic.

Recipe (the pages name Qwen-2.5 MLP shapes but print no data):
  * a CPU ``torch.Generator`` seeded with ``seed``;
  * W1 = randn(K, N) / sqrt(K), then W2 the same way, then A = randn(M, K),
    all drawn in fp32 in that order and rounded to BF16 (round to nearest even)
    so that, for one seed, the weights are identical across an M sweep;
  * FP8 E4M3 operands: the same fp32 draws, a per-tensor scale
    s = amax(|X|) / 448 (448 is the largest finite E4M3 value), and codes
    q = E4M3(X / s) with round-to-nearest-even and saturation (torch's
    ``float8_e4m3fn`` cast); the operand's value is q * s.

Shapes used by the tests and the benchmark (Qwen-2.5 MLP projections):
  0.5B: K=896,  N=4864;  7B: K=3584, N=18944;  72B: K=8192, N=29568.
"""
from __future__ import annotations

import math

import torch

E4M3_MAX = 448.0

QWEN_SHAPES = {
    "qwen2.5-0.5b": (896, 4864),
    "qwen2.5-7b": (3584, 18944),
    "qwen2.5-72b": (8192, 29568),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def draw_fp32(M: int, N: int, K: int, seed: int):
    """fp32 draws in the fixed order W1, W2, A."""
    g = _gen(seed)
    s = 1.0 / math.sqrt(K) if K > 0 else 1.0
    W1 = torch.randn(K, N, generator=g, dtype=torch.float32) * s
    W2 = torch.randn(K, N, generator=g, dtype=torch.float32) * s
    A = torch.randn(M, K, generator=g, dtype=torch.float32)
    return A, W1, W2


def make_bf16(M: int, N: int, K: int, seed: int):
    """A[M,K], W1[K,N], W2[K,N] as contiguous CPU bfloat16 tensors."""
    A, W1, W2 = draw_fp32(M, N, K, seed)
    return (A.to(torch.bfloat16).contiguous(), W1.to(torch.bfloat16).contiguous(),
            W2.to(torch.bfloat16).contiguous())


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor amax scale and saturating RNE E4M3 codes: returns (q, s).

    s is rounded to float32 (the type a device scale is stored in) before it
    is used, so both sides of a comparison see the same scale value."""
    import numpy as np
    amax = float(x.abs().max()) if x.numel() else 0.0
    s = float(np.float32(amax / E4M3_MAX)) if amax > 0 else 1.0
    q = (x / s).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).contiguous()
    return q, s


def make_e4m3(M: int, N: int, K: int, seed: int):
    """(Aq, W1q, W2q) float8_e4m3fn CPU tensors and their scales (sA, sW1, sW2)."""
    A, W1, W2 = draw_fp32(M, N, K, seed)
    Aq, sA = quantize_e4m3(A)
    W1q, sW1 = quantize_e4m3(W1)
    W2q, sW2 = quantize_e4m3(W2)
    return (Aq, W1q, W2q), (sA, sW1, sW2)


def bits_u16(t: torch.Tensor):
    """Raw 16-bit patterns of a bfloat16 tensor as a numpy uint16 array."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def bits_u8(t: torch.Tensor):
    """Raw 8-bit codes of a float8 tensor as a numpy uint8 array."""
    return t.contiguous().view(torch.uint8).numpy()


def sample_rows(M: int, tile_m: int, n_random: int, seed: int):
    """Row indices for checking a large M on a sample: the first and last row
    of every ``tile_m``-row block, the last row, plus ``n_random`` seeded
    random rows; sorted and unique."""
    import numpy as np
    rows = set()
    for b in range(0, M, tile_m):
        rows.add(b)
        rows.add(min(M - 1, b + tile_m - 1))
    rows.add(M - 1)
    rng = np.random.default_rng(seed)
    if n_random > 0 and M > 0:
        rows.update(int(r) for r in rng.integers(0, M, size=n_random))
    return np.array(sorted(r for r in rows if 0 <= r < M), dtype=np.int64)


def make_producer_inputs(M: int, K: int, seed: int):
    """Inputs of the RMSNorm + E4M3 producer: X [M,K] ~ N(0,1) (the
    distribution of A before quantisation) and gamma [K] = 1 + 0.1 N(0,1), both
    BF16 on the CPU.  gamma is drawn first, then X."""
    g = torch.Generator().manual_seed(seed)
    gamma = (1.0 + 0.1 * torch.randn(K, generator=g)).to(torch.bfloat16)
    X = torch.randn(M, K, generator=g).to(torch.bfloat16).contiguous()
    return X, gamma


def quantize_int4(W: torch.Tensor, G: int = 128):
    """Per-column, per-group symmetric INT4 codes of a [K,N] FP32 weight:
    scale s = max|w| over the group / 7 (rounded to BF16), q = round(w / s)
    clamped to [-8, 7]; returns (packed [K, N/2] uint8 with column n in the low
    nibble when even, scales [K/G, N] BF16)."""
    K, N = W.shape
    Wg = W.reshape(K // G, G, N)
    s = (Wg.abs().amax(dim=1) / 7.0).clamp_min(2.0 ** -100).to(torch.bfloat16)
    q = torch.round(Wg / s.float().unsqueeze(1)).clamp(-8, 7).to(torch.int32).reshape(K, N)
    nib = (q & 0xF).to(torch.uint8)
    packed = (nib[:, 0::2] | (nib[:, 1::2] << 4)).contiguous()
    return packed, s.contiguous()


def make_w4(M: int, N: int, K: int, seed: int, G: int = 128):
    """A [M,K] BF16 and INT4 weights of the same draws as make_bf16:
    returns (A, (W1q, S1), (W2q, S2))."""
    A, W1, W2 = draw_fp32(M, N, K, seed)
    return (A.to(torch.bfloat16).contiguous(), quantize_int4(W1, G), quantize_int4(W2, G))


_E2M1_MAG = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def quantize_mxfp8(W: torch.Tensor):
    """MXFP8 codes of a [K,N] FP32 weight: per block of 32 K rows of a column
    the E8M0 exponent e = 127 + ceil(log2(max|w| / 448)) (the smallest power of
    two that brings the block within E4M3's range), codes = E4M3(w / 2^(e-127))
    (torch's RNE cast).  Returns (codes [K,N] uint8, scales [K/32,N] uint8)."""
    K, N = W.shape
    Wb = W.reshape(K // 32, 32, N)
    amax = Wb.abs().amax(dim=1).clamp_min(2.0 ** -120)
    e = (127 + torch.ceil(torch.log2(amax / 448.0))).clamp(0, 254)
    scale = torch.pow(2.0, e - 127)
    q = (Wb / scale.unsqueeze(1)).clamp(-448, 448).to(torch.float8_e4m3fn)
    return q.reshape(K, N).view(torch.uint8).contiguous(), e.to(torch.uint8).contiguous()


def quantize_nvfp4(W: torch.Tensor):
    """NVFP4 codes of a [K,N] FP32 weight: a per-tensor FP32 scale
    g = max|w| / (6 * 448); per block of 16 K rows of a column the E4M3 scale
    s = E4M3(max|w| / 6 / g); codes = the E2M1 value nearest |w| / (s g) (ties
    to the smaller magnitude), with the sign bit, packed two per byte along N.
    Returns (packed [K, N/2] uint8, scales [K/16, N] uint8, g)."""
    K, N = W.shape
    g = float(W.abs().max()) / (6.0 * 448.0)
    g = g if g > 0 else 1.0
    Wb = W.reshape(K // 16, 16, N)
    amax = Wb.abs().amax(dim=1)
    s8 = (amax / 6.0 / g).clamp(max=448.0).to(torch.float8_e4m3fn)
    s = s8.float().clamp_min(2.0 ** -9)
    x = (Wb / (s.unsqueeze(1) * g)).abs()
    mags = torch.tensor(_E2M1_MAG)
    code = (x.unsqueeze(-1) - mags).abs().argmin(dim=-1).to(torch.uint8)
    code = code | ((Wb < 0).to(torch.uint8) << 3)
    code = code.reshape(K, N)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).contiguous()
    return packed, s8.view(torch.uint8).contiguous(), g


def make_mx(M: int, N: int, K: int, seed: int, fmt: str):
    """A [M,K] BF16 and the weights of the BF16 recipe's draws in MXFP8
    (fmt "mxfp8": (codes, scales)) or NVFP4 ("nvfp4": (codes, scales, g))."""
    A, W1, W2 = draw_fp32(M, N, K, seed)
    q = quantize_mxfp8 if fmt == "mxfp8" else quantize_nvfp4
    return A.to(torch.bfloat16).contiguous(), q(W1), q(W2)
