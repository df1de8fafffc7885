// weight_decode.cuh -- decoding of low-precision weight codes into the BF16
// operand tiles the tcgen05 MMA reads, for the kernels that take INT4, MXFP8
// or NVFP4 weights (the weight-only formats: A stays BF16).
//
// One call decodes [64 K rows x COLS columns] of one weight matrix.  The
// output is COLS/64 "atoms" of [64 rows x 64 columns] BF16, ATOM_BYTES apart,
// each in the layout a TMA copy with the 128-byte swizzle would leave: row k
// at 128 k bytes, its 16-byte chunk c (columns 8c .. 8c+7) at position
// c ^ (k % 8).  The MMA's shared-memory descriptors are the BF16 ones.
//
// Formats (codes row-major along N, scales one per column and block of K rows):
//   WF_INT4  : signed 4-bit two's complement, two per byte (even column in the
//              low nibble); BF16 scale per group of >= 64 rows (one scale row
//              per 64-row stage).  Weight = BF16(q * s), rounded once.
//   WF_MXFP8 : E4M3 codes; E8M0 scale (2^(e-127)) per 32 rows.  Weight =
//              BF16(E4M3 * 2^(e-127)) (exact in binary32, rounded once).
//   WF_NVFP4 : E2M1 codes, two per byte; E4M3 scale per 16 rows.  Weight =
//              E2M1 * E4M3, exact in BF16 (the per-tensor FP32 scale is applied
//              to the accumulated sums by the kernel).
//
// Thread `tid` of NTHREADS owns one 8-column chunk j of every row it visits
// (rows rr, rr + R, rr + 2R, ... with R = NTHREADS / (COLS / 8)): it loads its
// chunk's scales once per 64-row stage (once per scale row for MXFP8/NVFP4),
// and a warp's code loads and tile stores each cover contiguous bytes.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace swiglu {

enum : int { WF_BF16 = 0, WF_INT4 = 1, WF_MXFP8 = 2, WF_NVFP4 = 3 };

template <int WF>
struct WFormat {
  static constexpr int CODE_BITS = WF == WF_MXFP8 ? 8 : 4;
  static constexpr int SCALE_ROWS = WF == WF_INT4 ? 1 : WF == WF_MXFP8 ? 2 : 4;  // per 64 rows
  static constexpr int SCALE_BYTES = WF == WF_INT4 ? 2 : 1;                      // per scale
};

// Two E4M3 codes (low byte, high byte of `two`) to two floats, exactly.
__device__ __forceinline__ static float2 e4m3x2_to_float2(uint32_t two) {
  uint32_t h2;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
      : "=r"(h2)
      : "r"(two));
  return __half22float2(*reinterpret_cast<const __half2 *>(&h2));
}

// E2M1 code (1 sign, 2 exponent bits with bias 1, 1 mantissa bit) to float,
// exactly: 2^(e-1) (1 + m/2) for e > 0, m/2 for e = 0.
__device__ __forceinline__ static float e2m1_to_float(uint32_t code) {
  const uint32_t e = (code >> 1) & 3u, m = code & 1u;
  const uint32_t mag = e ? (((126u + e) << 23) | (m << 22)) : (m ? 0x3F000000u : 0u);
  return __uint_as_float(mag | ((code & 8u) << 28));
}

__device__ __forceinline__ static uint32_t bf16x2_bits(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// raw_w: the [64 x COLS] codes (COLS * CODE_BITS / 8 bytes per row);
// raw_s: the stage's scale rows (COLS scales each); tile: the first atom.
template <int WF, int COLS, int NTHREADS, int ATOM_BYTES>
__device__ __forceinline__ static void decode_weights(const uint8_t *raw_w, const uint8_t *raw_s,
                                                      uint8_t *tile, int tid) {
  constexpr int CHUNKS = COLS / 8;            // 8-column chunks per row
  constexpr int R = NTHREADS / CHUNKS;        // rows per pass
  constexpr int ROW_BYTES = COLS * WFormat<WF>::CODE_BITS / 8;
  static_assert(NTHREADS % CHUNKS == 0 && 64 % R == 0, "thread mapping");
  const int j = tid % CHUNKS;
  const int rr = tid / CHUNKS;
  uint8_t *atom = tile + (j / 8) * ATOM_BYTES;
  const int c = j % 8;
  if (WF == WF_INT4) {
    // flipping each code's sign bit gives n = q + 8; the BF16 pattern
    // 0x4300 | n is exactly 128 + n; minus 136 is q; one BF16 multiply by the
    // adjacent scale pair rounds q * s once
    const uint4 sv = *reinterpret_cast<const uint4 *>(raw_s + j * 16);
    const __nv_bfloat162 sc[4] = {*reinterpret_cast<const __nv_bfloat162 *>(&sv.x),
                                  *reinterpret_cast<const __nv_bfloat162 *>(&sv.y),
                                  *reinterpret_cast<const __nv_bfloat162 *>(&sv.z),
                                  *reinterpret_cast<const __nv_bfloat162 *>(&sv.w)};
    const __nv_bfloat162 k136 = __floats2bfloat162_rn(136.0f, 136.0f);
#pragma unroll
    for (int k = rr; k < 64; k += R) {
      const uint32_t codes =
          *reinterpret_cast<const uint32_t *>(raw_w + k * ROW_BYTES + j * 4) ^ 0x88888888u;
      uint32_t out[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t w = ((codes >> (8 * b)) & 0xFu) | (((codes >> (8 * b + 4)) & 0xFu) << 16) |
                           0x43004300u;
        const __nv_bfloat162 q = __hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&w), k136);
        const __nv_bfloat162 v = __hmul2(q, sc[b]);
        out[b] = *reinterpret_cast<const uint32_t *>(&v);
      }
      *reinterpret_cast<uint4 *>(atom + k * 128 + ((c ^ (k & 7)) * 16)) =
          make_uint4(out[0], out[1], out[2], out[3]);
    }
  } else if (WF == WF_MXFP8) {
#pragma unroll
    for (int k = rr; k < 64; k += R) {
      const uint2 codes = *reinterpret_cast<const uint2 *>(raw_w + k * ROW_BYTES + j * 8);
      const uint2 sc = *reinterpret_cast<const uint2 *>(raw_s + (k >> 5) * COLS + j * 8);
      uint32_t out[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t cw = b < 2 ? codes.x : codes.y, sw = b < 2 ? sc.x : sc.y;
        const int sh = 16 * (b & 1);
        const float2 f = e4m3x2_to_float2((cw >> sh) & 0xFFFFu);
        const uint32_t e0 = (sw >> sh) & 0xFFu, e1 = (sw >> (sh + 8)) & 0xFFu;
        // 2^(e-127) from its exponent bits; e = 0 is 2^-127, a binary32 subnormal
        const float p0 = __uint_as_float(e0 ? e0 << 23 : 0x00400000u);
        const float p1 = __uint_as_float(e1 ? e1 << 23 : 0x00400000u);
        out[b] = bf16x2_bits(__fmul_rn(f.x, p0), __fmul_rn(f.y, p1));
      }
      *reinterpret_cast<uint4 *>(atom + k * 128 + ((c ^ (k & 7)) * 16)) =
          make_uint4(out[0], out[1], out[2], out[3]);
    }
  } else if (WF == WF_NVFP4) {
#pragma unroll
    for (int k = rr; k < 64; k += R) {
      const uint32_t codes = *reinterpret_cast<const uint32_t *>(raw_w + k * ROW_BYTES + j * 4);
      const uint2 sc = *reinterpret_cast<const uint2 *>(raw_s + (k >> 4) * COLS + j * 8);
      uint32_t out[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float2 s2 = e4m3x2_to_float2(((b < 2 ? sc.x : sc.y) >> (16 * (b & 1))) & 0xFFFFu);
        const float v0 = e2m1_to_float((codes >> (8 * b)) & 0xFu);
        const float v1 = e2m1_to_float((codes >> (8 * b + 4)) & 0xFu);
        out[b] = bf16x2_bits(__fmul_rn(v0, s2.x), __fmul_rn(v1, s2.y));
      }
      *reinterpret_cast<uint4 *>(atom + k * 128 + ((c ^ (k & 7)) * 16)) =
          make_uint4(out[0], out[1], out[2], out[3]);
    }
  }
}

}  // namespace swiglu
