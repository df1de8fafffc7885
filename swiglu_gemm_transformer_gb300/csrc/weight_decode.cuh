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
// PAIRED (4-bit codes: INT4, NVFP4): the eight columns of a chunk are written
// in the order 0 4 1 5 2 6 3 7, so that each BF16 pair (c, c + 4) comes out of
// shifts and logic operations on the whole code word; the MMA's output columns
// then carry the same order, which the epilogue undoes.
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
// All of a thread's code words (and scales) are loaded before any is decoded,
// so the shared-memory loads overlap and the decode chains of different rows
// are independent.
template <int WF, int COLS, int NTHREADS, int ATOM_BYTES, bool PAIRED = false>
__device__ __forceinline__ static void decode_weights(const uint8_t *raw_w, const uint8_t *raw_s,
                                                      uint8_t *tile, int tid) {
  constexpr int CHUNKS = COLS / 8;            // 8-column chunks per row
  constexpr int R = NTHREADS / CHUNKS;        // rows per pass
  constexpr int ROWS = 64 / R;                // rows per thread
  constexpr int ROW_BYTES = COLS * WFormat<WF>::CODE_BITS / 8;
  constexpr int SR = WFormat<WF>::SCALE_ROWS;  // scale rows per 64 rows
  static_assert(NTHREADS % CHUNKS == 0 && 64 % R == 0, "thread mapping");
  static_assert(R <= 64 / SR, "a pass stays within one scale row");
  const int j = tid % CHUNKS;
  const int rr = tid / CHUNKS;
  uint8_t *atom = tile + (j / 8) * ATOM_BYTES;
  const int c = j % 8;
  // row rr + i R lies in scale row i R SR / 64 (rr < R <= 64 / SR)
  auto store = [&](int i, uint32_t o0, uint32_t o1, uint32_t o2, uint32_t o3) {
    const int k = rr + i * R;
    *reinterpret_cast<uint4 *>(atom + k * 128 + ((c ^ (k & 7)) * 16)) = make_uint4(o0, o1, o2, o3);
  };
  if (WF == WF_INT4 && PAIRED) {
    // nibble c of a code word is column c; (word >> 4b) & 0x000F000F holds
    // columns b and b + 4 in the two halves.  With the sign bits flipped
    // (n = q + 8) and 0x4300 or-ed in, each half is the BF16 value 128 + n;
    // minus 136 is q; one BF16 multiply by the scale pair rounds q * s once.
    const uint4 sv = *reinterpret_cast<const uint4 *>(raw_s + j * 16);
    uint32_t sp[4];  // scale pairs (b, b + 4)
    sp[0] = __byte_perm(sv.x, sv.z, 0x5410);
    sp[1] = __byte_perm(sv.x, sv.z, 0x7632);
    sp[2] = __byte_perm(sv.y, sv.w, 0x5410);
    sp[3] = __byte_perm(sv.y, sv.w, 0x7632);
    const __nv_bfloat162 k136 = __floats2bfloat162_rn(136.0f, 136.0f);
    uint32_t cw[ROWS];
#pragma unroll
    for (int i = 0; i < ROWS; ++i)
      cw[i] = *reinterpret_cast<const uint32_t *>(raw_w + (rr + i * R) * ROW_BYTES + j * 4);
#pragma unroll
    for (int i = 0; i < ROWS; ++i) {
      uint32_t out[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t w = ((cw[i] >> (4 * b)) & 0x000F000Fu) ^ 0x43084308u;
        const __nv_bfloat162 q = __hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&w), k136);
        const __nv_bfloat162 v = __hmul2(q, *reinterpret_cast<const __nv_bfloat162 *>(&sp[b]));
        out[b] = *reinterpret_cast<const uint32_t *>(&v);
      }
      store(i, out[0], out[1], out[2], out[3]);
    }
  } else if (WF == WF_NVFP4 && PAIRED) {
    // An E2M1 code s e1 e0 m with its three magnitude bits placed at BF16 bits
    // 8..6 (the exponent field's two low bits and the mantissa's top bit) and
    // its sign at bit 15 is the BF16 number E2M1 * 2^-126 (e = 0, m = 1 is the
    // subnormal 2^-127); a multiply by 2^126 and one by the E4M3 scale are
    // both exact (at most 2 + 4 significant bits, far inside BF16's range).
    // Columns b and b + 4 of a code word sit 16 bits apart, so one pair of
    // shifts and two logic operations build both halves.
    uint32_t sp[SR][4];  // scale pairs (b, b + 4) per scale row, BF16
#pragma unroll
    for (int s = 0; s < SR; ++s) {
      const uint2 sv = *reinterpret_cast<const uint2 *>(raw_s + s * COLS + j * 8);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float2 f = e4m3x2_to_float2(__byte_perm(sv.x, sv.y, b | ((4 + b) << 4)) & 0xFFFFu);
        sp[s][b] = bf16x2_bits(f.x, f.y);
      }
    }
    const uint32_t k126 = 0x7E807E80u;  // 2^126 in both halves
    uint32_t cw[ROWS];
#pragma unroll
    for (int i = 0; i < ROWS; ++i)
      cw[i] = *reinterpret_cast<const uint32_t *>(raw_w + (rr + i * R) * ROW_BYTES + j * 4);
#pragma unroll
    for (int i = 0; i < ROWS; ++i) {
      const int s = i * R * SR / 64;
      const uint32_t x = cw[i];
      uint32_t out[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        // magnitude bits of nibbles b, b + 4 to bits 8..6 and 24..22; sign bits to 15 and 31
        const uint32_t mag = (b == 0 ? x << 6 : b == 1 ? x << 2 : b == 2 ? x >> 2 : x >> 6) & 0x01C001C0u;
        const uint32_t sgn = (b == 0 ? x << 12 : b == 1 ? x << 8 : b == 2 ? x << 4 : x) & 0x80008000u;
        const uint32_t y = mag | sgn;
        const __nv_bfloat162 v = __hmul2(*reinterpret_cast<const __nv_bfloat162 *>(&y),
                                         *reinterpret_cast<const __nv_bfloat162 *>(&k126));
        const __nv_bfloat162 w = __hmul2(v, *reinterpret_cast<const __nv_bfloat162 *>(&sp[s][b]));
        out[b] = *reinterpret_cast<const uint32_t *>(&w);
      }
      store(i, out[0], out[1], out[2], out[3]);
    }
  } else if (WF == WF_INT4) {
    // flipping each code's sign bit gives n = q + 8; the BF16 pattern
    // 0x4300 | n is exactly 128 + n; minus 136 is q; one BF16 multiply by the
    // adjacent scale pair rounds q * s once
    const uint4 sv = *reinterpret_cast<const uint4 *>(raw_s + j * 16);
    const __nv_bfloat162 sc[4] = {*reinterpret_cast<const __nv_bfloat162 *>(&sv.x),
                                  *reinterpret_cast<const __nv_bfloat162 *>(&sv.y),
                                  *reinterpret_cast<const __nv_bfloat162 *>(&sv.z),
                                  *reinterpret_cast<const __nv_bfloat162 *>(&sv.w)};
    const __nv_bfloat162 k136 = __floats2bfloat162_rn(136.0f, 136.0f);
    uint32_t cw[ROWS];
#pragma unroll
    for (int i = 0; i < ROWS; ++i)
      cw[i] = *reinterpret_cast<const uint32_t *>(raw_w + (rr + i * R) * ROW_BYTES + j * 4);
#pragma unroll
    for (int i = 0; i < ROWS; ++i) {
      const uint32_t lo = (cw[i] ^ 0x88888888u) & 0x0F0F0F0Fu;         // even columns
      const uint32_t hi = ((cw[i] ^ 0x88888888u) >> 4) & 0x0F0F0F0Fu;  // odd columns
      uint32_t out[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        // byte b of lo to bits 0-7, byte b of hi to bits 16-23
        const uint32_t w = (__byte_perm(lo, hi, b | ((4 + b) << 8)) & 0x00FF00FFu) | 0x43004300u;
        const __nv_bfloat162 q = __hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&w), k136);
        const __nv_bfloat162 v = __hmul2(q, sc[b]);
        out[b] = *reinterpret_cast<const uint32_t *>(&v);
      }
      store(i, out[0], out[1], out[2], out[3]);
    }
  } else if (WF == WF_MXFP8) {
    // 2^(e-127) from the exponent bits; e = 0 is 2^-127, a binary32 subnormal
    float p[SR][8];
#pragma unroll
    for (int s = 0; s < SR; ++s) {
      const uint2 sc = *reinterpret_cast<const uint2 *>(raw_s + s * COLS + j * 8);
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const uint32_t e = ((b < 4 ? sc.x : sc.y) >> (8 * (b & 3))) & 0xFFu;
        p[s][b] = __uint_as_float(e ? e << 23 : 0x00400000u);
      }
    }
    uint2 cw[ROWS];
#pragma unroll
    for (int i = 0; i < ROWS; ++i)
      cw[i] = *reinterpret_cast<const uint2 *>(raw_w + (rr + i * R) * ROW_BYTES + j * 8);
#pragma unroll
    for (int i = 0; i < ROWS; ++i) {
      const int s = i * R * SR / 64;
      uint32_t out[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float2 f = e4m3x2_to_float2(((b < 2 ? cw[i].x : cw[i].y) >> (16 * (b & 1))) & 0xFFFFu);
        out[b] = bf16x2_bits(__fmul_rn(f.x, p[s][2 * b]), __fmul_rn(f.y, p[s][2 * b + 1]));
      }
      store(i, out[0], out[1], out[2], out[3]);
    }
  } else if (WF == WF_NVFP4) {
    uint2 sv[SR];
#pragma unroll
    for (int s = 0; s < SR; ++s)
      sv[s] = *reinterpret_cast<const uint2 *>(raw_s + s * COLS + j * 8);
    uint32_t cw[ROWS];
#pragma unroll
    for (int i = 0; i < ROWS; ++i)
      cw[i] = *reinterpret_cast<const uint32_t *>(raw_w + (rr + i * R) * ROW_BYTES + j * 4);
#pragma unroll
    for (int i = 0; i < ROWS; ++i) {
      const int s = i * R * SR / 64;
      uint32_t out[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float2 s2 = e4m3x2_to_float2(((b < 2 ? sv[s].x : sv[s].y) >> (16 * (b & 1))) & 0xFFFFu);
        const float v0 = e2m1_to_float((cw[i] >> (8 * b)) & 0xFu);
        const float v1 = e2m1_to_float((cw[i] >> (8 * b + 4)) & 0xFu);
        out[b] = bf16x2_bits(__fmul_rn(v0, s2.x), __fmul_rn(v1, s2.y));
      }
      store(i, out[0], out[1], out[2], out[3]);
    }
  }
}

}  // namespace swiglu
