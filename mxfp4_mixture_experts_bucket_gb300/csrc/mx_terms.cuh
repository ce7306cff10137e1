// E4M3 activation terms of the block-scaled tensor-core rails.
//
// An activation block of 32 values (one MXFP4 scale block along K) is carried
// as a sum of E4M3 blocks ("terms"), each on its own E8M0 scale; every term
// takes the exact rounding residual of the ones before it, so each adds about
// four significant bits. Inside a block the E4M3 bytes sit in the MMA's K
// order: stored column c at position 2*(c%16) + c/16, the order in which the
// MXFP4 nibble layout (byte i: column i low, column 16+i high) presents the
// weights once a stored 16-byte block is split into two 8-byte chunks.
#pragma once

#include "moe_common.cuh"

namespace moe {
namespace mx {

// ---------------------------------------------------------------- E4M3 terms
// Position of stored column c (0..31) of a block in the MMA's K order.
__device__ __forceinline__ int mx_pos(int c) { return 2 * (c & 15) + (c >> 4); }

// E8M0 code of a block whose largest magnitude has the bit pattern am: the
// block divided by 2^(code-127) has its largest element in [128, 256), inside
// E4M3's range (448), never saturating.
__device__ __forceinline__ uint32_t block_code(uint32_t am) {
  const int eb = (int)(am >> 23);
  return (uint32_t)(eb > 7 ? eb - 7 : 0);
}
// 2^(127 - code) for code in [0, 248], a normal float
__device__ __forceinline__ float inv_scale(uint32_t code) { return __uint_as_float((254u - code) << 23); }
// 2^(code - 127) for code in [0, 254]
__device__ __forceinline__ float fwd_scale(uint32_t code) {
  return code ? __uint_as_float(code << 23) : __uint_as_float(0x00400000u);
}
__device__ __forceinline__ uint32_t f32_to_e4m3(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(v));  // second operand -> low byte
  return r & 0xFFu;
}
// Exact value of an E4M3 code (never the NaN code here): its seven magnitude
// bits placed at the top of an fp32 exponent/mantissa give value * 2^-120.
__device__ __forceinline__ float e4m3_to_f32(uint32_t q) {
  const float s = __uint_as_float(((q & 0x80u) << 24) | ((q & 0x7Fu) << 20));
  return __fmul_rn(s, __uint_as_float(0x7B800000u));  // * 2^120
}

// One block of 32 values, one per lane (all lanes of the warp take part):
// v = sum_t E4M3(q[t]) * 2^(s[t]-127) + (rounding of the last term); each term
// encodes the residual of the ones before it exactly, then rounds it.
template <int NT>
__device__ __forceinline__ void split_terms(float v, uint32_t (&q)[NT], uint32_t (&s)[NT]) {
  float r = v;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const uint32_t am = __reduce_max_sync(0xffffffffu, __float_as_uint(r) & 0x7FFFFFFFu);
    s[t] = block_code(am);
    q[t] = f32_to_e4m3(__fmul_rn(r, inv_scale(s[t])));
    if (t + 1 < NT) r = __fmaf_rn(-e4m3_to_f32(q[t]), fwd_scale(s[t]), r);  // exact residual
  }
}

// ---------------------------------------------------------------- E2M1 terms
// The same split in the MXFP4 element format itself (the decode rail's
// activation operand for kind::mxf4): each term is 32 E2M1 codes on the power
// of two 2^e with the smallest e such that the block's largest |r| <= 6 * 2^e.
// E8M0 code of that scale for a block whose largest magnitude has the bit
// pattern am (e clamped to [-127, 127]; zero and subnormal blocks take 2^-127).
__device__ __forceinline__ uint32_t e2m1_block_code(uint32_t am) {
  const int eb = (int)(am >> 23);
  if (eb == 0) return 0u;
  const int e = (eb - 127) - ((am & 0x7FFFFFu) > 0x400000u ? 1 : 2);  // mantissa above 1.5: one step up
  return (uint32_t)(e < -127 ? 0 : (e > 127 ? 254 : e + 127));
}
// One value to its E2M1 code, rounded to nearest (ties to even), saturating at 6.
__device__ __forceinline__ uint32_t f32_to_e2m1(float v) {
  uint16_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u16.u8 %0, t;\n}" : "=h"(r) : "f"(0.f), "f"(v));
  return r & 0xFu;  // the second operand lands in the low nibble
}
// Exact value of an E2M1 code: 0, 0.5 (subnormals) or 2^(e-1) * (1 + m/2).
__device__ __forceinline__ float e2m1_to_f32(uint32_t q) {
  const uint32_t e = (q >> 1) & 3u, m = q & 1u;
  const uint32_t bits = e ? (((e + 126u) << 23) | (m << 22)) : (m ? 0x3F000000u : 0u);
  return __uint_as_float(bits | ((q & 8u) << 28));
}

// Two E2M1 codes (one byte: low nibble, high nibble) to their exact values as
// an f16 pair (low nibble in the low half); every E2M1 value is an f16 value.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t h2;
  asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}" : "=r"(h2) : "r"(byte));
  return h2;
}

// One block of 32 values, one per lane (all lanes of the warp take part): v as
// NT E2M1 terms, q[t] the lane's code and s[t] the block's E8M0 code of term t;
// each term rounds the exact residual of the ones before it.
template <int NT>
__device__ __forceinline__ void split_terms_e2m1(float v, uint32_t (&q)[NT], uint32_t (&s)[NT]) {
  float r = v;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const uint32_t am = __reduce_max_sync(0xffffffffu, __float_as_uint(r) & 0x7FFFFFFFu);
    s[t] = e2m1_block_code(am);
    q[t] = f32_to_e2m1(__fmul_rn(r, inv_scale(s[t])));
    if (t + 1 < NT) r = __fmaf_rn(-e2m1_to_f32(q[t]), fwd_scale(s[t]), r);  // exact residual
  }
}

// The same split with a block held by a lane pair (lanes 2i and 2i + 1, both
// calling it; pair = the pair's lane mask), one term at a time, with the same
// arithmetic: lane h holds columns 8h .. 8h + 7 in r[0..7] and 16 + 8h ..
// 16 + 8h + 7 in r[8..15]; the pair exchanges its largest magnitudes once, so
// both lanes take the same scale code s. The lane's 8 bytes of the packed
// block (byte i = column i low nibble, column 16 + i high; bytes 8h .. 8h + 7)
// come back in `packed`; r becomes the residual unless `last` (then r is left
// scaled). The residual is taken in the scaled domain: v = r * 2^-e is exact,
// v - code (the code's value exact in f16, one mixed-precision FMA) is exact
// because the code is v's nearest E2M1 value, and * 2^e rounds once, as
// r - code * 2^e would.
__device__ __forceinline__ void split_half_block_e2m1_term(float (&r)[16], bool last, uint32_t pair, uint2& packed,
                                                           uint32_t& s) {
  float am[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) am[i] = fmaxf(fabsf(r[i]), fabsf(r[8 + i]));
#pragma unroll
  for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) am[i] = fmaxf(am[i], am[i + w]);
  const float m = fmaxf(am[0], __shfl_xor_sync(pair, am[0], 1));
  s = e2m1_block_code(__float_as_uint(m));
  const float inv = inv_scale(s), fwd = fwd_scale(s);
  uint32_t b[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 v = __fmul2_rn(make_float2(r[i], r[8 + i]), make_float2(inv, inv));
    r[i] = v.x;
    r[8 + i] = v.y;
    asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u32.u8 %0, t;\n}" : "=r"(b[i]) : "f"(v.y), "f"(v.x));
  }
  packed = make_uint2(__byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410),
                      __byte_perm(__byte_perm(b[4], b[5], 0x0040), __byte_perm(b[6], b[7], 0x0040), 0x5410));
  if (!last) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t h2 = e2m1x2_to_f16x2(b[i]);
      float d0, d1;
      asm("{\n .reg .b16 c0, c1, m;\n mov.b32 {c0, c1}, %2;\n mov.b16 m, 0xBC00;\n"
          " fma.rn.f32.f16 %0, c0, m, %3;\n fma.rn.f32.f16 %1, c1, m, %4;\n}"
          : "=f"(d0), "=f"(d1)
          : "r"(h2), "f"(r[i]), "f"(r[8 + i]));  // v - code, exact
      const float2 rr = __fmul2_rn(make_float2(d0, d1), make_float2(fwd, fwd));
      r[i] = rr.x;
      r[8 + i] = rr.y;
    }
  }
}

// A warp's block of E2M1 codes (lane l holds column l) packed as the MXFP4 block
// layout: byte i = column i in the low nibble, column 16 + i in the high nibble.
// Lanes 0..15 return their byte; the other lanes' result is unused.
__device__ __forceinline__ uint32_t pack_e2m1_block(uint32_t q) {
  const uint32_t hi = __shfl_down_sync(0xffffffffu, q, 16);
  return (q & 0xFu) | ((hi & 0xFu) << 4);
}

}  // namespace mx
}  // namespace moe
