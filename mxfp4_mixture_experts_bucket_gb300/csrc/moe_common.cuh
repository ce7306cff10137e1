// Shared device helpers for the MXFP4 routed-MoE kernels (sm_103a only).
//
// MXFP4 storage (the library's layout): a matrix W[R, C] is a nibble plane
// qs[R][C/2] and an exponent plane sc[R][C/32]. Block b of a row covers
// columns 32b..32b+31 in bytes 16b..16b+15; byte i holds column 32b+i in its
// low nibble and column 32b+16+i in its high nibble. A value is
// E2M1[q] * 2^(s-127) ("dasLLAMA: dig the last two board reds green",
// section "gpt-oss: mx4 kernels to the lab-winning shape": 16-value E2M1
// table, E8M0 exponent computed in the ALU as a float bit pattern).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "../../include/moe_mxfp4.h"
#include "moe_internal.h"

namespace moe {

// ---------------------------------------------------------------------------
// status word
// ---------------------------------------------------------------------------
__device__ __forceinline__ void set_status(int* status, int bits) {
  if (status) atomicOr(status, bits);
}

// Device-side bounds checks of the checked build (-DMOE_CHECKED): a failed
// check sets MOE_STATUS_OUT_OF_BOUNDS and the caller skips the access. In the
// regular build the condition is not evaluated.
__device__ __forceinline__ bool check_bounds(int* status, bool ok) {
  if (!ok) set_status(status, MOE_STATUS_OUT_OF_BOUNDS);
  return ok;
}
#ifdef MOE_CHECKED
#define MOE_IN_BOUNDS(status, cond) (::moe::check_bounds((status), (cond)))
#else
#define MOE_IN_BOUNDS(status, cond) true
#endif

// A bounded wait gave up: set the timeout bit and keep the first site that did
// (status[1], see moe_get_timeout_site): kernel << 24 | role << 20 |
// (stage & 0xff) << 12 | (sequence index & 0xfff).
__device__ __forceinline__ void report_timeout(int* status, int kernel, int role, int stage, int seq) {
  if (!status) return;
  atomicOr(status, 0x2);
  const int site = (kernel << 24) | ((role & 0xf) << 20) | ((stage & 0xff) << 12) | (seq & 0xfff);
  atomicCAS(status + 1, 0, site);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// E8M0 and E2M1 decode
// ---------------------------------------------------------------------------

// 2^(s-127) built directly as an fp32 bit pattern: exponent field s for
// s = 1..254, the denormal 2^-127 for s = 0, NaN for s = 255.
__device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
  uint32_t bits = (s == 0u) ? 0x00400000u : ((s == 255u) ? 0x7FC00000u : (s << 23));
  return __uint_as_float(bits);
}

// One byte holding two E2M1 codes -> f16x2 (low nibble -> low half). Exact.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t word, int byte_idx) {
  uint32_t r;
  switch (byte_idx) {
    case 0:
      asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b0;\n}"
          : "=r"(r) : "r"(word));
      break;
    case 1:
      asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b1;\n}"
          : "=r"(r) : "r"(word));
      break;
    case 2:
      asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b2;\n}"
          : "=r"(r) : "r"(word));
      break;
    default:
      asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b3;\n}"
          : "=r"(r) : "r"(word));
      break;
  }
  return r;
}

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t h) {
  __half2 v = *reinterpret_cast<__half2*>(&h);
  return __half22float2(v);
}

// Four bytes of E2M1 pairs -> four f16x2 (byte i -> h[i], low nibble -> low half).
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// ---------------------------------------------------------------------------
// Pair-swizzled float vectors used by the decode (GEMV) rail.
//
// A length-C vector v is stored as C/32 groups of 8 float4. Group b holds the
// pairs (v[32b+i], v[32b+16+i]) for i = 0..15, two pairs per float4: float4 j
// holds pairs 2j and 2j+1 as (v[32b+2j], v[32b+16+2j], v[32b+2j+1],
// v[32b+16+2j+1]), and sits at position j ^ (b & 7) inside its group so that
// eight lanes reading eight consecutive groups hit distinct shared-memory
// banks. The pair order matches the byte order of an MXFP4 block.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int pairswz_offset(int c) {
  int b = c >> 5, i = c & 31;
  int p = i & 15, slot = i >> 4;
  int j = p >> 1;
  int phys = (b << 3) + (j ^ (b & 7));
  return (phys << 2) + ((p & 1) << 1) + slot;
}

// Loads the group of block b of a pair-swizzled vector into registers, in
// logical float4 order (pairs 2j, 2j+1 in xv[j]).
__device__ __forceinline__ void load_pair_group(const float4* __restrict__ vec, int b, float4 (&xv)[8]) {
  const float4* grp = vec + (b << 3);
#pragma unroll
  for (int j = 0; j < 8; ++j) xv[j] = grp[j ^ (b & 7)];
}

// Dot of one MXFP4 block (16 nibble bytes, unscaled E2M1 values) with the
// block's pairs of a vector (xv from load_pair_group). fp32 products and sums,
// two lanes per instruction on the Blackwell f32x2 FMA path.
__device__ __forceinline__ float mx_block_dot(uint4 q, const float4 (&xv)[8]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    // bytes 4m..4m+3 of the block are pairs 4m..4m+3 -> xv[2m], xv[2m+1]
    uint32_t h[4];
    e2m1x8_to_f16x2x4(w[m], h);
    const float4 xa = xv[2 * m];
    const float4 xb = xv[2 * m + 1];
    acc0 = __ffma2_rn(f16x2_to_float2(h[0]), make_float2(xa.x, xa.y), acc0);
    acc1 = __ffma2_rn(f16x2_to_float2(h[1]), make_float2(xa.z, xa.w), acc1);
    acc0 = __ffma2_rn(f16x2_to_float2(h[2]), make_float2(xb.x, xb.y), acc0);
    acc1 = __ffma2_rn(f16x2_to_float2(h[3]), make_float2(xb.z, xb.w), acc1);
  }
  const float2 acc = __fadd2_rn(acc0, acc1);
  return acc.x + acc.y;
}

// ---------------------------------------------------------------------------
// swiglu_oai
// ---------------------------------------------------------------------------
__device__ __forceinline__ float sigmoid_f(float z) {
  // 1/(1+e^-z) for z >= 0 and e^z/(1+e^z) otherwise: never inf/inf.
  if (z >= 0.f) return 1.f / (1.f + __expf(-z));
  const float ez = __expf(z);
  return ez / (1.f + ez);
}

__device__ __forceinline__ float swiglu_oai_f(float g, float u, float alpha, float limit) {
  g = fminf(g, limit);
  u = fminf(fmaxf(u, -limit), limit);
  return g * sigmoid_f(alpha * g) * (u + 1.f);
}

// The same with a fast reciprocal and no branch (a few ulp): 1/(1 + e^-z)
// tends to 0 as z -> -inf (e^-z = inf, reciprocal 0), never NaN for finite g.
__device__ __forceinline__ float swiglu_oai_fast(float g, float u, float alpha, float limit) {
  g = fminf(g, limit);
  u = fminf(fmaxf(u, -limit), limit);
  return g * __fdividef(1.f, 1.f + __expf(-alpha * g)) * (u + 1.f);
}

// ---------------------------------------------------------------------------
// warp helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ldg_nc_u8(const uint8_t* p) {
  uint16_t r;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(r) : "l"(p));
  return (uint32_t)r;
}

// ---------------------------------------------------------------------------
// Router top-k then softmax over the k selected, one warp per token (E <= 256,
// k <= 32). Order: descending logit, lower expert index first on equal
// logits; NaN logits never win. Lane j < k gets slot j's expert and weight
// exp(l_j - l_0) / sum_m exp(l_m - l_0).
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool topk_better(float va, int ia, float vb, int ib) {
  return (va > vb) || (va == vb && ia < ib);
}

__device__ __forceinline__ void warp_topk_softmax(const float* __restrict__ lt, int E, int k, int lane,
                                                  int& my_id, float& my_w) {
  if (E <= 32) {
    // One expert per lane: its slot is its rank, the number of experts ahead
    // of it in the order above (32 independent broadcasts, no argmax chain).
    float v = (lane < E) ? lt[lane] : -INFINITY;
    if (v != v) v = -INFINITY;
    const int me = (lane < E) ? lane : 0x7fffffff;
    int rank = 0;
#pragma unroll
    for (int o = 0; o < 32; ++o) {
      const float ov = __shfl_sync(0xffffffffu, v, o);
      rank += (o < E) && topk_better(ov, o, v, me);
    }
    const bool sel = (lane < E) && rank < k;
    // the lane holding slot j, for j = 0..k-1 (k <= E <= 32 lanes are ranked 0..E-1)
    const float top0 = __shfl_sync(0xffffffffu, v, __ffs(__ballot_sync(0xffffffffu, sel && rank == 0)) - 1);
    const float ex = expf(v - top0);
    float sum = 0.f;
    for (int j = 0; j < k; ++j)  // slot order, as below
      sum += __shfl_sync(0xffffffffu, ex, __ffs(__ballot_sync(0xffffffffu, sel && rank == j)) - 1);
    // hand slot j to lane j
    my_id = -1;
    float my_ex = 0.f;
    for (int j = 0; j < k; ++j) {
      const int src = __ffs(__ballot_sync(0xffffffffu, sel && rank == j)) - 1;
      const float exj = __shfl_sync(0xffffffffu, ex, src);
      if (lane == j) {
        my_id = src;
        my_ex = exj;
      }
    }
    my_w = my_ex / sum;
    return;
  }
  constexpr int MAXPER = 8;
  float v[MAXPER];
#pragma unroll
  for (int q = 0; q < MAXPER; ++q) {
    const int e = lane + 32 * q;
    float val = (e < E) ? lt[e] : -INFINITY;
    if (val != val) val = -INFINITY;
    v[q] = val;
  }
  uint32_t taken = 0;  // bit q: expert lane+32q already selected
  float top0 = 0.f, sum = 0.f, my_ex = 0.f;
  my_id = -1;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int q = 0; q < MAXPER; ++q) {
      const int e = lane + 32 * q;
      if (e < E && !((taken >> q) & 1u) && topk_better(v[q], e, bv, bi)) {
        bv = v[q];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (topk_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (j == 0) top0 = bv;
    const float ex = expf(bv - top0);
    sum += ex;
    if (lane == j) {
      my_ex = ex;
      my_id = bi;
    }
  }
  my_w = my_ex / sum;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace moe
