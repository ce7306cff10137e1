// Q8 activation rail of the decode GEMV: activations requantised in blocks of
// 32 to int8 codes on a float32 scale, and the MXFP4 x Q8 dot taken in
// integers ("dasLLAMA gpt-oss arc": the dot_mx4q8 template looks a weight
// block's nibbles up in a table, the low nibble masked with 15 and the high
// one shifted down by 4, and accumulates four-lane integer dot products; the
// fused MoE expert chain commit requantises its first stage's activations in
// blocks of 32).
//
// On sm_103a the table lookup is a byte permute: the E2M1 table doubled
// ({0, 1, 2, 3, 4, 6, 8, 12} and their negatives: integers) sits in two pairs of
// 32-bit words, one prmt turns four nibbles into four int8 weights, and dp4a
// multiplies them with four int8 activation codes. A block's 32 products add
// up exactly in an int32; the float32 block products are added in a fixed
// order (lane l of the warp takes blocks l, l+32, ...; then a butterfly over
// lane distances 16, 8, 4, 2, 1; the bias last), so the result is a fixed
// function of the inputs, bit for bit.
#include "moe_common.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Requant: one warp per block of 32 values (lane = element).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quant_q8_kernel(const float* __restrict__ v, int64_t nblocks,
                                                       int8_t* __restrict__ q, float* __restrict__ d) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t b = w0; b < nblocks; b += nw) {
    const float x = v[b * 32 + lane];
    // the largest magnitude (non-negative floats order like their bit patterns)
    const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(x) & 0x7FFFFFFFu));
    int code = 0;
    float scale = 0.f;
    if (amax > 0.f) {
      const float inv = __fdiv_rn(127.f, amax);
      code = __float2int_rn(__fmul_rn(x, inv));
      scale = __fdiv_rn(amax, 127.f);
    }
    q[b * 32 + lane] = (int8_t)code;
    if (lane == 0) d[b] = scale;
  }
}

// ---------------------------------------------------------------------------
// MXFP4 x Q8 GEMV: out[i][r] = W[experts[i]][r] . (q, d)[i / act_div] + bias.
// One warp per row; grid = (row groups of kQ8Warps, n).
// ---------------------------------------------------------------------------
constexpr int kQ8Warps = 8;

// Four E2M1 codes (one nibble in the low half of each byte of `nib`) to four
// int8 values of the doubled table.
__device__ __forceinline__ uint32_t e2m1x4_to_i8x4(uint32_t nib) {
  constexpr uint32_t kPosLo = 0x03020100u, kPosHi = 0x0C080604u;  // 0 1 2 3 | 4 6 8 12
  constexpr uint32_t kNegLo = 0xFDFEFF00u, kNegHi = 0xF4F8FAFCu;  // 0 -1 -2 -3 | -4 -6 -8 -12
  // the four nibbles as a byte-permute selector (nibble j of the low 16 bits = byte j's code)
  const uint32_t packed = nib | (nib >> 4);                  // bytes 0 and 2 hold two codes each
  const uint32_t sel = __byte_perm(packed, 0u, 0x4420u) & 0x7777u;  // magnitude index of each code
  const uint32_t pos = __byte_perm(kPosLo, kPosHi, sel);
  const uint32_t neg = __byte_perm(kNegLo, kNegHi, sel);
  const uint32_t m = ((nib >> 3) & 0x01010101u) * 0xFFu;    // 0xFF in the bytes of negative codes
  return (pos & ~m) | (neg & m);
}

// 2^(s - 128) for an E8M0 byte s (s = 255: NaN), as the float bit pattern.
__device__ __forceinline__ float e8m0_half_scale(uint32_t s) {
  if (s == 255u) return __uint_as_float(0x7FC00000u);
  if (s >= 2u) return __uint_as_float((s - 1u) << 23);
  return __uint_as_float(s ? 0x00400000u : 0x00200000u);  // 2^-127, 2^-128 (subnormal)
}

template <int NBL>
__global__ void __launch_bounds__(kQ8Warps * 32) gemv_q8_kernel(
    const uint8_t* __restrict__ qs, const uint8_t* __restrict__ sc, int E, int R, int C,
    const int32_t* __restrict__ experts, int act_div, const int8_t* __restrict__ aq, const float* __restrict__ ad,
    const float* __restrict__ bias, float* __restrict__ out, int* status, int wrs) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int i = blockIdx.y;
  const int r = blockIdx.x * kQ8Warps + warp;
  if (r >= R) return;
  const int e = experts[i];
  if (e < 0 || e >= E) {
    if (lane == 0) {
      set_status(status, 0x1);
      out[(size_t)i * R + r] = 0.f;
    }
    return;
  }
  const int nb = C >> 5;
  const int a = i / act_div;
  const int8_t* qa = aq + (size_t)a * C;
  const float* da = ad + (size_t)a * nb;
  const size_t row = ((size_t)e * R + r) * wrs;  // wrs = 2: gate/up rows interleaved in one plane
  float acc = 0.f;
#pragma unroll
  for (int j = 0; j < NBL; ++j) {
    const int b = lane + 32 * j;
    if (b < nb) {
      const uint4 w = ldg_nc_v4(qs + row * (C / 2) + (size_t)b * 16);
      const uint32_t s = ldg_nc_u8(sc + row * nb + b);
      const int4 x0 = __ldg(reinterpret_cast<const int4*>(qa + (size_t)b * 32));       // columns 0..15
      const int4 x1 = __ldg(reinterpret_cast<const int4*>(qa + (size_t)b * 32 + 16));  // columns 16..31
      const float dx = __ldg(da + b);
      int isum = 0;
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
      const int lo[4] = {x0.x, x0.y, x0.z, x0.w}, hi[4] = {x1.x, x1.y, x1.z, x1.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {  // bytes 4t..4t+3: columns 4t.. (low nibbles), 16+4t.. (high)
        isum = __dp4a((int)e2m1x4_to_i8x4(ww[t] & 0x0F0F0F0Fu), lo[t], isum);
        isum = __dp4a((int)e2m1x4_to_i8x4((ww[t] >> 4) & 0x0F0F0F0Fu), hi[t], isum);
      }
      const float fac = __fmul_rn(dx, e8m0_half_scale(s));
      acc = __fadd_rn(acc, __fmul_rn((float)isum, fac));
    }
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, m));
  if (lane == 0) out[(size_t)i * R + r] = bias ? __fadd_rn(acc, bias[row]) : acc;
}

// ---------------------------------------------------------------------------
// Slot-order combine: y[t][c] = sum_j w[t][j] * o[t*k+j][c] over the valid slots.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) combine_slots_kernel(const float* __restrict__ o, const float* __restrict__ w,
                                                            const int32_t* __restrict__ ids, int k, int D, int E,
                                                            float* __restrict__ y) {
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.y, c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= D) return;
  float acc = 0.f;
  for (int j = 0; j < k; ++j) {
    const int a = t * k + j, e = ids[a];
    if (e >= 0 && e < E) acc = fmaf(w[a], o[(size_t)a * D + c], acc);
  }
  y[(size_t)t * D + c] = acc;
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
static int grid_for(int64_t threads) {
  const int64_t cap = (int64_t)device_sm_count() * 8;
  int64_t b = (threads + 255) / 256;
  if (b > cap) b = cap;
  return (int)(b < 1 ? 1 : b);
}

cudaError_t launch_quant_q8(const float* v, int64_t rows, int C, int8_t* q, float* d, Launch L) {
  const int64_t nblocks = rows * (C / 32);
  if (nblocks <= 0) return cudaSuccess;
  return launch_kernel(quant_q8_kernel, dim3(grid_for(nblocks * 32)), dim3(256), 0, L, v, nblocks, q, d);
}

cudaError_t launch_gemv_q8(const uint8_t* qs, const uint8_t* sc, int E, int R, int C, const int32_t* experts,
                           int n, int act_div, const int8_t* aq, const float* ad, const float* bias, float* out,
                           int* status, Launch L, int wrs) {
  if (n <= 0 || R <= 0) return cudaSuccess;
  if (wrs != 1 && wrs != 2) return cudaErrorInvalidValue;
  const dim3 grid((R + kQ8Warps - 1) / kQ8Warps, n);
  switch (((C >> 5) + 31) / 32) {
    case 1:
      return launch_kernel(gemv_q8_kernel<1>, grid, dim3(kQ8Warps * 32), 0, L, qs, sc, E, R, C, experts, act_div,
                           aq, ad, bias, out, status, wrs);
    case 2:
      return launch_kernel(gemv_q8_kernel<2>, grid, dim3(kQ8Warps * 32), 0, L, qs, sc, E, R, C, experts, act_div,
                           aq, ad, bias, out, status, wrs);
    case 3:
      return launch_kernel(gemv_q8_kernel<3>, grid, dim3(kQ8Warps * 32), 0, L, qs, sc, E, R, C, experts, act_div,
                           aq, ad, bias, out, status, wrs);
    case 4:
      return launch_kernel(gemv_q8_kernel<4>, grid, dim3(kQ8Warps * 32), 0, L, qs, sc, E, R, C, experts, act_div,
                           aq, ad, bias, out, status, wrs);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_combine_slots(const float* o, const float* w, const int32_t* ids, int T, int k, int D, int E,
                                 float* y, Launch L) {
  if (T <= 0) return cudaSuccess;
  return launch_kernel(combine_slots_kernel, dim3((D + 255) / 256, T), dim3(256), 0, L, o, w, ids, k, D, E, y);
}

}  // namespace moe
