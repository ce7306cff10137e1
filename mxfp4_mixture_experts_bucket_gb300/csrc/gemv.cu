// Standalone MXFP4 GEMV and elementwise swiglu_oai on the CUDA cores.
//
// The routed-expert GEMV (MetalMoeGemvMx4 of "dasLLAMA: dig the last two board
// reds green", section "gpt-oss: mx4 kernels to the lab-winning shape") loads
// every weight byte exactly once with wide loads and computes the E8M0 scale
// in the ALU. On sm_103a one 128-bit load per lane carries a whole 32-element
// MXFP4 block; the E2M1 nibble pairs go through the hardware e2m1x2 -> f16x2
// conversion and packed f32x2 FMAs, partial sums reduce with warp shuffles.
// The fused decode expert kernels live in decode.cu.
#include "tcgen05.cuh"

namespace moe {

constexpr int kGemvWarps = 8;
constexpr int kGemvThreads = kGemvWarps * 32;

// Copies a length-C float vector into pair-swizzled shared memory.
__device__ __forceinline__ void stage_pairswz(float* __restrict__ dst, const float* __restrict__ src,
                                              int C) {
  for (int c = threadIdx.x; c < C; c += blockDim.x) dst[pairswz_offset(c)] = src[c];
}

// ---------------------------------------------------------------------------
// Standalone GEMV: out[i][r] = W[experts[i]][r] . x_i + bias[experts[i]][r]
// grid = (row tiles of 2*kGemvWarps rows, n); each warp computes two rows.
// ---------------------------------------------------------------------------
template <int NBL>
__global__ void __launch_bounds__(kGemvThreads) mxfp4_gemv_kernel(
    const uint8_t* __restrict__ qs, const uint8_t* __restrict__ sc, int E, int R, int C,
    const int32_t* __restrict__ experts, const float* __restrict__ x, int64_t x_stride,
    const float* __restrict__ bias, float* __restrict__ out, int* status) {
  extern __shared__ float4 smem_f4[];
  float* xs = reinterpret_cast<float*>(smem_f4);
  const int i = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  pdl_launch_dependents();
  pdl_wait();
  stage_pairswz(xs, x + (size_t)i * x_stride, C);
  __syncthreads();
  const int e = experts[i];
  const int r0 = (blockIdx.x * kGemvWarps + warp) * 2;
  if (r0 >= R) return;
  const bool valid_e = (e >= 0 && e < E);
  if (!valid_e) {
    if (lane == 0) {
      set_status(status, 0x1);
      out[(size_t)i * R + r0] = 0.f;
      if (r0 + 1 < R) out[(size_t)i * R + r0 + 1] = 0.f;
    }
    return;
  }
  const int nb = C >> 5;
  const int nr = (r0 + 1 < R) ? 2 : 1;
  uint4 q[2][NBL];
  uint32_t s[2][NBL];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const size_t row = (size_t)e * R + r0 + (r < nr ? r : 0);
#pragma unroll
    for (int j = 0; j < NBL; ++j) {
      const int b = lane + 32 * j;
      if (b < nb) {
        q[r][j] = ldg_nc_v4(qs + row * (C / 2) + (size_t)b * 16);
        s[r][j] = ldg_nc_u8(sc + row * nb + b);
      }
    }
  }
  float acc[2] = {0.f, 0.f};
  const float4* xv4 = reinterpret_cast<const float4*>(xs);
#pragma unroll
  for (int j = 0; j < NBL; ++j) {
    const int b = lane + 32 * j;
    if (b < nb) {
      float4 xv[8];
      load_pair_group(xv4, b, xv);
#pragma unroll
      for (int r = 0; r < 2; ++r) acc[r] = fmaf(mx_block_dot(q[r][j], xv), e8m0_to_f32(s[r][j]), acc[r]);
    }
  }
  acc[0] = warp_sum(acc[0]);
  acc[1] = warp_sum(acc[1]);
  if (lane < nr) {
    const int r = r0 + lane;
    const float v = (lane == 0 ? acc[0] : acc[1]) + (bias ? bias[(size_t)e * R + r] : 0.f);
    out[(size_t)i * R + r] = v;
  }
}

// ---------------------------------------------------------------------------
// Elementwise swiglu_oai.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) swiglu_kernel(const float* __restrict__ g,
                                                     const float* __restrict__ u, void* h, int64_t n,
                                                     int h_dtype, float alpha, float limit) {
  pdl_launch_dependents();
  pdl_wait();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float v = swiglu_oai_f(g[i], u[i], alpha, limit);
    if (h_dtype == 0) {
      static_cast<float*>(h)[i] = v;
    } else {
      __nv_bfloat16 b = __float2bfloat16_rn(v);
      static_cast<__nv_bfloat16*>(h)[i] = b;
    }
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
template <typename K>
static cudaError_t set_smem(K kern, size_t bytes) {
  return ensure_smem_limit(kern, bytes);
}

cudaError_t launch_mxfp4_gemv(const uint8_t* qs, const uint8_t* sc, int E, int R, int C,
                              const int32_t* experts, int n, const float* x, int64_t x_stride,
                              const float* bias, float* out, int* status, Launch L) {
  if (n <= 0 || R <= 0) return cudaSuccess;
  const size_t smem = (size_t)C * sizeof(float);
  dim3 grid((R + 2 * kGemvWarps - 1) / (2 * kGemvWarps), n);
  const int nbl = ((C >> 5) + 31) / 32;
  cudaError_t err;
#define MOE_GEMV_CASE(N)                                                                        \
  case N:                                                                                       \
    if ((err = set_smem(mxfp4_gemv_kernel<N>, smem)) != cudaSuccess) return err;                \
    return launch_kernel(mxfp4_gemv_kernel<N>, grid, dim3(kGemvThreads), smem, L, qs, sc, E, R, \
                         C, experts, x, x_stride, bias, out, status);
  switch (nbl) {
    MOE_GEMV_CASE(1)
    MOE_GEMV_CASE(2)
    MOE_GEMV_CASE(3)
    MOE_GEMV_CASE(4)
    default:
      return cudaErrorInvalidValue;
  }
#undef MOE_GEMV_CASE
}

cudaError_t launch_swiglu(const float* g, const float* u, void* h, int64_t n, int h_dtype,
                          float alpha, float limit, Launch L) {
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  return launch_kernel(swiglu_kernel, dim3((unsigned)blocks), dim3(256), 0, L, g, u, h, n, h_dtype,
                       alpha, limit);
}

// ---------------------------------------------------------------------------
// RMS renormalisation of token rows, y[t] = x[t] / sqrt(mean_c x[t][c]^2) (a
// zero row stays zero): the step between the layers of a stack of MoE layers.
// One block per row; the sum of squares is added in a fixed order (strided
// per-thread sums, then a tree over the threads), so the result is
// deterministic. In place is allowed.
// ---------------------------------------------------------------------------
constexpr int kRmsThreads = 256;
__global__ void __launch_bounds__(kRmsThreads) rms_renorm_kernel(const float* x, int D, float* y) {
  __shared__ float part[kRmsThreads];
  pdl_launch_dependents();
  pdl_wait();
  const float* xr = x + (size_t)blockIdx.x * D;
  float* yr = y + (size_t)blockIdx.x * D;
  float s = 0.f;
  for (int c = threadIdx.x; c < D; c += kRmsThreads) s = fmaf(xr[c], xr[c], s);
  part[threadIdx.x] = s;
  __syncthreads();
  for (int w = kRmsThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
    __syncthreads();
  }
  const float mean = part[0] / (float)D;
  const float inv = mean > 0.f ? 1.f / sqrtf(mean) : 0.f;
  for (int c = threadIdx.x; c < D; c += kRmsThreads) yr[c] = xr[c] * inv;
}

cudaError_t launch_rms_renorm(const float* x, int T, int D, float* y, Launch L) {
  if (T <= 0) return cudaSuccess;
  return launch_kernel(rms_renorm_kernel, dim3(T), dim3(kRmsThreads), 0, L, x, D, y);
}

}  // namespace moe
