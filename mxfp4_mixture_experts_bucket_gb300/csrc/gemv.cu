// Decode rail: MXFP4 GEMVs on the CUDA cores, fp32 accumulation.
//
// The routed-expert GEMV (MetalMoeGemvMx4 of "dasLLAMA: dig the last two board
// reds green", section "gpt-oss: mx4 kernels to the lab-winning shape") loads
// every weight byte exactly once with wide loads and computes the E8M0 scale
// in the ALU. On sm_103a one 128-bit load per lane carries a whole 32-element
// MXFP4 block; the E2M1 nibble pairs go through the hardware e2m1x2 -> f16x2
// conversion and packed f32x2 FMAs (see the design doc for the measured comparison
// with a shared-memory lookup table), partial sums reduce with warp shuffles.
//
// The fused pair of kernels mirrors the fused decode expert chain of
// "dasLLAMA gpt-oss arc" (fused MoE expert chain commit): stage 0 = gate+up
// rows + bias + activation per (expert, row span); stage 1 = every expert's
// down rows + bias + the router-weighted sum in slot order per output span.
#include "moe_common.cuh"

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
// Active-expert list of a bucket: experts with counts > 0, ascending.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int build_active(const int32_t* __restrict__ counts, int E, int* s_active) {
  __shared__ int s_n;
  if (threadIdx.x < 32) {
    int n = 0;
    const int lane = threadIdx.x;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const bool on = (e < E) && counts[e] > 0;
      const uint32_t bal = __ballot_sync(0xffffffffu, on);
      if (on) s_active[n + __popc(bal & ((1u << lane) - 1u))] = e;
      n += __popc(bal);
    }
    if (lane == 0) s_n = n;
  }
  __syncthreads();
  return s_n;
}

// ---------------------------------------------------------------------------
// Fused gate/up + bias + swiglu over the bucketed assignments.
// Task = (active expert, pair of rows f0, f0+1): each warp streams the gate
// and up rows once and applies them to every token routed to that expert.
// h[a] (a = t*k+j) is written pair-swizzled for the down kernel.
// ---------------------------------------------------------------------------
template <int NBL>
__global__ void __launch_bounds__(kGemvThreads) gemv_gateup_swiglu_kernel(
    const uint8_t* __restrict__ g_qs, const uint8_t* __restrict__ g_sc, const float* __restrict__ bg,
    const uint8_t* __restrict__ u_qs, const uint8_t* __restrict__ u_sc, const float* __restrict__ bu,
    int E, int F, int D, int T, int k, const float* __restrict__ x,
    const int32_t* __restrict__ counts, const int32_t* __restrict__ basep,
    const int32_t* __restrict__ rows, float alpha, float limit, float* __restrict__ h) {
  extern __shared__ float4 smem_f4[];
  float* xs = reinterpret_cast<float*>(smem_f4);  // [T][D] pair-swizzled
  __shared__ int s_active[256];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  pdl_launch_dependents();
  // prologue independent of the previous kernels: stage the tokens
  for (int t = 0; t < T; ++t) stage_pairswz(xs + (size_t)t * D, x + (size_t)t * D, D);
  pdl_wait();
  const int nact = build_active(counts, E, s_active);  // includes __syncthreads
  const int nb = D >> 5;
  const int half = F >> 1;
  const int ntask = nact * half;
  const float4* xv4 = reinterpret_cast<const float4*>(xs);
  for (int task = blockIdx.x + gridDim.x * warp; task < ntask; task += gridDim.x * kGemvWarps) {
    const int ai = task / half;
    const int f0 = (task - ai * half) * 2;
    const int e = s_active[ai];
    uint4 q[2][2][NBL];
    uint32_t s[2][2][NBL];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const size_t row = (size_t)e * F + f0 + r;
#pragma unroll
      for (int j = 0; j < NBL; ++j) {
        const int b = lane + 32 * j;
        if (b < nb) {
          q[0][r][j] = ldg_nc_v4(g_qs + row * (D / 2) + (size_t)b * 16);
          q[1][r][j] = ldg_nc_v4(u_qs + row * (D / 2) + (size_t)b * 16);
          s[0][r][j] = ldg_nc_u8(g_sc + row * nb + b);
          s[1][r][j] = ldg_nc_u8(u_sc + row * nb + b);
        }
      }
    }
    const int cnt = counts[e];
    const int pb = basep[e];
    for (int tok = 0; tok < cnt; ++tok) {
      const int a = rows[pb + tok];
      const int t = a / k;
      const float4* xt = xv4 + (size_t)t * (D >> 2);
      float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
      for (int j = 0; j < NBL; ++j) {
        const int b = lane + 32 * j;
        if (b < nb) {
          float4 xv[8];
          load_pair_group(xt, b, xv);
#pragma unroll
          for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int r = 0; r < 2; ++r)
              acc[m][r] = fmaf(mx_block_dot(q[m][r][j], xv), e8m0_to_f32(s[m][r][j]), acc[m][r]);
        }
      }
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int r = 0; r < 2; ++r) acc[m][r] = warp_sum(acc[m][r]);
      if (lane < 2) {
        const int f = f0 + lane;
        const float gv = (lane == 0 ? acc[0][0] : acc[0][1]) + (bg ? bg[(size_t)e * F + f] : 0.f);
        const float uv = (lane == 0 ? acc[1][0] : acc[1][1]) + (bu ? bu[(size_t)e * F + f] : 0.f);
        h[(size_t)a * F + pairswz_offset(f)] = swiglu_oai_f(gv, uv, alpha, limit);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Fused down + bias + router-weighted combine in slot order.
// Task = pair of output rows c0, c0+1: each warp loads those rows of every
// active expert (up to kDownGroup experts in flight at once), dots them with
// the h rows of that expert's assignments, then lanes t < T sum the k slots of
// token t in slot order.
// ---------------------------------------------------------------------------
constexpr int kDownGroup = 4;

template <int NBL>
__global__ void __launch_bounds__(kGemvThreads) gemv_down_combine_kernel(
    const uint8_t* __restrict__ d_qs, const uint8_t* __restrict__ d_sc, const float* __restrict__ bd,
    int E, int D, int F, int T, int k, const float* __restrict__ h, const int32_t* __restrict__ ids,
    const float* __restrict__ w, const int32_t* __restrict__ counts,
    const int32_t* __restrict__ basep, const int32_t* __restrict__ rows, int h_in_smem,
    float* __restrict__ y) {
  extern __shared__ float4 smem_f4[];
  __shared__ int s_active[256];
  __shared__ float s_o[kGemvWarps][64][2];  // per warp: o[a][r] for a < T*k <= 64
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  pdl_launch_dependents();
  pdl_wait();
  const int TK = T * k;
  const float4* hv4;
  if (h_in_smem) {
    const float4* src = reinterpret_cast<const float4*>(h);
    const int n4 = TK * (F >> 2);
    for (int i = threadIdx.x; i < n4; i += blockDim.x) smem_f4[i] = src[i];
    hv4 = smem_f4;
  } else {
    hv4 = reinterpret_cast<const float4*>(h);
  }
  const int nact = build_active(counts, E, s_active);  // includes __syncthreads
  const int nb = F >> 5;
  const int ntask = D >> 1;
  for (int task = blockIdx.x + gridDim.x * warp; task < ntask; task += gridDim.x * kGemvWarps) {
    const int c0 = task * 2;
    for (int g0 = 0; g0 < nact; g0 += kDownGroup) {
      uint4 q[kDownGroup][2][NBL];
      uint32_t s[kDownGroup][2][NBL];
#pragma unroll
      for (int g = 0; g < kDownGroup; ++g) {
        if (g0 + g < nact) {
          const int e = s_active[g0 + g];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const size_t row = (size_t)e * D + c0 + r;
#pragma unroll
            for (int j = 0; j < NBL; ++j) {
              const int b = lane + 32 * j;
              if (b < nb) {
                q[g][r][j] = ldg_nc_v4(d_qs + row * (F / 2) + (size_t)b * 16);
                s[g][r][j] = ldg_nc_u8(d_sc + row * nb + b);
              }
            }
          }
        }
      }
#pragma unroll
      for (int g = 0; g < kDownGroup; ++g) {
        if (g0 + g < nact) {
          const int e = s_active[g0 + g];
          const int cnt = counts[e];
          const int pb = basep[e];
          for (int tok = 0; tok < cnt; ++tok) {
            const int a = rows[pb + tok];
            const float4* ha = hv4 + (size_t)a * (F >> 2);
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int j = 0; j < NBL; ++j) {
              const int b = lane + 32 * j;
              if (b < nb) {
                float4 xv[8];
                load_pair_group(ha, b, xv);
                acc0 = fmaf(mx_block_dot(q[g][0][j], xv), e8m0_to_f32(s[g][0][j]), acc0);
                acc1 = fmaf(mx_block_dot(q[g][1][j], xv), e8m0_to_f32(s[g][1][j]), acc1);
              }
            }
            acc0 = warp_sum(acc0);
            acc1 = warp_sum(acc1);
            if (lane == 0) {
              s_o[warp][a][0] = acc0;
              s_o[warp][a][1] = acc1;
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane < T) {
      const int t = lane;
      float y0 = 0.f, y1 = 0.f;
      for (int j = 0; j < k; ++j) {  // slot order
        const int a = t * k + j;
        const int e = ids[a];
        const float wt = w[a];
        const float b0 = bd ? bd[(size_t)e * D + c0] : 0.f;
        const float b1 = bd ? bd[(size_t)e * D + c0 + 1] : 0.f;
        y0 = fmaf(wt, s_o[warp][a][0] + b0, y0);
        y1 = fmaf(wt, s_o[warp][a][1] + b1, y1);
      }
      y[(size_t)t * D + c0] = y0;
      y[(size_t)t * D + c0 + 1] = y1;
    }
    __syncwarp();
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

size_t gemv_gateup_smem_bytes(int T, int D) { return (size_t)T * D * sizeof(float); }

size_t gemv_down_smem_bytes(int T, int k, int F) {
  const size_t b = (size_t)T * k * F * sizeof(float);
  return b <= 160 * 1024 ? b : 0;  // 0: read h from global memory
}

cudaError_t launch_gemv_gateup_swiglu(const uint8_t* g_qs, const uint8_t* g_sc, const float* bg,
                                      const uint8_t* u_qs, const uint8_t* u_sc, const float* bu,
                                      int E, int F, int D, int T, int k, const float* x,
                                      const int32_t* counts, const int32_t* basep,
                                      const int32_t* rows, float alpha, float limit, float* h,
                                      Launch L) {
  if (T <= 0) return cudaSuccess;
  const size_t smem = gemv_gateup_smem_bytes(T, D);
  const int sms = device_sm_count();
  dim3 grid(sms);
  const int nbl = ((D >> 5) + 31) / 32;
  cudaError_t err;
#define MOE_GU_CASE(N)                                                                           \
  case N:                                                                                        \
    if ((err = set_smem(gemv_gateup_swiglu_kernel<N>, smem)) != cudaSuccess) return err;         \
    grid = dim3(sms * resident_blocks_per_sm(gemv_gateup_swiglu_kernel<N>, kGemvThreads, smem));  \
    return launch_kernel(gemv_gateup_swiglu_kernel<N>, grid, dim3(kGemvThreads), smem, L, g_qs,  \
                         g_sc, bg, u_qs, u_sc, bu, E, F, D, T, k, x, counts, basep, rows, alpha, \
                         limit, h);
  switch (nbl) {
    MOE_GU_CASE(1)
    MOE_GU_CASE(2)
    MOE_GU_CASE(3)
    MOE_GU_CASE(4)
    default:
      return cudaErrorInvalidValue;
  }
#undef MOE_GU_CASE
}

cudaError_t launch_gemv_down_combine(const uint8_t* d_qs, const uint8_t* d_sc, const float* bd,
                                     int E, int D, int F, int T, int k, const float* h,
                                     const int32_t* ids, const float* w, const int32_t* counts,
                                     const int32_t* basep, const int32_t* rows, float* y,
                                     Launch L) {
  if (T <= 0) return cudaSuccess;
  const size_t smem = gemv_down_smem_bytes(T, k, F);
  const int h_in_smem = smem > 0 ? 1 : 0;
  const int sms = device_sm_count();
  dim3 grid(sms);
  const int nbl = ((F >> 5) + 31) / 32;
  cudaError_t err;
#define MOE_DN_CASE(N)                                                                           \
  case N:                                                                                        \
    if ((err = set_smem(gemv_down_combine_kernel<N>, smem)) != cudaSuccess) return err;          \
    grid = dim3(sms * resident_blocks_per_sm(gemv_down_combine_kernel<N>, kGemvThreads, smem));   \
    return launch_kernel(gemv_down_combine_kernel<N>, grid, dim3(kGemvThreads), smem, L, d_qs,   \
                         d_sc, bd, E, D, F, T, k, h, ids, w, counts, basep, rows, h_in_smem, y);
  switch (nbl) {
    MOE_DN_CASE(1)
    MOE_DN_CASE(2)
    MOE_DN_CASE(3)
    MOE_DN_CASE(4)
    default:
      return cudaErrorInvalidValue;
  }
#undef MOE_DN_CASE
}

}  // namespace moe
