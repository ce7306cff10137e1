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
// Decode-rail routing table, built in shared memory by one warp per CTA from
// the router logits (top-k + softmax, the same routine as moe_route_topk) or
// from given ids: the active experts in ascending order and, per expert, its
// assignments a = t*k + j in ascending order. T*k <= 64.
// ---------------------------------------------------------------------------
constexpr int kMaxAssign = 64;

struct DecodeRouting {
  int nact;
  int act_e[kMaxAssign];
  int act_off[kMaxAssign + 1];
  int lst[kMaxAssign];
  int ids[kMaxAssign];
  float w[kMaxAssign];
  unsigned mask[8];
  int cnt[kMaxAssign];
  int rank[kMaxAssign];
  int idx[kMaxAssign];
};

__device__ __forceinline__ void build_routing(DecodeRouting& R, int TK, int E, int lane, int* status) {
  if (lane < 8) R.mask[lane] = 0u;
  __syncwarp();
  for (int a = lane; a < TK; a += 32) {
    const int e = R.ids[a];
    if (e >= 0 && e < E) {
      atomicOr(&R.mask[e >> 5], 1u << (e & 31));
    } else {
      set_status(status, 0x1);
    }
  }
  __syncwarp();
  int nact = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) nact += __popc(R.mask[i]);
  for (int a = lane; a < TK; a += 32) {
    const int e = R.ids[a];
    if (e < 0 || e >= E) continue;
    int ix = __popc(R.mask[e >> 5] & ((1u << (e & 31)) - 1u));
    for (int i = 0; i < (e >> 5); ++i) ix += __popc(R.mask[i]);
    int rank = 0, cnt = 0;
    for (int b = 0; b < TK; ++b) {
      const bool same = (R.ids[b] == e);
      cnt += same;
      rank += same && (b < a);
    }
    R.act_e[ix] = e;
    R.cnt[ix] = cnt;
    R.rank[a] = rank;
    R.idx[a] = ix;
  }
  __syncwarp();
  for (int i = lane; i < nact; i += 32) {
    int off = 0;
    for (int j = 0; j < i; ++j) off += R.cnt[j];
    R.act_off[i] = off;
    if (i == nact - 1) R.act_off[nact] = off + R.cnt[i];
  }
  __syncwarp();
  for (int a = lane; a < TK; a += 32) {
    const int e = R.ids[a];
    if (e >= 0 && e < E) R.lst[R.act_off[R.idx[a]] + R.rank[a]] = a;
  }
  if (lane == 0) R.nact = nact;
  __syncwarp();
}

// Fills R.ids / R.w for T tokens: top-k + softmax of the logits, or the given ids (and weights).
__device__ __forceinline__ void routing_inputs(DecodeRouting& R, int T, int k, int E, int lane,
                                               const float* __restrict__ logits,
                                               const int32_t* __restrict__ ids_in,
                                               const float* __restrict__ w_in) {
  if (logits) {
    for (int t = 0; t < T; ++t) {
      int id;
      float wt;
      warp_topk_softmax(logits + (size_t)t * E, E, k, lane, id, wt);
      if (lane < k) {
        R.ids[t * k + lane] = id;
        R.w[t * k + lane] = wt;
      }
    }
  } else {
    for (int a = lane; a < T * k; a += 32) {
      R.ids[a] = ids_in[a];
      R.w[a] = w_in ? w_in[a] : 0.f;
    }
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// Fused gate/up + bias + swiglu (stage 0 of the decode expert chain).
// Task = (active expert, rows f0, f0+1). Warp 0 streams each task's two gate
// rows and two up rows (2*D bytes, contiguous per matrix) into a ring of
// shared-memory stages with TMA bulk copies; consumer warps 1..8 take the
// CTA's tasks round-robin, read the nibbles from shared memory, and apply
// them to every token routed to the expert. The E8M0 bytes are loaded by the
// consumer lanes one task ahead. h[a] is written block-pair ordered.
// ---------------------------------------------------------------------------
constexpr int kGvConsumers = 12;
constexpr int kGvThreads = (kGvConsumers + 1) * 32;
constexpr int kGvMaxStages = 48;

template <int NBL>
__global__ void __launch_bounds__(kGvThreads, 1) gemv_gateup_kernel(
    const uint8_t* __restrict__ g_qs, const uint8_t* __restrict__ g_sc, const float* __restrict__ bg,
    const uint8_t* __restrict__ u_qs, const uint8_t* __restrict__ u_sc, const float* __restrict__ bu,
    int E, int F, int D, int T, int k, const float* __restrict__ x, const float* __restrict__ logits,
    const int32_t* __restrict__ ids_in, int32_t* __restrict__ ids_out, float* __restrict__ w_out,
    float alpha, float limit, float* __restrict__ h, int nstages, int* status) {
  extern __shared__ float4 smem_f4[];
  float* xs = reinterpret_cast<float*>(smem_f4);                         // [T][D] block-pair order
  uint8_t* ring = reinterpret_cast<uint8_t*>(smem_f4) + (size_t)T * D * 4;  // nstages x 2D bytes
  __shared__ DecodeRouting R;
  __shared__ __align__(8) uint64_t full_bar[kGvMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kGvMaxStages];
  __shared__ int s_abort;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  pdl_launch_dependents();
  for (int t = 0; t < T; ++t) stage_pairswz(xs + (size_t)t * D, x + (size_t)t * D, D);
  if (threadIdx.x == 0) {
    for (int i = 0; i < nstages; ++i) {
      tc::mbar_init(tc::smem_u32(&full_bar[i]), 1);
      tc::mbar_init(tc::smem_u32(&empty_bar[i]), 1);
    }
    s_abort = 0;
    tc::fence_mbar_init();
  }
  pdl_wait();  // router logits / ids come from the previous kernel
  if (warp == 0) {
    routing_inputs(R, T, k, E, lane, logits, ids_in, nullptr);
    build_routing(R, T * k, E, lane, status);
    if (blockIdx.x == 0 && ids_out)
      for (int a = lane; a < T * k; a += 32) {
        ids_out[a] = R.ids[a];
        if (w_out) w_out[a] = R.w[a];
      }
  }
  __syncthreads();
  const int nact = R.nact;
  const int nb = D >> 5;
  const int half = F >> 1;
  const int ntask = nact * half;
  const int G = gridDim.x;
  const uint32_t stage_bytes = (uint32_t)(2 * D);
  const int spc = nstages / kGvConsumers;  // stages owned by each consumer warp
  const volatile int* abort_flag = &s_abort;

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      for (int m = 0;; ++m) {
        const int i = blockIdx.x + G * m;
        if (i >= ntask) break;
        const int ai = i / half;
        const int f0 = (i - ai * half) * 2;
        const int e = R.act_e[ai];
        const int j = m / kGvConsumers;  // the consumer's own task counter
        const int s = (m % kGvConsumers) * spc + j % spc, n = j / spc;
        if (n > 0 && !tc::mbar_wait(tc::smem_u32(&empty_bar[s]), (n - 1) & 1, abort_flag)) {
          s_abort = 1;
          report_timeout(status, 1, 0, s, m);
          break;
        }
        const uint32_t fb = tc::smem_u32(&full_bar[s]);
        const uint32_t dst = tc::smem_u32(ring + (size_t)s * stage_bytes);
        tc::mbar_expect_tx(fb, stage_bytes);
        tc::bulk_load(dst, g_qs + ((size_t)e * F + f0) * (D / 2), (uint32_t)D, fb);
        tc::bulk_load(dst + D, u_qs + ((size_t)e * F + f0) * (D / 2), (uint32_t)D, fb);
        issued = m + 1;
      }
      if (s_abort)  // let every copy already issued land before shared memory goes away
        for (int m = (issued > 2 * nstages ? issued - 2 * nstages : 0); m < issued; ++m) {
          const int j = m / kGvConsumers;
          tc::mbar_wait(tc::smem_u32(&full_bar[(m % kGvConsumers) * spc + j % spc]), (j / spc) & 1, nullptr);
        }
    }
  } else {
    const int cw = warp - 1;
    const float4* xv4 = reinterpret_cast<const float4*>(xs);
    uint32_t sc_cur[2][2][NBL], sc_nxt[2][2][NBL];
    auto load_scales = [&](int i, uint32_t (&sc)[2][2][NBL]) {
      const int ai = i / half;
      const int f0 = (i - ai * half) * 2;
      const int e = R.act_e[ai];
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int j = 0; j < NBL; ++j) {
          const int b = lane + 32 * j;
          if (b < nb) {
            const size_t row = (size_t)e * F + f0 + r;
            sc[0][r][j] = ldg_nc_u8(g_sc + row * nb + b);
            sc[1][r][j] = ldg_nc_u8(u_sc + row * nb + b);
          }
        }
    };
    int m = cw;
    if (blockIdx.x + G * m < ntask) load_scales(blockIdx.x + G * m, sc_cur);
    for (; blockIdx.x + G * m < ntask; m += kGvConsumers) {
      const int i = blockIdx.x + G * m;
      const int inext = blockIdx.x + G * (m + kGvConsumers);
      if (inext < ntask) load_scales(inext, sc_nxt);
      const int ai = i / half;
      const int f0 = (i - ai * half) * 2;
      const int e = R.act_e[ai];
      const int j = m / kGvConsumers;
      const int s = cw * spc + j % spc, n = j / spc;
      if (!tc::mbar_wait(tc::smem_u32(&full_bar[s]), n & 1, abort_flag)) {
        s_abort = 1;
        report_timeout(status, 1, 1, s, m);
        break;
      }
      const uint8_t* st = ring + (size_t)s * stage_bytes;
      uint4 q[2][2][NBL];
#pragma unroll
      for (int mat = 0; mat < 2; ++mat)
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int j = 0; j < NBL; ++j) {
            const int b = lane + 32 * j;
            if (b < nb)
              q[mat][r][j] = *reinterpret_cast<const uint4*>(st + mat * D + r * (D / 2) + b * 16);
          }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tc::smem_u32(&empty_bar[s]));  // the stage is in registers now
      for (int li = R.act_off[ai]; li < R.act_off[ai + 1]; ++li) {
        const int a = R.lst[li];
        const float4* xt = xv4 + (size_t)(a / k) * (D >> 2);
        float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
        for (int j = 0; j < NBL; ++j) {
          const int b = lane + 32 * j;
          if (b < nb) {
            float4 xv[8];
            load_pair_group(xt, b, xv);
#pragma unroll
            for (int mat = 0; mat < 2; ++mat)
#pragma unroll
              for (int r = 0; r < 2; ++r)
                acc[mat][r] = fmaf(mx_block_dot(q[mat][r][j], xv), e8m0_to_f32(sc_cur[mat][r][j]), acc[mat][r]);
          }
        }
#pragma unroll
        for (int mat = 0; mat < 2; ++mat)
#pragma unroll
          for (int r = 0; r < 2; ++r) acc[mat][r] = warp_sum(acc[mat][r]);
        if (lane < 2) {
          const int f = f0 + lane;
          const float gv = (lane == 0 ? acc[0][0] : acc[0][1]) + (bg ? bg[(size_t)e * F + f] : 0.f);
          const float uv = (lane == 0 ? acc[1][0] : acc[1][1]) + (bu ? bu[(size_t)e * F + f] : 0.f);
          h[(size_t)a * F + pairswz_offset(f)] = swiglu_oai_f(gv, uv, alpha, limit);
        }
      }
#pragma unroll
      for (int mat = 0; mat < 2; ++mat)
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int j = 0; j < NBL; ++j) sc_cur[mat][r][j] = sc_nxt[mat][r][j];
    }
  }
}

// ---------------------------------------------------------------------------
// Fused down + bias + router-weighted combine in slot order (stage 1).
// A CTA owns output rows c = blockIdx.x + G*m; for each it needs row c of
// every active expert's down matrix (F/2 nibble bytes each). Warp 0 streams
// them in (row, expert) order into stages owned by the consumer of that row
// (warp m % kGvConsumers), which dots each expert's row with the h rows of that
// expert's assignments, then lets lanes t < T sum the k slots of token t in
// slot order.
// ---------------------------------------------------------------------------
template <int NBL>
__global__ void __launch_bounds__(kGvThreads) gemv_down_kernel(
    const uint8_t* __restrict__ d_qs, const uint8_t* __restrict__ d_sc, const float* __restrict__ bd,
    int E, int D, int F, int T, int k, const float* __restrict__ h, const float* __restrict__ logits,
    const int32_t* __restrict__ ids_in, const float* __restrict__ w_in, float* __restrict__ y,
    int nstages, int h_in_smem, int* status) {
  extern __shared__ float4 smem_f4[];
  const int TK = T * k;
  const size_t h_bytes = h_in_smem ? (size_t)TK * F * 4 : 0;
  uint8_t* ring = reinterpret_cast<uint8_t*>(smem_f4) + h_bytes;  // nstages x F/2 bytes
  __shared__ DecodeRouting R;
  __shared__ __align__(8) uint64_t full_bar[kGvMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kGvMaxStages];
  __shared__ float s_o[kGvConsumers][kMaxAssign];
  __shared__ int s_abort;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int i = 0; i < nstages; ++i) {
      tc::mbar_init(tc::smem_u32(&full_bar[i]), 1);
      tc::mbar_init(tc::smem_u32(&empty_bar[i]), 1);
    }
    s_abort = 0;
    tc::fence_mbar_init();
  }
  pdl_wait();  // h (and the logits) come from earlier kernels
  const float4* hv4;
  if (h_in_smem) {
    const float4* src = reinterpret_cast<const float4*>(h);
    const int n4 = TK * (F >> 2);
    for (int i = threadIdx.x; i < n4; i += blockDim.x) smem_f4[i] = src[i];
    hv4 = smem_f4;
  } else {
    hv4 = reinterpret_cast<const float4*>(h);
  }
  if (warp == 0) {
    routing_inputs(R, T, k, E, lane, logits, ids_in, w_in);
    build_routing(R, TK, E, lane, nullptr);
  }
  __syncthreads();
  const int nact = R.nact;
  if (nact == 0) return;
  const int nb = F >> 5;
  const int G = gridDim.x;
  const int nmine = blockIdx.x < D ? (D - 1 - blockIdx.x) / G + 1 : 0;  // rows of this CTA
  const uint32_t stage_bytes = (uint32_t)(F / 2);
  const int spc = nstages / kGvConsumers;  // stages owned by each consumer warp
  const volatile int* abort_flag = &s_abort;

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      for (int u = 0; u < nmine * nact; ++u) {
        const int m = u / nact, ai = u - m * nact;
        const int c = blockIdx.x + G * m;
        const int e = R.act_e[ai];
        const int j = (m / kGvConsumers) * nact + ai;  // the consumer's own step counter
        const int s = (m % kGvConsumers) * spc + j % spc, n = j / spc;
        if (n > 0 && !tc::mbar_wait(tc::smem_u32(&empty_bar[s]), (n - 1) & 1, abort_flag)) {
          s_abort = 1;
          report_timeout(status, 2, 0, s, u);
          break;
        }
        const uint32_t fb = tc::smem_u32(&full_bar[s]);
        tc::mbar_expect_tx(fb, stage_bytes);
        tc::bulk_load(tc::smem_u32(ring + (size_t)s * stage_bytes), d_qs + ((size_t)e * D + c) * (F / 2),
                      stage_bytes, fb);
        issued = u + 1;
      }
      if (s_abort)  // let every copy already issued land before shared memory goes away
        for (int u = (issued > 2 * nstages ? issued - 2 * nstages : 0); u < issued; ++u) {
          const int m = u / nact, ai = u - m * nact;
          const int j = (m / kGvConsumers) * nact + ai;
          tc::mbar_wait(tc::smem_u32(&full_bar[(m % kGvConsumers) * spc + j % spc]), (j / spc) & 1, nullptr);
        }
    }
  } else {
    const int cw = warp - 1;
    for (int m = cw; m < nmine; m += kGvConsumers) {
      const int c = blockIdx.x + G * m;
      bool ok = true;
      uint32_t sc_nxt[NBL];
      auto load_scales = [&](int ai, uint32_t (&scl)[NBL]) {
        const int e = R.act_e[ai];
#pragma unroll
        for (int jb = 0; jb < NBL; ++jb) {
          const int b = lane + 32 * jb;
          if (b < nb) scl[jb] = ldg_nc_u8(d_sc + ((size_t)e * D + c) * nb + b);
        }
      };
      load_scales(0, sc_nxt);
      for (int ai = 0; ai < nact; ++ai) {
        uint32_t scl[NBL];
#pragma unroll
        for (int jb = 0; jb < NBL; ++jb) scl[jb] = sc_nxt[jb];
        if (ai + 1 < nact) load_scales(ai + 1, sc_nxt);
        const int u = m * nact + ai;
        const int j = (m / kGvConsumers) * nact + ai;
        const int s = cw * spc + j % spc, n = j / spc;
        if (!tc::mbar_wait(tc::smem_u32(&full_bar[s]), n & 1, abort_flag)) {
          s_abort = 1;
          report_timeout(status, 2, 1, s, u);
          ok = false;
          break;
        }
        const uint8_t* st = ring + (size_t)s * stage_bytes;
        uint4 q[NBL];
#pragma unroll
        for (int jb = 0; jb < NBL; ++jb) {
          const int b = lane + 32 * jb;
          if (b < nb) q[jb] = *reinterpret_cast<const uint4*>(st + b * 16);
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_u32(&empty_bar[s]));
        for (int li = R.act_off[ai]; li < R.act_off[ai + 1]; ++li) {
          const int a = R.lst[li];
          const float4* ha = hv4 + (size_t)a * (F >> 2);
          float acc = 0.f;
#pragma unroll
          for (int jb = 0; jb < NBL; ++jb) {
            const int b = lane + 32 * jb;
            if (b < nb) {
              float4 xv[8];
              load_pair_group(ha, b, xv);
              acc = fmaf(mx_block_dot(q[jb], xv), e8m0_to_f32(scl[jb]), acc);
            }
          }
          acc = warp_sum(acc);
          if (lane == 0) s_o[cw][a] = acc;
        }
      }
      if (!ok) break;
      __syncwarp();
      if (lane < T) {
        const int t = lane;
        float yv = 0.f;
        for (int jj = 0; jj < k; ++jj) {  // slot order
          const int a = t * k + jj;
          const int ej = R.ids[a];
          if (ej < 0 || ej >= E) continue;
          yv = fmaf(R.w[a], s_o[cw][a] + (bd ? bd[(size_t)ej * D + c] : 0.f), yv);
        }
        y[(size_t)t * D + c] = yv;
      }
      __syncwarp();
    }
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

// Shared memory of the decode kernels: the tokens (or h) plus weight stages,
// an equal number owned by each consumer warp (at most four each).
static int gv_stages(size_t fixed_bytes, size_t stage_bytes) {
  const size_t budget = 210 * 1024;
  size_t per = (budget > fixed_bytes) ? (budget - fixed_bytes) / (stage_bytes * kGvConsumers) : 0;
  if (per > 4) per = 4;
  return (int)per * kGvConsumers;
}

cudaError_t launch_gemv_gateup(const uint8_t* g_qs, const uint8_t* g_sc, const float* bg,
                               const uint8_t* u_qs, const uint8_t* u_sc, const float* bu, int E,
                               int F, int D, int T, int k, const float* x, const float* logits,
                               const int32_t* ids_in, int32_t* ids_out, float* w_out, float alpha,
                               float limit, float* h, int* status, Launch L) {
  if (T <= 0) return cudaSuccess;
  const size_t xbytes = (size_t)T * D * 4;
  const int nstages = gv_stages(xbytes, (size_t)2 * D);
  if (nstages < kGvConsumers) return cudaErrorInvalidValue;
  const size_t smem = xbytes + (size_t)nstages * 2 * D;
  const int sms = device_sm_count();
  const int nbl = ((D >> 5) + 31) / 32;
  cudaError_t err;
#define MOE_GU_CASE(N)                                                                              \
  case N: {                                                                                         \
    if ((err = ensure_smem_limit(gemv_gateup_kernel<N>, smem)) != cudaSuccess) return err;         \
    const dim3 grid(sms * resident_blocks_per_sm(gemv_gateup_kernel<N>, kGvThreads, smem));         \
    return launch_kernel(gemv_gateup_kernel<N>, grid, dim3(kGvThreads), smem, L, g_qs, g_sc, bg,    \
                         u_qs, u_sc, bu, E, F, D, T, k, x, logits, ids_in, ids_out, w_out, alpha,   \
                         limit, h, nstages, status);                                                \
  }
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

cudaError_t launch_gemv_down(const uint8_t* d_qs, const uint8_t* d_sc, const float* bd, int E,
                             int D, int F, int T, int k, const float* h, const float* logits,
                             const int32_t* ids_in, const float* w_in, float* y, int* status,
                             Launch L) {
  if (T <= 0) return cudaSuccess;
  size_t hbytes = (size_t)T * k * F * 4;
  int h_in_smem = 1;
  if (hbytes > 128 * 1024) {
    hbytes = 0;
    h_in_smem = 0;
  }
  const int nstages = gv_stages(hbytes, (size_t)F / 2);
  if (nstages < kGvConsumers) return cudaErrorInvalidValue;
  const size_t smem = hbytes + (size_t)nstages * (F / 2);
  const int sms = device_sm_count();
  const int nbl = ((F >> 5) + 31) / 32;
  cudaError_t err;
#define MOE_DN_CASE(N)                                                                              \
  case N: {                                                                                         \
    if ((err = ensure_smem_limit(gemv_down_kernel<N>, smem)) != cudaSuccess) return err;           \
    const dim3 grid(sms * resident_blocks_per_sm(gemv_down_kernel<N>, kGvThreads, smem));           \
    return launch_kernel(gemv_down_kernel<N>, grid, dim3(kGvThreads), smem, L, d_qs, d_sc, bd, E,   \
                         D, F, T, k, h, logits, ids_in, w_in, y, nstages, h_in_smem, status);       \
  }
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
