// Router (logits, top-k, softmax over the k) and the single-kernel expert bucket.
//
// The bucket follows the Metal fusion lane of "dasLLAMA gpt-oss arc" (third
// bullet of the fusion commit): the serial one-threadgroup prefix walk is
// folded into the bucket kernel, each expert's block computing its own padded
// base in-block and publishing basep[e]; the resulting CSR is bit-identical
// to the two-pass one.
#include <algorithm>

#include "decode_mx.cuh"

#include "moe_common.cuh"
#include "mx_terms.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Router logits: logits[t][e] = x[t] . wr[e] + br[e]
// Each block computes TT tokens x EG experts; every dot product is spread over
// G = 128 / (TT*EG) consecutive threads (float4 loads, shuffle / smem reduce).
// ---------------------------------------------------------------------------
// One block's dots (block coordinates bx over tokens, by over experts); shared
// with the decode prologue of the block-scaled rail.
template <int TT, int EG>
__device__ __forceinline__ void router_logits_block(const float* __restrict__ x, int T, int D,
                                                    const float* __restrict__ wr, const float* __restrict__ br,
                                                    int E, float* __restrict__ logits, float* __restrict__ x_copy,
                                                    int bx, int by) {
  constexpr int NDOT = TT * EG;
  constexpr int G = 128 / NDOT;
  static_assert(G * NDOT == 128, "threads per dot");
  const int tid = threadIdx.x;
  const int d = tid / G;   // which dot of this block
  const int gi = tid % G;  // thread within the dot's group
  const int t = bx * TT + d / EG;
  const int e = by * EG + d % EG;
  const bool live = (t < T) && (e < E);
  float acc = 0.f;
  if (live) {
    const float4* xr = reinterpret_cast<const float4*>(x + (size_t)t * D);
    const float4* wrr = reinterpret_cast<const float4*>(wr + (size_t)e * D);
    const int n4 = D >> 2;
    // the copy of x (if asked for) comes from the expert-0 dots of the first block column
    float4* xc = (x_copy && by == 0 && d % EG == 0) ? reinterpret_cast<float4*>(x_copy + (size_t)t * D)
                                                            : nullptr;
    float a0 = 0.f, a1 = 0.f;
    if constexpr (NDOT == 1) {
      // one dot per block (T = 1): all of the thread's loads in flight at once,
      // summed in the same order as the loop below (even steps a0, odd steps a1)
      constexpr int MAXJ = 8;  // D <= 4096
      float4 xv[MAXJ], wv[MAXJ];
#pragma unroll
      for (int j = 0; j < MAXJ; ++j)
        if (gi + G * j < n4) {
          xv[j] = xr[gi + G * j];
          wv[j] = wrr[gi + G * j];
        }
#pragma unroll
      for (int j = 0; j < MAXJ; ++j)
        if (gi + G * j < n4) {
          float& a = (j & 1) ? a1 : a0;
          a = fmaf(xv[j].x, wv[j].x, a); a = fmaf(xv[j].y, wv[j].y, a);
          a = fmaf(xv[j].z, wv[j].z, a); a = fmaf(xv[j].w, wv[j].w, a);
          if (xc) xc[gi + G * j] = xv[j];
        }
    } else {
      int i = gi;
      for (; i + G < n4; i += 2 * G) {
        const float4 xa = xr[i], wa = wrr[i];
        const float4 xb = xr[i + G], wb = wrr[i + G];
        a0 = fmaf(xa.x, wa.x, a0); a0 = fmaf(xa.y, wa.y, a0);
        a0 = fmaf(xa.z, wa.z, a0); a0 = fmaf(xa.w, wa.w, a0);
        a1 = fmaf(xb.x, wb.x, a1); a1 = fmaf(xb.y, wb.y, a1);
        a1 = fmaf(xb.z, wb.z, a1); a1 = fmaf(xb.w, wb.w, a1);
        if (xc) {
          xc[i] = xa;
          xc[i + G] = xb;
        }
      }
      for (; i < n4; i += G) {
        const float4 xa = xr[i], wa = wrr[i];
        a0 = fmaf(xa.x, wa.x, a0); a0 = fmaf(xa.y, wa.y, a0);
        a0 = fmaf(xa.z, wa.z, a0); a0 = fmaf(xa.w, wa.w, a0);
        if (xc) xc[i] = xa;
      }
    }
    acc = a0 + a1;
  }
  if constexpr (G <= 32) {
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (gi == 0 && live) logits[(size_t)t * E + e] = acc + (br ? br[e] : 0.f);
  } else {
    __shared__ float part[4];
    acc = warp_sum(acc);
    if ((tid & 31) == 0) part[tid >> 5] = acc;
    __syncthreads();
    if (gi == 0 && live) {
      float s = 0.f;
      for (int w = 0; w < G / 32; ++w) s += part[d * (G / 32) + w];
      logits[(size_t)t * E + e] = s + (br ? br[e] : 0.f);
    }
  }
}

template <int TT, int EG>
__global__ void __launch_bounds__(128) router_logits_kernel(const float* __restrict__ x, int T, int D,
                                                            const float* __restrict__ wr,
                                                            const float* __restrict__ br, int E,
                                                            float* __restrict__ logits,
                                                            float* __restrict__ x_copy) {
  pdl_launch_dependents();
  pdl_wait();
  router_logits_block<TT, EG>(x, T, D, wr, br, E, logits, x_copy, blockIdx.x, blockIdx.y);
}

// ---------------------------------------------------------------------------
// Decode prologue of the block-scaled decode rail (T <= 8): the router logits
// (blocks [0, nlog), laid out as router_logits_kernel's grid), the x operand of
// the gate/up MMAs as kDecTerms E2M1 terms per value in the operand-chunk
// layout of decode_mx.cuh (the remaining blocks, a warp per (token, 32-block)),
// and the zeroing of the expert kernels' arrival counters. x may live in
// mapped host memory: every value is read once.
// ---------------------------------------------------------------------------
template <int TT, int EG>
__global__ void __launch_bounds__(128) decode_prologue_kernel(const float* __restrict__ x, int T, int D,
                                                              const float* __restrict__ wr,
                                                              const float* __restrict__ br, int E,
                                                              float* __restrict__ logits, int nlog_x, int nlog,
                                                              uint8_t* __restrict__ xq, uint8_t* __restrict__ xsf,
                                                              int npad, int* __restrict__ zero, int nzero) {
  pdl_launch_dependents();
  pdl_wait();
  if ((int)blockIdx.x < nlog) {
    router_logits_block<TT, EG>(x, T, D, wr, br, E, logits, nullptr, blockIdx.x % nlog_x, blockIdx.x / nlog_x);
    return;
  }
  using namespace dmx;
  const int qb = blockIdx.x - nlog, nqb = gridDim.x - nlog;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = D / 32, NK = (D + 127) / 128;
  if (qb == 0)
    for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero[i] = 0;
  const int gw = qb * 4 + warp, nw = nqb * 4;
  for (int task = gw; task < T * nb; task += nw) {
    const int t = task / nb, blk = task - t * nb;
    const float v = x[(size_t)t * D + 32 * blk + lane];
    uint32_t q[kDecTerms], sc[kDecTerms];
    mx::split_terms_e2m1<kDecTerms>(v, q, sc);
    const int j = blk >> 2, kb = blk & 3;
    uint8_t* chunk = xq + (size_t)j * npad * 64;
#pragma unroll
    for (int term = 0; term < kDecTerms; ++term) {
      const int n = t * kDecTerms + term;
      const uint32_t byte = mx::pack_e2m1_block(q[term]);
      if (lane < 16) chunk[chunk_off(n, kb, lane)] = (uint8_t)byte;
      if (lane == 0) xsf[(size_t)j * 512 + atom_off(n, kb)] = (uint8_t)sc[term];
    }
  }
  // rows past T * kDecTerms: zero codes on a scale of 1
  const int npr = npad - T * kDecTerms;
  for (int task = gw; task < NK * npr; task += nw) {
    const int j = task / npr, n = T * kDecTerms + (task - j * npr);
    if (lane < 16) reinterpret_cast<uint32_t*>(xq + (size_t)j * npad * 64 + chunk_off(n, lane >> 2, 4 * (lane & 3)))[0] = 0u;
    if (lane < 4) xsf[(size_t)j * 512 + atom_off(n, lane)] = 127;
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");  // read next by the copy engine
}

// Prefill sizes (T > 8): a block takes 4 tokens x 16 experts with 16 warps:
// warp w computes 4 tokens x 4 experts (experts 4 (w % 4) ..) over one quarter
// of the dot length (w / 4), its lanes splitting that quarter in float4 steps;
// x rows come through L1 (every row is read by the block's four expert
// groups). The four partial sums of a dot are added in quarter order through
// shared memory, so the result does not depend on scheduling.
constexpr int kRouterTileT = 4;
constexpr int kRouterTileE = 16;
__global__ void __launch_bounds__(512) router_logits_tile_kernel(const float* __restrict__ x, int T, int D,
                                                                 const float* __restrict__ wr,
                                                                 const float* __restrict__ br, int E,
                                                                 float* __restrict__ logits) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float part[4][kRouterTileT * kRouterTileE];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int eg = warp & 3, kq = warp >> 2;
  const int n4 = D >> 2;
  const int q4 = (n4 + 3) >> 2;
  const int i0 = kq * q4, i1 = min(n4, i0 + q4);
  const int t0 = blockIdx.x * kRouterTileT;
  const int e0 = blockIdx.y * kRouterTileE + 4 * eg;
  const float4* xrow[kRouterTileT];
#pragma unroll
  for (int tt = 0; tt < kRouterTileT; ++tt)
    xrow[tt] = reinterpret_cast<const float4*>(x + (size_t)min(t0 + tt, T - 1) * D);
  const float4* wrow[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) wrow[j] = reinterpret_cast<const float4*>(wr + (size_t)min(e0 + j, E - 1) * D);
  float acc[kRouterTileT][4];
#pragma unroll
  for (int tt = 0; tt < kRouterTileT; ++tt)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[tt][j] = 0.f;
  auto step = [&](const float4 (&xv)[kRouterTileT], const float4 (&wv)[4]) {
#pragma unroll
    for (int tt = 0; tt < kRouterTileT; ++tt)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float a = acc[tt][j];
        a = fmaf(xv[tt].x, wv[j].x, a);
        a = fmaf(xv[tt].y, wv[j].y, a);
        a = fmaf(xv[tt].z, wv[j].z, a);
        a = fmaf(xv[tt].w, wv[j].w, a);
        acc[tt][j] = a;
      }
  };
  int i = i0 + lane;
  for (; i + 32 < i1; i += 64) {  // two steps' loads in flight before any use
    float4 xa[kRouterTileT], wa[4], xb[kRouterTileT], wb[4];
#pragma unroll
    for (int tt = 0; tt < kRouterTileT; ++tt) {
      xa[tt] = __ldg(xrow[tt] + i);
      xb[tt] = __ldg(xrow[tt] + i + 32);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      wa[j] = __ldg(wrow[j] + i);
      wb[j] = __ldg(wrow[j] + i + 32);
    }
    step(xa, wa);
    step(xb, wb);
  }
  if (i < i1) {
    float4 xa[kRouterTileT], wa[4];
#pragma unroll
    for (int tt = 0; tt < kRouterTileT; ++tt) xa[tt] = __ldg(xrow[tt] + i);
#pragma unroll
    for (int j = 0; j < 4; ++j) wa[j] = __ldg(wrow[j] + i);
    step(xa, wa);
  }
#pragma unroll
  for (int tt = 0; tt < kRouterTileT; ++tt)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float v = warp_sum(acc[tt][j]);
      if (lane == 0) part[kq][tt * kRouterTileE + 4 * eg + j] = v;
    }
  __syncthreads();
  if (threadIdx.x < kRouterTileT * kRouterTileE) {
    const int tt = threadIdx.x / kRouterTileE, el = threadIdx.x % kRouterTileE;
    const int t = t0 + tt, e = blockIdx.y * kRouterTileE + el;
    const float v = ((part[0][threadIdx.x] + part[1][threadIdx.x]) + part[2][threadIdx.x]) + part[3][threadIdx.x];
    if (t < T && e < E) logits[(size_t)t * E + e] = v + (br ? br[e] : 0.f);
  }
}

// ---------------------------------------------------------------------------
// Prefill sizes, split over the dot length: block (token tile of 64, slice s
// of D, expert tile of 32) writes part[s][t][e], the slice's partial dot, and
// the top-k kernel adds the slices in slice order (so the result does not
// depend on scheduling). Each thread holds 4 tokens x 4 experts (tokens
// tt + 16 i, experts te + 8 j) and reads them from shared-memory tiles of
// 32 columns staged by the whole block, the next tile's loads in flight
// while the current one is used. Row pitch 36 floats: a quarter-warp's
// float4 reads of 8 consecutive rows fall in 8 different bank groups.
// ---------------------------------------------------------------------------
constexpr int kRsT = 64, kRsE = 32, kRsPitch = 36;
__global__ void __launch_bounds__(128) router_splitk_kernel(const float* __restrict__ x, int T, int D,
                                                            const float* __restrict__ wr, int E, int ks,
                                                            float* __restrict__ part) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ __align__(16) float xs[kRsT][kRsPitch];
  __shared__ __align__(16) float ws[kRsE][kRsPitch];
  const int t0 = blockIdx.x * kRsT, s = blockIdx.y, e0 = blockIdx.z * kRsE;
  const int kb = s * ks, ke = min(D, kb + ks);
  const int tid = threadIdx.x, tt = tid >> 3, te = tid & 7;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  float4 xr[4], wv[2];
  auto gload = [&](int k0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = tid + 128 * i, r = idx >> 3, k = k0 + 4 * (idx & 7);
      xr[i] = (t0 + r < T && k < ke) ? __ldg(reinterpret_cast<const float4*>(x + (size_t)(t0 + r) * D + k))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int idx = tid + 128 * i, r = idx >> 3, k = k0 + 4 * (idx & 7);
      wv[i] = (e0 + r < E && k < ke) ? __ldg(reinterpret_cast<const float4*>(wr + (size_t)(e0 + r) * D + k))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  gload(kb);
  for (int k0 = kb; k0 < ke; k0 += 32) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = tid + 128 * i;
      *reinterpret_cast<float4*>(&xs[idx >> 3][4 * (idx & 7)]) = xr[i];
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int idx = tid + 128 * i;
      *reinterpret_cast<float4*>(&ws[idx >> 3][4 * (idx & 7)]) = wv[i];
    }
    __syncthreads();
    if (k0 + 32 < ke) gload(k0 + 32);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float4 a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4*>(&xs[tt + 16 * i][4 * c]);
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = *reinterpret_cast<const float4*>(&ws[te + 8 * j][4 * c]);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float v = acc[i][j];
          v = fmaf(a[i].x, b[j].x, v);
          v = fmaf(a[i].y, b[j].y, v);
          v = fmaf(a[i].z, b[j].z, v);
          v = fmaf(a[i].w, b[j].w, v);
          acc[i][j] = v;
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int t = t0 + tt + 16 * i, e = e0 + te + 8 * j;
      if (t < T && e < E) part[((size_t)s * T + t) * E + e] = acc[i][j];
    }
}

// The slices' partial dots added in slice order, plus the bias, into
// logits[t][e]; then top-k and softmax as topk_softmax_kernel. One warp per token.
__global__ void __launch_bounds__(256) topk_partials_kernel(const float* __restrict__ part, int S,
                                                            const float* __restrict__ br, int T, int E, int k,
                                                            float* __restrict__ logits, int32_t* __restrict__ ids,
                                                            float* __restrict__ w) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  for (int e = lane; e < E; e += 32) {
    float v = 0.f;
    for (int q = 0; q < S; ++q) v += part[((size_t)q * T + t) * E + e];
    logits[(size_t)t * E + e] = v + (br ? br[e] : 0.f);
  }
  __syncwarp();
  int my_id;
  float my_w;
  warp_topk_softmax(logits + (size_t)t * E, E, k, lane, my_id, my_w);
  if (lane < k) {
    ids[(size_t)t * k + lane] = my_id;
    w[(size_t)t * k + lane] = my_w;
  }
}

// ---------------------------------------------------------------------------
// Top-k then softmax over the k selected; one warp per token.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) topk_softmax_kernel(const float* __restrict__ logits, int T,
                                                           int E, int k, int32_t* __restrict__ ids,
                                                           float* __restrict__ w) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  int my_id;
  float my_w;
  warp_topk_softmax(logits + (size_t)t * E, E, k, lane, my_id, my_w);
  if (lane < k) {
    ids[(size_t)t * k + lane] = my_id;
    w[(size_t)t * k + lane] = my_w;
  }
}

// ---------------------------------------------------------------------------
// Bucket: one block per expert. Each block histograms all ids, derives its own
// padded base with a warp reduction over the lower experts, then compacts its
// assignments in ascending order with ballot/popc warp scans.
// ---------------------------------------------------------------------------
constexpr int kBucketThreads = 512;

__global__ void __launch_bounds__(kBucketThreads) bucket_kernel(const int32_t* __restrict__ ids, int n,
                                                                int E, int tile, int max_rows,
                                                                int32_t* __restrict__ counts,
                                                                int32_t* __restrict__ basep,
                                                                int32_t* __restrict__ rows,
                                                                int32_t* __restrict__ inv,
                                                                int* status) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ int hist[];  // [E]
  __shared__ int s_wtot[kBucketThreads / 32];
  __shared__ int s_base, s_mpad;
  const int e = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < E; i += kBucketThreads) hist[i] = 0;
  __syncthreads();
#pragma unroll 4
  for (int a = tid; a < n; a += kBucketThreads) {
    const int id = ids[a];
    if (id >= 0 && id < E) {
      atomicAdd(&hist[id], 1);
    } else if (e == 0) {
      set_status(status, 0x1);
      inv[a] = -1;
    }
  }
  __syncthreads();
  if (warp == 0) {
    int below = 0, all = 0;
    for (int i = lane; i < E; i += 32) {
      const int padded = ((hist[i] + tile - 1) / tile) * tile;
      all += padded;
      if (i < e) below += padded;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      below += __shfl_xor_sync(0xffffffffu, below, o);
      all += __shfl_xor_sync(0xffffffffu, all, o);
    }
    if (lane == 0) {
      s_base = below;
      s_mpad = all;
      counts[e] = hist[e];
      basep[e] = below;
      if (e == E - 1) basep[E] = all;
    }
  }
  __syncthreads();
  const int base = s_base;
  const int mine = hist[e];
  // stable compaction of the assignments that chose expert e: warp w owns the
  // ids [w L, (w + 1) L); it counts its matches, a prefix over the warps gives
  // its first row, and a second pass over its ids writes them in order (one
  // block barrier in all)
  constexpr int kWarps = kBucketThreads / 32;
  const int L = ((n + kWarps - 1) / kWarps + 31) & ~31;
  const int a0 = warp * L, a1 = min(n, a0 + L);
  int cnt = 0;
#pragma unroll 8
  for (int c = a0; c < a1; c += 32) {
    const int a = c + lane;
    cnt += __popc(__ballot_sync(0xffffffffu, a < a1 && ids[a] == e));
  }
  if (lane == 0) s_wtot[warp] = cnt;
  __syncthreads();
  int p0 = base;
  for (int w = 0; w < warp; ++w) p0 += s_wtot[w];
#pragma unroll 8
  for (int c = a0; c < a1; c += 32) {
    const int a = c + lane;
    const bool match = a < a1 && ids[a] == e;
    const uint32_t ballot = __ballot_sync(0xffffffffu, match);
    if (match) {
      const int p = p0 + __popc(ballot & ((1u << lane) - 1u));
      if (MOE_IN_BOUNDS(status, p < max_rows)) {
        rows[p] = a;
        inv[a] = p;
      }
    }
    p0 += __popc(ballot);
  }
  // pad rows of this expert's last tile
  const int padded = ((mine + tile - 1) / tile) * tile;
  for (int p = base + mine + tid; p < base + padded; p += kBucketThreads) rows[p] = -1;
  // tail past mpad
  if (e == E - 1)
    for (int p = s_mpad + tid; p < max_rows; p += kBucketThreads) rows[p] = -1;
}

// ---------------------------------------------------------------------------
// Gather token rows into bucket order as bf16 (the grouped GEMM's B operand),
// zero pad rows, and optionally zero y. One warp per bucket row. With xg_lo,
// each value is also split: hi = bf16(x), lo = bf16(x - hi), so hi + lo keeps
// 16 significant bits of x.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo_as_float(uint32_t packed, int half) {
  return __uint_as_float(half ? (packed & 0xFFFF0000u) : (packed << 16));
}

__global__ void __launch_bounds__(256) gather_bf16_kernel(const float* __restrict__ x, int T, int D,
                                                          int k, const int32_t* __restrict__ rows,
                                                          const int32_t* __restrict__ basep, int E,
                                                          uint16_t* __restrict__ xg,
                                                          uint16_t* __restrict__ xg_lo,
                                                          float* __restrict__ y_zero, int zero_pads) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int warp_global = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * 8;
  const int mpad = basep[E];
  const int n4 = D >> 2;
  for (int p = warp_global; p < mpad; p += nwarps) {
    const int a = rows[p];
    uint2* dst = reinterpret_cast<uint2*>(xg + (size_t)p * D);
    uint2* dst_lo = xg_lo ? reinterpret_cast<uint2*>(xg_lo + (size_t)p * D) : nullptr;
    if (a >= 0) {
      const float4* src = reinterpret_cast<const float4*>(x + (size_t)(a / k) * D);
      for (int i = lane; i < n4; i += 32) {
        const float4 v = src[i];
        uint2 o;
        o.x = pack_bf16x2(v.x, v.y);
        o.y = pack_bf16x2(v.z, v.w);
        dst[i] = o;
        if (dst_lo) {
          uint2 r;
          r.x = pack_bf16x2(v.x - bf16_lo_as_float(o.x, 0), v.y - bf16_lo_as_float(o.x, 1));
          r.y = pack_bf16x2(v.z - bf16_lo_as_float(o.y, 0), v.w - bf16_lo_as_float(o.y, 1));
          dst_lo[i] = r;
        }
      }
    } else if (zero_pads) {
      for (int i = lane; i < n4; i += 32) {
        dst[i] = make_uint2(0u, 0u);
        if (dst_lo) dst_lo[i] = make_uint2(0u, 0u);
      }
    }  // otherwise pad rows are left as they are (the layer never stores their MMA columns)
  }
  if (y_zero) {
    float4* y4 = reinterpret_cast<float4*>(y_zero);
    const size_t ny = (size_t)T * D / 4;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < ny;
         i += (size_t)gridDim.x * blockDim.x)
      y4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
cudaError_t launch_router_logits(const float* x, int T, int D, const float* wr, const float* br,
                                 int E, float* logits, float* x_copy, Launch L) {
  if (T <= 0) return cudaSuccess;
  if (T == 1) {
    dim3 grid(1, E);
    return launch_kernel(router_logits_kernel<1, 1>, grid, dim3(128), 0, L, x, T, D, wr, br, E,
                         logits, x_copy);
  }
  if (T <= 8) {
    // 2 tokens x 2 experts per block, a warp per dot: coalesced loads and enough
    // blocks to keep every SM's loads in flight
    dim3 grid((T + 1) / 2, (E + 1) / 2);
    return launch_kernel(router_logits_kernel<2, 2>, grid, dim3(128), 0, L, x, T, D, wr, br, E,
                         logits, x_copy);
  }
  if (x_copy) return cudaErrorInvalidValue;  // prefill sizes take x from device memory
  dim3 grid((T + kRouterTileT - 1) / kRouterTileT, (E + kRouterTileE - 1) / kRouterTileE);
  return launch_kernel(router_logits_tile_kernel, grid, dim3(512), 0, L, x, T, D, wr, br, E, logits);
}

cudaError_t launch_decode_prologue(const float* x, int T, int D, const float* wr, const float* br, int E,
                                   float* logits, uint8_t* xq, uint8_t* xsf, int npad, int* zero, int nzero,
                                   Launch L) {
  if (T <= 0 || T > 8) return cudaErrorInvalidValue;
  const int nb = D / 32;
  int nq = (T * nb + 7) / 8;
  if (nq < 1) nq = 1;
  if (nq > 64) nq = 64;
  if (T == 1) {
    const int nlog = E;
    return launch_kernel(decode_prologue_kernel<1, 1>, dim3(nlog + nq), dim3(128), 0, L, x, T, D, wr, br, E,
                         logits, 1, nlog, xq, xsf, npad, zero, nzero);
  }
  const int nlx = (T + 1) / 2, nlog = nlx * ((E + 1) / 2);
  return launch_kernel(decode_prologue_kernel<2, 2>, dim3(nlog + nq), dim3(128), 0, L, x, T, D, wr, br, E,
                       logits, nlx, nlog, xq, xsf, npad, zero, nzero);
}

namespace {
// Slices of D for the split router: about eight blocks per SM, slices a
// multiple of 32 wide, at most kRouterMaxSplits of them.
void router_split(int T, int D, int E, int& S, int& ks) {
  const int tiles = ((T + kRsT - 1) / kRsT) * ((E + kRsE - 1) / kRsE);
  int s = (8 * device_sm_count() + tiles - 1) / tiles;
  s = std::max(1, std::min(s, std::min(kRouterMaxSplits, D / 32)));
  ks = ((D + s - 1) / s + 31) / 32 * 32;
  S = (D + ks - 1) / ks;
}
}  // namespace

size_t router_partials_bytes(int T, int E) { return (size_t)kRouterMaxSplits * T * E * sizeof(float); }

cudaError_t launch_route_topk(const float* x, int T, int D, const float* wr, const float* br, int E, int k,
                              float* logits, float* part, int32_t* ids, float* w, Launch L) {
  if (T <= 0) return cudaSuccess;
  if (T <= 8 || part == nullptr) {
    cudaError_t err = launch_router_logits(x, T, D, wr, br, E, logits, nullptr, L);
    if (err != cudaSuccess) return err;
    L.pdl = true;
    return launch_topk_softmax(logits, T, E, k, ids, w, L);
  }
  int S = 1, ks = D;
  router_split(T, D, E, S, ks);
  dim3 grid((T + kRsT - 1) / kRsT, S, (E + kRsE - 1) / kRsE);
  cudaError_t err = launch_kernel(router_splitk_kernel, grid, dim3(128), 0, L, x, T, D, wr, E, ks, part);
  if (err != cudaSuccess) return err;
  L.pdl = true;
  return launch_kernel(topk_partials_kernel, dim3((T + 7) / 8), dim3(256), 0, L, (const float*)part, S, br, T, E, k,
                       logits, ids, w);
}

cudaError_t launch_topk_softmax(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                                Launch L) {
  if (T <= 0) return cudaSuccess;
  return launch_kernel(topk_softmax_kernel, dim3((T + 7) / 8), dim3(256), 0, L, logits, T, E, k,
                       ids, w);
}

cudaError_t launch_bucket(const int32_t* ids, int T, int k, int E, int tile, int max_rows,
                          int32_t* counts, int32_t* basep, int32_t* rows, int32_t* inv,
                          int* status, Launch L) {
  return launch_kernel(bucket_kernel, dim3(E), dim3(kBucketThreads), sizeof(int) * (size_t)E, L,
                       ids, T * k, E, tile, max_rows, counts, basep, rows, inv, status);
}

cudaError_t launch_gather_bf16(const float* x, int T, int D, int k, const int32_t* rows,
                               const int32_t* basep, int E, int max_rows, uint16_t* xg,
                               uint16_t* xg_lo, float* y_zero, bool zero_pads, Launch L) {
  int blocks = (max_rows + 7) / 8;
  const int cap = device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_kernel(gather_bf16_kernel, dim3(blocks), dim3(256), 0, L, x, T, D, k, rows, basep,
                       E, xg, xg_lo, y_zero, zero_pads ? 1 : 0);
}

}  // namespace moe
