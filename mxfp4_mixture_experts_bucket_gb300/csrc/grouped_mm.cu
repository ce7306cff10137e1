// Prefill rail: per-expert MXFP4 grouped GEMM on the tcgen05 tensor cores.
//
// Design source: MetalMoeMulMmMx4 of the Metal fusion lane ("dasLLAMA gpt-oss
// arc", fusion commit, first bullet: the expert's bias row seeds the
// accumulator tiles; the per-layer bias dispatches fold away) and its A-stage
// (block load + E2M1 table + computed E8M0, "dasLLAMA: dig the last two board
// reds green", section "gpt-oss: mx4 kernels to the lab-winning shape"); the
// 128-row tile height of the MoE tensor pair ("dasLLAMA: M5 pp deep-dense -
// board v8", section "Claims - stated, not tested"); ghost rows past the last
// bucket's padded end exit early (fusion commit, second bullet).
//
// GB300 mapping (one CTA per 128 weight rows x one 128-row bucket tile):
//   warp 0      TMA producer of the MXFP4 nibble tiles (3D map [E][R][C/2])
//               into a raw ring as deep as shared memory allows (HBM latency
//               is hidden here), plus the tile's E8M0 rows (one bulk copy)
//   warp 1      TMEM owner and single-thread tcgen05.mma issuer
//   warp 2      TMA producer of the bf16 activation tiles (2D map, 128-byte
//               swizzle, only the live 32-row chunks) into its own ring, whose
//               depth grows as the tile's live rows shrink
//   warps 3-18  two groups of eight dequantise MXFP4 -> bf16 into the UMMA
//               128B-swizzled K-major layout, alternate k-steps each, so two
//               dequant chains are in flight (three-stage hand-off ring); the
//               first group seeds the accumulator with the bias (tcgen05.st);
//               all sixteen run the epilogue from TMEM (tcgen05.ld)
// The MMA is "swap-AB": weight rows fill M = 128 and the bucket rows fill N,
// rounded up to 16, so rows past counts[e] cost no tensor work.
#include <cuda.h>

#include "tcgen05.cuh"

namespace moe {
namespace mm {

constexpr int BM = 128;  // weight rows per tile (MMA M)
constexpr int BN = 128;  // bucket rows per tile (CSR tile height, MMA N <= BN)
constexpr int BK = 64;   // reduction columns per stage (one 128-byte bf16 row)
constexpr int OSA = 3;   // dequantised A stages (dequant -> MMA hand-off)
constexpr int MAX_RS = 16;   // raw MXFP4 stages (HBM latency is hidden here)
constexpr int MAX_BS = 8;    // activation (B) stages
constexpr int kDqGroups = 2;     // dequant groups, taking alternate k-steps
constexpr int kThreads = (3 + 8 * kDqGroups) * 32;  // 19 warps
constexpr int kDqWarp0 = 3;      // warps 3..18 dequantise (group g: warps 3+8g..10+8g) and run the epilogue
constexpr int kDqThreads = 256;  // per group
constexpr int kDqWarps = kDqThreads / 32;  // hand-off barriers count one arrival per warp
constexpr int kATile = BM * BK * 2;      // 16 KB
constexpr int kBChunk = 32 * BK * 2;     // 4 KB: 32 activation rows
constexpr int kBPool = 64 * 1024;        // activation ring, carved per tile
constexpr int kRawTile = BM * (BK / 2);  // 4 KB of nibbles
constexpr uint32_t kSmemLimit = 232448;  // 227 KB opt-in per block

struct Params {
  const uint8_t* w_sc[2];
  const float* bias[2];
  int E, R, C;
  const int32_t* counts;
  const int32_t* basep;
  const int32_t* rows;
  int k;
  const float* weights;
  float alpha, limit;
  void* out;
  int64_t out_ld;
  int64_t out_rows;  // rows of out, 0 if unknown (bounds checks of the checked build)
  int* status;
  int box_rows;  // rows of one weight TMA box: min(BM, R)
  int wrs;       // weight row stride in rows: 1, or 2 for gate/up rows interleaved in one plane
};

// Shared-memory plan (identical on host and device): A ring, activation pool,
// raw ring as deep as the remaining space allows, the tile's E8M0 rows,
// barriers, small per-tile tables.
struct Layout {
  uint32_t a, b, raw, sc, bars, misc, total;
  uint32_t sc_stride;  // bytes per matrix
  int rs;              // raw stages
};

__host__ __device__ inline Layout make_layout(int nmat, int C) {
  Layout L;
  L.a = 0;
  L.b = OSA * nmat * kATile;
  L.raw = L.b + kBPool;
  L.sc_stride = (uint32_t)((BM * (C / 32) + 15) & ~15);
  const uint32_t sc_size = nmat * L.sc_stride;
  const uint32_t tail = 64 * 8 + (BN * 8 + 64) + 1024;  // barriers, tables, alignment slack
  const uint32_t budget = kSmemLimit - L.raw - sc_size - tail;
  int rs = (int)(budget / (uint32_t)(nmat * kRawTile));
  L.rs = rs > MAX_RS ? MAX_RS : rs;
  L.sc = L.raw + L.rs * nmat * kRawTile;
  L.bars = (L.sc + sc_size + 7) & ~7u;
  L.misc = L.bars + 64 * 8;
  L.total = L.misc + BN * 8 + 64 + 1024;
  return L;
}

// barrier indices
constexpr int kRawFull = 0;
constexpr int kRawEmpty = kRawFull + MAX_RS;
constexpr int kAFull = kRawEmpty + MAX_RS;
constexpr int kAEmpty = kAFull + OSA;
constexpr int kBFull = kAEmpty + OSA;
constexpr int kBEmpty = kBFull + MAX_BS;
constexpr int kAccFull = kBEmpty + MAX_BS;
constexpr int kScFull = kAccFull + 1;
constexpr int kBiasReady = kScFull + 1;
constexpr int kTFree = kBiasReady + 1;  // the epilogue warps and the MMA thread are done with tensor memory
constexpr int kNumBars = kTFree + 1;
static_assert(kNumBars <= 64, "barrier space");

// f16x2 (unscaled E2M1 pair) * 2^(s-127) -> bf16x2, exact whenever representable.
__device__ __forceinline__ uint32_t scale_to_bf16x2(uint32_t h2, float scale) {
  const float2 f = f16x2_to_float2(h2);
  __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
  return *reinterpret_cast<uint32_t*>(&b);
}

// One MXFP4 block (16 bytes, 32 elements) -> 32 bf16 in natural column order.
// o[w] holds columns 2w, 2w+1. The nibbles of two neighbouring columns are
// first gathered into one byte so that each hardware e2m1x2 conversion yields
// an adjacent pair.
__device__ __forceinline__ void dequant_block_bf16(uint4 q, float scale, uint32_t (&o)[16]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint32_t lo = w[m] & 0x0F0F0F0Fu;         // columns 4m..4m+3, one per byte
    const uint32_t hi = (w[m] >> 4) & 0x0F0F0F0Fu;  // columns 16+4m..16+4m+3
    const uint32_t pl = lo | (lo >> 4);  // byte0: (4m, 4m+1), byte2: (4m+2, 4m+3)
    const uint32_t ph = hi | (hi >> 4);
    o[2 * m] = scale_to_bf16x2(e2m1x2_to_f16x2(pl, 0), scale);
    o[2 * m + 1] = scale_to_bf16x2(e2m1x2_to_f16x2(pl, 2), scale);
    o[8 + 2 * m] = scale_to_bf16x2(e2m1x2_to_f16x2(ph, 0), scale);
    o[8 + 2 * m + 1] = scale_to_bf16x2(e2m1x2_to_f16x2(ph, 2), scale);
  }
}

template <int NMAT, int EPI, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_mm_kernel(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                      const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_alo,
                      const Params p) {
  constexpr int NB = SPLIT ? 2 : 1;  // activation tiles per stage (hi, lo)
  // TMEM columns per matrix. With split activations one MMA covers the hi and
  // the lo rows of the stage (N = 2 * 32 * nchunk <= 256): the hi products land
  // in columns [0, HN), the lo products in [HN, 2 HN), and the epilogue adds
  // the two halves.
  constexpr uint32_t AW = SPLIT ? 256 : 128;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_launch_dependents();
  pdl_wait();  // the bucket, the gathered rows and h come from earlier kernels

  const int m0 = blockIdx.x * BM;
  const int tile_row0 = blockIdx.y * BN;
  const int mpad = p.basep[p.E];
  if (tile_row0 >= mpad) return;  // ghost tile past the last bucket's padded end
  // expert owning this tile: basep[e] <= tile_row0 < basep[e+1]
  int lo = 0, hi = p.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.basep[mid] <= tile_row0) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int live = min(BN, p.counts[e] - (tile_row0 - p.basep[e]));
  if (live <= 0) return;
  const int n_mma = (live + 15) & ~15;
  const int nchunk = (live + 31) >> 5;
  const int hn = 32 * nchunk;  // split: first TMEM column of the lo products
  const int nk = p.C / BK;
  const int nbc = p.C / 32;
  const int rows_here = min(BM, p.R - m0);
  const bool seeded = (p.bias[0] != nullptr) || (NMAT == 2 && p.bias[1] != nullptr);

  const Layout L = make_layout(NMAT, p.C);
  const int RS = L.rs;
  const uint32_t b_stage = (uint32_t)(NB * nchunk * kBChunk);
  const int NBS = min(MAX_BS, (int)(kBPool / b_stage));
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t sA = sbase + L.a, sB = sbase + L.b, sRaw = sbase + L.raw;
  const uint8_t* scs = smem + L.sc;
  // the tile's scale rows in shared memory: separate planes one matrix after the
  // other; interleaved gate/up rows alternating
  const int sc_rs = p.wrs == 2 ? 2 * nbc : nbc;
  const int sc_ms = p.wrs == 2 ? nbc : (int)L.sc_stride;
  const uint32_t bars = sbase + L.bars;
  int* s_rows = reinterpret_cast<int*>(smem + L.misc);
  float* s_w = reinterpret_cast<float*>(smem + L.misc + BN * 4);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L.misc + BN * 8);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L.misc + BN * 8 + 4);
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < RS; ++i) {
      tc::mbar_init(bar(kRawFull + i), 1);
      tc::mbar_init(bar(kRawEmpty + i), kDqWarps);
    }
    for (int i = 0; i < OSA; ++i) {
      tc::mbar_init(bar(kAFull + i), kDqWarps);
      tc::mbar_init(bar(kAEmpty + i), 1);
    }
    for (int i = 0; i < NBS; ++i) {
      tc::mbar_init(bar(kBFull + i), 1);
      tc::mbar_init(bar(kBEmpty + i), 1);
    }
    tc::mbar_init(bar(kAccFull), 1);
    tc::mbar_init(bar(kScFull), 1);
    tc::mbar_init(bar(kBiasReady), kDqWarps);
    tc::mbar_init(bar(kTFree), 2 * kDqWarps + 1);
    *s_abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == kDqWarp0) tc::tmem_alloc(tc::smem_u32(s_tmem), NMAT * AW);
  if (EPI == MOE_EPI_SCATTER_WEIGHTED_ID) {
    for (int i = threadIdx.x; i < BN; i += kThreads) {
      const int a = (i < live) ? p.rows[tile_row0 + i] : -1;
      s_rows[i] = a;
      s_w[i] = (a >= 0) ? p.weights[a] : 0.f;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;

  auto fail = [&]() {
    *s_abort = 1;
    report_timeout(p.status, 3, warp < kDqWarp0 ? warp : 3, 0, blockIdx.y);
  };

  if (warp == 0) {
    // ------------------------------------------------ raw MXFP4 producer
    if (lane == 0) {
      tc::prefetch_tmap(&tm_w0);
      if (NMAT == 2) tc::prefetch_tmap(&tm_w1);
      const uint32_t sc_bytes = (uint32_t)(rows_here * nbc);
      tc::mbar_expect_tx(bar(kScFull), NMAT * sc_bytes);
      if (p.wrs == 2) {  // interleaved gate/up: both matrices' scale rows are one run
        tc::bulk_load(sbase + L.sc, p.w_sc[0] + ((size_t)e * p.R + m0) * 2 * nbc, 2 * sc_bytes, bar(kScFull));
      } else {
        for (int mat = 0; mat < NMAT; ++mat)
          tc::bulk_load(sbase + L.sc + mat * L.sc_stride,
                        p.w_sc[mat] + ((size_t)e * p.R + m0) * nbc, sc_bytes, bar(kScFull));
      }
      const uint32_t raw_bytes = (uint32_t)(NMAT * p.box_rows * (BK / 2));
      int issued = 0;
      for (int ks = 0; ks < nk; ++ks) {
        const int rs = ks % RS, rn = ks / RS;
        if (rn > 0 && !tc::mbar_wait(bar(kRawEmpty + rs), (rn - 1) & 1, s_abort)) { fail(); break; }
        tc::mbar_expect_tx(bar(kRawFull + rs), raw_bytes);
        tc::tma_load_3d(sRaw + (rs * NMAT + 0) * kRawTile, &tm_w0, ks * (BK / 2), m0, e,
                        bar(kRawFull + rs));
        if (NMAT == 2)
          tc::tma_load_3d(sRaw + (rs * NMAT + 1) * kRawTile, &tm_w1, ks * (BK / 2), m0, e,
                          bar(kRawFull + rs));
        issued = ks + 1;
      }
      if (*s_abort) {  // let every copy already issued land before shared memory goes away
        for (int s = 0; s < RS; ++s) {
          const int n = (issued > s) ? (issued - 1 - s) / RS + 1 : 0;
          if (n > 0) tc::mbar_wait(bar(kRawFull + s), (n - 1) & 1, nullptr);
        }
        tc::mbar_wait(bar(kScFull), 0, nullptr);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------ activation producer
    if (lane == 0) {
      tc::prefetch_tmap(&tm_a);
      if (SPLIT) tc::prefetch_tmap(&tm_alo);
      int issued = 0;
      for (int ks = 0; ks < nk; ++ks) {
        const int bs = ks % NBS, bn = ks / NBS;
        if (bn > 0 && !tc::mbar_wait(bar(kBEmpty + bs), (bn - 1) & 1, s_abort)) { fail(); break; }
        tc::mbar_expect_tx(bar(kBFull + bs), b_stage);
        const uint32_t dst = sB + bs * b_stage;
        for (int c = 0; c < nchunk; ++c) {
          tc::tma_load_2d(dst + c * kBChunk, &tm_a, ks * BK, tile_row0 + 32 * c, bar(kBFull + bs));
          if (SPLIT)
            tc::tma_load_2d(dst + (nchunk + c) * kBChunk, &tm_alo, ks * BK, tile_row0 + 32 * c,
                            bar(kBFull + bs));
        }
        issued = ks + 1;
      }
      if (*s_abort) {
        for (int s = 0; s < NBS; ++s) {
          const int n = (issued > s) ? (issued - 1 - s) / NBS + 1 : 0;
          if (n > 0) tc::mbar_wait(bar(kBFull + s), (n - 1) & 1, nullptr);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(BM, SPLIT ? 2 * hn : n_mma);
      bool ok = true;
      if (seeded && !tc::mbar_wait(bar(kBiasReady), 0, s_abort)) { fail(); ok = false; }
      tc::fence_after_sync();
      for (int ks = 0; ok && ks < nk; ++ks) {
        const int as = ks % OSA, an = ks / OSA;
        const int bs = ks % NBS, bn = ks / NBS;
        if (!tc::mbar_wait2(bar(kAFull + as), an & 1, bar(kBFull + bs), bn & 1, s_abort)) {
          fail();
          break;
        }
        tc::fence_after_sync();
        // Descriptors once per k-step; a K slice of 16 bf16 is 32 bytes further,
        // i.e. +2 in the 16-byte start-address field (tiles stay below 256 KB).
        const uint64_t a_desc = tc::sw128_kmajor_desc(sA + as * NMAT * kATile);
        // B rows: the live chunks, then (split) their lo parts right behind them
        const uint64_t b_desc = tc::sw128_kmajor_desc(sB + bs * b_stage);
#pragma unroll
        for (int mat = 0; mat < NMAT; ++mat) {
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = a_desc + (uint64_t)((mat * kATile + kk * 32) >> 4);
            const uint64_t bd = b_desc + (uint64_t)(kk * 2);
            tc::mma_bf16(tmem + mat * AW, ad, bd, idesc, (ks > 0 || kk > 0 || seeded) ? 1u : 0u);
          }
        }
        tc::mma_commit(bar(kAEmpty + as));
        tc::mma_commit(bar(kBEmpty + bs));
      }
      // completes once every MMA issued above has finished
      tc::mma_commit(bar(kAccFull));
      tc::mma_commit(bar(kTFree));  // on every path, once the MMAs issued have finished
    }
  } else {
    // ------------------------------------------------ dequant + epilogue
    const int group = (warp - kDqWarp0) >> 3;
    const int dt = threadIdx.x - kDqWarp0 * 32 - kDqThreads * group;  // 0..255 within the group
    const int q = warp & 3;                      // TMEM lane quarter this warp may access
    const int colhalf = ((warp - kDqWarp0) >> 2) & 1;  // bias seeding (group 0)
    const int colquarter = (warp - kDqWarp0) >> 2;      // epilogue: 0..3
    const int trow = 32 * q + lane;              // TMEM lane = weight row within the tile
    const int f = m0 + trow;
    if (seeded && group == 0) {
      for (int mat = 0; mat < NMAT; ++mat) {
        const float bv = (p.bias[mat] != nullptr && f < p.R) ? p.bias[mat][((size_t)e * p.R + f) * p.wrs] : 0.f;
        const int ncols = SPLIT ? 2 * hn : n_mma;
        for (int c = colhalf; c < ncols / 16; c += 2)
          tc::tmem_st16(tmem + ((uint32_t)(32 * q) << 16) + mat * AW + 16 * c,
                        __float_as_uint(16 * c < (SPLIT ? hn : ncols) ? bv : 0.f));
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bar(kBiasReady));
    }
    const int r = dt >> 1, kb = dt & 1;
    const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(bar(kScFull), 0, s_abort));
    if (!ok && lane == 0) fail();
    for (int ks = group; ok && ks < nk; ks += kDqGroups) {
      const int rs = ks % RS, rn = ks / RS;
      const int as = ks % OSA, an = ks / OSA;
      // every lane waits (each then sees the stage's data); the warp leaves
      // together if any lane's wait gave up, so the __syncwarp below stays uniform
      const bool w_ok = tc::mbar_wait(bar(kRawFull + rs), rn & 1, s_abort) &&
                        (an == 0 || tc::mbar_wait(bar(kAEmpty + as), (an - 1) & 1, s_abort));
      if (!__all_sync(0xffffffffu, w_ok)) {
        if (lane == 0) fail();
        break;
      }
#pragma unroll
      for (int mat = 0; mat < NMAT; ++mat) {
        const uint4 qv = *reinterpret_cast<const uint4*>(smem + L.raw + (rs * NMAT + mat) * kRawTile +
                                                         r * (BK / 2) + kb * 16);
        const float scale = e8m0_to_f32(scs[mat * sc_ms + r * sc_rs + 2 * ks + kb]);
        uint32_t o[16];
        dequant_block_bf16(qv, scale, o);
        uint8_t* arow = smem + L.a + (as * NMAT + mat) * kATile + r * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int chunk = kb * 4 + c;
          *reinterpret_cast<uint4*>(arow + ((chunk ^ (r & 7)) << 4)) =
              make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
        }
      }
      // every thread's stores become visible to the tensor core's async proxy,
      // then one lane per warp hands the stage on
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(bar(kRawEmpty + rs));
        tc::mbar_arrive(bar(kAFull + as));
      }
    }
    // epilogue: TMEM -> registers -> global (warp-uniform decision: tcgen05.ld is warp-wide)
    __syncwarp();
    bool go = tc::mbar_wait(bar(kAccFull), 0, nullptr);
    go = __all_sync(0xffffffffu, go && (*s_abort == 0));
    if (go) {
      tc::fence_after_sync();
      const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16);
      for (int c = colquarter; c < n_mma / 16; c += 4) {
        uint32_t v0[16], v1[16];
        if (NMAT == 2) {
          tc::tmem_ld16x2_wait(tbase + 16 * c, tbase + AW + 16 * c, v0, v1);
          if (SPLIT) {  // add the lo products
            uint32_t l0[16], l1[16];
            tc::tmem_ld16x2_wait(tbase + hn + 16 * c, tbase + AW + hn + 16 * c, l0, l1);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              v0[i] = __float_as_uint(__uint_as_float(v0[i]) + __uint_as_float(l0[i]));
              v1[i] = __float_as_uint(__uint_as_float(v1[i]) + __uint_as_float(l1[i]));
            }
          }
        } else {
          tc::tmem_ld16_wait(tbase + 16 * c, v0);
          if (SPLIT) {  // add the lo products
            uint32_t l0[16];
            tc::tmem_ld16_wait(tbase + hn + 16 * c, l0);
#pragma unroll
            for (int i = 0; i < 16; ++i) v0[i] = __float_as_uint(__uint_as_float(v0[i]) + __uint_as_float(l0[i]));
          }
        }
        if (f < p.R) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int n = 16 * c + i;
            if (n < live) {
              const float g = __uint_as_float(v0[i]);
              if (EPI == MOE_EPI_SCATTER_WEIGHTED_ID) {
                const int a = s_rows[n];
                if (MOE_IN_BOUNDS(p.status, a >= 0 && (p.out_rows == 0 || a / p.k < p.out_rows))) {
                  float* dst = static_cast<float*>(p.out) + (size_t)(a / p.k) * p.out_ld + f;
                  atomicAdd(dst, s_w[n] * g);
                }
              } else {
                float v = g;
                if (EPI == MOE_EPI_SWIGLU_BF16_ID) v = swiglu_oai_f(g, __uint_as_float(v1[i]), p.alpha, p.limit);
                if (MOE_IN_BOUNDS(p.status, p.out_rows == 0 || tile_row0 + n < p.out_rows))
                  static_cast<__nv_bfloat16*>(p.out)[(size_t)(tile_row0 + n) * p.out_ld + f] =
                      __float2bfloat16_rn(v);
              }
            }
          }
        }
      }
    }
  }

  // Tensor memory goes back once every epilogue warp and the MMA thread have
  // arrived on an mbarrier, freed by warp kDqWarp0, whose code is warp-uniform
  // throughout. (No CTA-wide barrier: it would also count warps whose lane 0 is
  // still in its role loop.) Shared memory lives until every thread has exited;
  // the producers wait for their copies in flight before they leave on an abort.
  if (warp >= kDqWarp0) {
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(bar(kTFree));
    if (warp == kDqWarp0) {
      tc::mbar_wait_sleep(bar(kTFree), 0, nullptr, 64);
      tc::fence_after_sync();
      tc::tmem_dealloc(tmem, NMAT * AW);
    }
  }
}

}  // namespace mm

// ---------------------------------------------------------------------------
// host side: tensor maps and launch
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool encode_tiled_map(CUtensorMap* tm, CUtensorMapDataType dtype, int rank, const void* base,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      CUtensorMapSwizzle swizzle) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  return enc(tm, dtype, (cuuint32_t)rank, const_cast<void*>(base), d, s, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool make_weight_map(CUtensorMap* tm, const uint8_t* qs, int E, int R, int C, int box_rows, int wrs) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)(C / 2), (cuuint64_t)R, (cuuint64_t)E};
  cuuint64_t strides[2] = {(cuuint64_t)wrs * (C / 2), (cuuint64_t)wrs * R * (C / 2)};
  cuuint32_t box[3] = {(cuuint32_t)(mm::BK / 2), (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(qs), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool make_act_map(CUtensorMap* tm, const uint16_t* a, int rows, int C) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)C * 2};
  cuuint32_t box[2] = {(cuuint32_t)mm::BK, 32};
  cuuint32_t es[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(a), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NMAT, int EPI, bool SPLIT>
static cudaError_t launch_mm(const GroupedMMArgs& g, const CUtensorMap& t0, const CUtensorMap& t1,
                             const CUtensorMap& ta, const CUtensorMap& talo, const mm::Params& prm,
                             Launch L) {
  const mm::Layout lay = mm::make_layout(NMAT, g.C);
  if (lay.rs < 2 || lay.total > mm::kSmemLimit) return cudaErrorInvalidValue;
  cudaError_t err = ensure_smem_limit(mm::grouped_mm_kernel<NMAT, EPI, SPLIT>, lay.total);
  if (err != cudaSuccess) return err;
  dim3 grid((g.R + mm::BM - 1) / mm::BM, g.max_rows / mm::BN);
  return launch_kernel(mm::grouped_mm_kernel<NMAT, EPI, SPLIT>, grid, dim3(mm::kThreads), lay.total,
                       L, t0, t1, ta, talo, prm);
}

template <int NMAT, int EPI>
static cudaError_t launch_mm_split(const GroupedMMArgs& g, const CUtensorMap& t0,
                                   const CUtensorMap& t1, const CUtensorMap& ta,
                                   const CUtensorMap& talo, const mm::Params& prm, Launch L) {
  if (g.a_lo) return launch_mm<NMAT, EPI, true>(g, t0, t1, ta, talo, prm, L);
  return launch_mm<NMAT, EPI, false>(g, t0, t1, ta, talo, prm, L);
}

cudaError_t launch_grouped_mm(const GroupedMMArgs& g, Launch L) {
  if (g.max_rows <= 0) return cudaSuccess;
  if (g.C % mm::BK != 0 || g.C > 4096 || g.R % 8 != 0 || g.max_rows % mm::BN != 0)
    return cudaErrorInvalidValue;
  const int box_rows = g.R < mm::BM ? g.R : mm::BM;
  CUtensorMap t0, t1, ta;
  const int wrs = g.rs == 2 && g.nmat == 2 ? 2 : 1;
  if (!make_weight_map(&t0, g.w_qs[0], g.E, g.R, g.C, box_rows, wrs)) return cudaErrorInvalidValue;
  if (g.nmat == 2) {
    if (!make_weight_map(&t1, g.w_qs[1], g.E, g.R, g.C, box_rows, wrs)) return cudaErrorInvalidValue;
  } else {
    t1 = t0;
  }
  if (!make_act_map(&ta, g.a, g.max_rows, g.C)) return cudaErrorInvalidValue;
  CUtensorMap talo = ta;
  if (g.a_lo && !make_act_map(&talo, g.a_lo, g.max_rows, g.C)) return cudaErrorInvalidValue;
  mm::Params prm;
  prm.w_sc[0] = g.w_sc[0];
  prm.w_sc[1] = g.nmat == 2 ? g.w_sc[1] : g.w_sc[0];
  prm.bias[0] = g.bias[0];
  prm.bias[1] = g.nmat == 2 ? g.bias[1] : nullptr;
  prm.wrs = wrs;
  prm.E = g.E;
  prm.R = g.R;
  prm.C = g.C;
  prm.counts = g.counts;
  prm.basep = g.basep;
  prm.rows = g.rows;
  prm.k = g.k;
  prm.weights = g.weights;
  prm.alpha = g.alpha;
  prm.limit = g.limit;
  prm.out = g.out;
  prm.out_ld = g.out_ld;
  prm.out_rows = g.out_rows;
  prm.status = g.status;
  prm.box_rows = box_rows;
  if (g.nmat == 2) {
    if (g.epilogue != MOE_EPI_SWIGLU_BF16_ID) return cudaErrorInvalidValue;
    return launch_mm_split<2, MOE_EPI_SWIGLU_BF16_ID>(g, t0, t1, ta, talo, prm, L);
  }
  if (g.epilogue == MOE_EPI_STORE_BF16_ID)
    return launch_mm_split<1, MOE_EPI_STORE_BF16_ID>(g, t0, t1, ta, talo, prm, L);
  if (g.epilogue == MOE_EPI_SCATTER_WEIGHTED_ID)
    return launch_mm_split<1, MOE_EPI_SCATTER_WEIGHTED_ID>(g, t0, t1, ta, talo, prm, L);
  return cudaErrorInvalidValue;
}

}  // namespace moe
