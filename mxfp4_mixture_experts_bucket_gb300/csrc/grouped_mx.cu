// Prefill rail on the block-scaled tensor cores: MXFP4 weights go into
// tcgen05.mma kind::mxf8f6f4 as they are stored (E2M1 codes, one E8M0 scale
// per 32 reduction columns), so no weight is ever dequantised.
//
// Method: the routed expert chain of the Metal fusion lane ("dasLLAMA gpt-oss
// arc", fusion commit: bias seeds the accumulator, swiglu_oai in the gate/up
// epilogue, router-weighted scatter in the down epilogue, ghost rows exit),
// with the MXFP4 format of "gpt-oss: mx4 kernels to the lab-winning shape"
// (block of 32 E2M1 codes + one E8M0 exponent). On GB300 the tensor core takes
// that format natively; only the activation side changes: each activation
// block of 32 values is carried as a sum of E4M3 blocks ("terms"), each on its
// own E8M0 scale, every term taking the rounding residual of the ones before
// (about 4 more significant bits per term). x enters gate/up as three terms:
// with E8M0 scales up to 2^8 the gate/up pre-activations reach 10^3..10^4
// while swiglu_oai resolves features of size ~1 (the clamp at 7), so their
// absolute error must stay well below 1. h enters down as two terms (it is
// bounded by the clamp: |h| <= 56).
//
// Operand layouts (checked on the hardware against brute force):
//   A (weights), K-major, 128-byte swizzle, 128 K per 128-byte row: each
//     16-byte chunk holds 16 E2M1 codes packed in its first 8 bytes (code 2j in
//     the low nibble of byte j), the other 8 bytes are ignored. The stored
//     block of 16 bytes (byte i: column i low, column 16+i high) therefore
//     becomes two chunks without moving a nibble, and MMA position p of a
//     32-block reads stored column 8(p/16) + (p%16)/2 + 16(p%2).
//   B (activations), K-major, 128-byte swizzle, one E4M3 byte per K, in the
//     same per-block order: stored column c of a block sits at position
//     2(c%16) + c/16.
//   Scales in tensor memory: A row m at lane m, column base + m/32; B row n
//     at column base + n/32 and, for the output rows of each lane quarter, in
//     that quarter's lane 32q + n%32 (the B words are present four times);
//     byte i of the 32-bit cell belongs to the i-th K block of the stage,
//     chosen per MMA by the scale-factor id.
//
// CTA = 128 weight rows x one 128-row bucket tile (swap-AB: weight rows are
// M, bucket rows N <= 128). The activation terms are stacked along N (term t
// at B rows t*hn, hn = 32 * live chunks) so that one MMA can take several
// terms while reading its A slice from shared memory once; the terms land in
// separate accumulator column blocks that the epilogue adds. Warps:
//   0       TMA producer: packed nibble tiles [E][R][C/2] (64 B x 128 rows per
//           matrix per stage) into a raw ring
//   1       TMEM owner, single-thread MMA issuer
//   2       activation producer: the E4M3 term tiles (live 32-row chunks) and
//           their scale words
//   3       idle
//   4..11   two groups of four (one per TMEM lane quarter) taking alternate
//           stages: expand the nibble tiles into the padded operand layout,
//           write the stage's scales into tensor memory (the weights' scale
//           words come straight from global memory, one stage ahead); group 0
//           seeds the accumulators with the bias; all eight run the epilogue.
#include <cuda.h>

#include "mx_terms.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace mx {

constexpr int BM = 128;                  // weight rows per tile (MMA M)
constexpr int BN = 128;                  // bucket rows per tile (MMA N <= BN)
constexpr int BK = 128;                  // K per stage: four scale blocks
constexpr int OSA = 2;                   // expanded A stages (and TMEM scale slots)
constexpr int MAX_RS = 12;               // raw nibble stages
constexpr int MAX_BS = 4;                // activation stages
constexpr int kXTerms = 3;               // E4M3 terms of x (gate/up operand)
constexpr int kHTerms = 2;               // E4M3 terms of h (down operand)
constexpr int kThreads = 12 * 32;
constexpr int kGrpWarp0 = 4;             // first expansion / epilogue warp
constexpr int kGrpWarps = 4;             // warps per expansion group (one per lane quarter)
constexpr int kRawTile = BM * BK / 2;    // 8 KB packed
constexpr int kATile = BM * BK;          // 16 KB padded
constexpr int kBChunk = 32 * BK;         // 4 KB: 32 activation rows of one term
constexpr int kBScTerm = 512;            // one term's scale words for 128 rows
constexpr uint32_t kSmemLimit = 232448;

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
  const uint32_t* a_sc;  // activation scale words [NT][C/128 rounded up][max_rows]; byte i = K block i of the stage
  int max_rows;
  uint8_t* out_q;        // gate/up: h terms [kHTerms][max_rows][R]
  uint8_t* out_sc;       // gate/up: h scale words [kHTerms][R/128 rounded up][max_rows], as bytes
  float* y;              // down: [T][R]
  int* status;
  int box_rows;
  int wrs;  // weight row stride in rows: 1, or 2 for gate/up rows interleaved in one plane
};

__device__ __forceinline__ uint32_t idesc_mx(int M, int N) {
  return (5u << 7)                      // A: E2M1
         | (0u << 10)                   // B: E4M3
         | ((uint32_t)(N >> 3) << 17)   // N / 8
         | (1u << 23)                   // scales are E8M0
         | ((uint32_t)(M >> 4) << 24);  // M / 16
}

__device__ __forceinline__ void mma_mx(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%5], [%6], p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(a), "r"(b),
               "r"(c), "r"(d)
               : "memory");
}

// Shared-memory plan, identical on host and device.
struct Layout {
  uint32_t a, b, bsc, raw, bars, misc, total, b_pool;
  int rs;
};

__host__ __device__ inline Layout make_layout(int nmat, int nt) {
  Layout L;
  L.a = 0;
  L.b = OSA * nmat * kATile;
  L.b_pool = (uint32_t)(nt * 8 * kBChunk);  // two stages of four chunks
  L.bsc = L.b + L.b_pool;
  L.raw = L.bsc + MAX_BS * nt * kBScTerm;
  const uint32_t tail = 64 * 8 + (BN * 8 + 64) + 1024;
  const uint32_t budget = kSmemLimit - L.raw - tail;
  int rs = (int)(budget / (uint32_t)(nmat * kRawTile));
  L.rs = rs > MAX_RS ? MAX_RS : rs;
  L.bars = L.raw + L.rs * nmat * kRawTile;
  L.misc = L.bars + 64 * 8;
  L.total = L.misc + BN * 8 + 64 + 1024;
  return L;
}

constexpr int kRawFull = 0;
constexpr int kRawEmpty = kRawFull + MAX_RS;
constexpr int kAFull = kRawEmpty + MAX_RS;
constexpr int kAEmpty = kAFull + OSA;
constexpr int kBFull = kAEmpty + OSA;
constexpr int kBEmpty = kBFull + MAX_BS;
constexpr int kAccFull = kBEmpty + MAX_BS;
constexpr int kBiasReady = kAccFull + 1;
constexpr int kTFree = kBiasReady + 1;  // the epilogue warps and the MMA thread are done with tensor memory
constexpr int kNumBars = kTFree + 1;
static_assert(kNumBars <= 64, "barrier space");
static_assert(kXTerms == kMxXTerms && kHTerms == kMxHTerms, "workspace plan and kernels agree");

// NMAT = 2: gate/up (two accumulators, swiglu, h written as kHTerms E4M3 terms).
// NMAT = 1: down (router-weighted scatter-add into y). NT: activation terms.
template <int NMAT, int NT>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_mx_kernel(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                      const __grid_constant__ CUtensorMap tm_b, const Params p) {
  constexpr uint32_t kScCols = 4 * (NMAT + NT);        // A words per matrix, then B words per term
  constexpr uint32_t kTmemCols = 512;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_launch_dependents();
  pdl_wait();  // the bucket and the activation terms come from earlier kernels

  const int m0 = blockIdx.x * BM;
  const int tile_row0 = blockIdx.y * BN;
  const int mpad = p.basep[p.E];
  if (tile_row0 >= mpad) return;  // ghost tile past the last bucket's padded end
  int lo = 0, hi = p.E - 1;       // expert owning the tile: basep[e] <= tile_row0 < basep[e+1]
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.basep[mid] <= tile_row0) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int live = min(BN, p.counts[e] - (tile_row0 - p.basep[e]));
  if (live <= 0) return;
  const int n_mma = (live + 15) & ~15;
  const int nchunk = (live + 31) >> 5;
  const int hn = 32 * nchunk;  // rows of one term in the B tile
  // The terms' B rows are stacked (term t at rows t*hn) so that one MMA can take
  // several terms at once (N = terms * hn <= 256): the A slice is then read from
  // shared memory once for all of them. Term blocks land in separate
  // accumulator column blocks, summed by the epilogue. TMEM: NMAT accumulators
  // of acc_w columns, then the scale slots (<= 512 columns in all).
  //   mode 0: all terms in one MMA; mode 1: all but the last in one MMA, the
  //   last accumulating into block 0; mode 2: one MMA per term, all into block 0.
  int mode = 2;
  if (NT * hn <= 256 && NMAT * NT * hn + OSA * (int)kScCols <= (int)kTmemCols) mode = 0;
  else if ((NT - 1) * hn <= 256 && NMAT * (NT - 1) * hn + OSA * (int)kScCols <= (int)kTmemCols) mode = 1;
  const int acc_w = mode == 0 ? NT * hn : (mode == 1 ? (NT - 1) * hn : hn);
  const int nsum = mode == 0 ? NT : (mode == 1 ? NT - 1 : 1);  // accumulator blocks the epilogue adds
  const uint32_t sc0 = (uint32_t)(NMAT * acc_w);                // first scale slot column
  const int nbc = p.C / 32;             // scale blocks along K (even)
  const int nk = (nbc + 3) >> 2;        // stages; the last may hold only two blocks
  const int rows_here = min(BM, p.R - m0);
  const bool seeded = (p.bias[0] != nullptr) || (NMAT == 2 && p.bias[1] != nullptr);

  const Layout L = make_layout(NMAT, NT);
  const int RS = L.rs;
  const uint32_t b_term = (uint32_t)(nchunk * kBChunk);
  const uint32_t b_stage = NT * b_term;
  const int NBS = min(MAX_BS, (int)(L.b_pool / b_stage));
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t sA = sbase + L.a, sB = sbase + L.b;
  const uint32_t bars = sbase + L.bars;
  int* s_rows = reinterpret_cast<int*>(smem + L.misc);
  float* s_w = reinterpret_cast<float*>(smem + L.misc + BN * 4);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L.misc + BN * 8);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L.misc + BN * 8 + 4);
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < RS; ++i) {
      tc::mbar_init(bar(kRawFull + i), 1);
      tc::mbar_init(bar(kRawEmpty + i), kGrpWarps);
    }
    for (int i = 0; i < OSA; ++i) {
      tc::mbar_init(bar(kAFull + i), kGrpWarps);
      tc::mbar_init(bar(kAEmpty + i), 1);
    }
    for (int i = 0; i < NBS; ++i) {
      tc::mbar_init(bar(kBFull + i), 1);
      tc::mbar_init(bar(kBEmpty + i), 1);
    }
    tc::mbar_init(bar(kAccFull), 1);
    tc::mbar_init(bar(kBiasReady), kGrpWarps);
    tc::mbar_init(bar(kTFree), kThreads / 32 - kGrpWarp0 + 1);
    *s_abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == kGrpWarp0) tc::tmem_alloc(tc::smem_u32(s_tmem), kTmemCols);
  if (NMAT == 1) {
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
    report_timeout(p.status, 4, warp < kGrpWarp0 ? warp : kGrpWarp0, 0, blockIdx.y);
  };

  if (warp == 0) {
    // ------------------------------------------------ packed nibble producer
    if (lane == 0) {
      tc::prefetch_tmap(&tm_w0);
      if (NMAT == 2) tc::prefetch_tmap(&tm_w1);
      const uint32_t raw_bytes = (uint32_t)(NMAT * p.box_rows * (BK / 2));
      int issued = 0;
      for (int ks = 0; ks < nk; ++ks) {
        const int rs = ks % RS, rn = ks / RS;
        if (rn > 0 && !tc::mbar_wait(bar(kRawEmpty + rs), (rn - 1) & 1, s_abort)) { fail(); break; }
        tc::mbar_expect_tx(bar(kRawFull + rs), raw_bytes);
        const uint32_t dst = sbase + L.raw + (uint32_t)(rs * NMAT) * kRawTile;
        tc::tma_load_3d(dst, &tm_w0, ks * (BK / 2), m0, e, bar(kRawFull + rs));
        if (NMAT == 2) tc::tma_load_3d(dst + kRawTile, &tm_w1, ks * (BK / 2), m0, e, bar(kRawFull + rs));
        issued = ks + 1;
      }
      if (*s_abort) {  // every copy already issued lands before shared memory goes away
        for (int s = 0; s < RS; ++s) {
          const int n = (issued > s) ? (issued - 1 - s) / RS + 1 : 0;
          if (n > 0) tc::mbar_wait(bar(kRawFull + s), (n - 1) & 1, nullptr);
        }
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------ activation producer
    if (lane == 0) {
      tc::prefetch_tmap(&tm_b);
      const uint32_t sc_bytes = (uint32_t)(32 * nchunk * 4);
      int issued = 0;
      for (int ks = 0; ks < nk; ++ks) {
        const int bs = ks % NBS, bn = ks / NBS;
        if (bn > 0 && !tc::mbar_wait(bar(kBEmpty + bs), (bn - 1) & 1, s_abort)) { fail(); break; }
        tc::mbar_expect_tx(bar(kBFull + bs), NT * (b_term + sc_bytes));
        const uint32_t dst = sB + bs * b_stage;
        const uint32_t sdst = sbase + L.bsc + (uint32_t)(bs * NT) * kBScTerm;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          for (int c = 0; c < nchunk; ++c)
            tc::tma_load_3d(dst + t * b_term + c * kBChunk, &tm_b, ks * BK, tile_row0 + 32 * c, t, bar(kBFull + bs));
          tc::bulk_load(sdst + t * kBScTerm, p.a_sc + ((size_t)t * nk + ks) * p.max_rows + tile_row0, sc_bytes,
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
      const uint32_t id_wide = idesc_mx(BM, mode == 0 ? NT * hn : (NT - 1) * hn);
      const uint32_t id_one = idesc_mx(BM, mode == 2 ? n_mma : hn);
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
        const uint64_t a_desc = tc::sw128_kmajor_desc(sA + as * NMAT * kATile);
        const uint64_t b_desc = tc::sw128_kmajor_desc(sB + bs * b_stage);
        const uint32_t slot = tmem + sc0 + (uint32_t)as * kScCols;
        const uint32_t sfb = slot + 4 * NMAT;  // term t's words at sfb + t * nchunk
        const int nkb = min(4, nbc - 4 * ks);
#pragma unroll
        for (int mat = 0; mat < NMAT; ++mat) {
          const uint32_t d = tmem + (uint32_t)(mat * acc_w);
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
            if (kb < nkb) {
              const uint32_t sfid = ((uint32_t)kb << 4) | ((uint32_t)kb << 29);
              const uint64_t ad = a_desc + (uint64_t)((mat * kATile + kb * 32) >> 4);
              const uint32_t acc0 = (ks > 0 || kb > 0 || seeded) ? 1u : 0u;
              if (mode == 2) {
#pragma unroll
                for (int t = 0; t < NT; ++t)
                  mma_mx(d, ad, b_desc + (uint64_t)((t * b_term + kb * 32) >> 4), id_one | sfid, slot + 4 * mat,
                         sfb + t * nchunk, t > 0 ? 1u : acc0);
              } else {
                mma_mx(d, ad, b_desc + (uint64_t)((kb * 32) >> 4), id_wide | sfid, slot + 4 * mat, sfb, acc0);
                if (mode == 1)
                  mma_mx(d, ad, b_desc + (uint64_t)(((NT - 1) * b_term + kb * 32) >> 4), id_one | sfid,
                         slot + 4 * mat, sfb + (NT - 1) * nchunk, 1u);
              }
            }
          }
        }
        tc::mma_commit(bar(kAEmpty + as));
        tc::mma_commit(bar(kBEmpty + bs));
      }
      tc::mma_commit(bar(kAccFull));  // completes once every MMA issued above has finished
      tc::mma_commit(bar(kTFree));    // on every path, once the MMAs issued have finished
    }
  } else if (warp >= kGrpWarp0) {
    // ------------------------------------------------ expansion groups + epilogue
    const int g = (warp - kGrpWarp0) >> 2;  // group: stages ks = g, g + 2, ...
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int trow = 32 * q + lane;         // TMEM lane = weight row within the tile
    const int f = m0 + trow;
    const uint32_t qlane = (uint32_t)(32 * q) << 16;
    if (seeded && g == 0) {
      for (int mat = 0; mat < NMAT; ++mat) {
        const float bv = (p.bias[mat] != nullptr && f < p.R) ? p.bias[mat][((size_t)e * p.R + f) * p.wrs] : 0.f;
        for (int c = 0; c < acc_w / 16; ++c)
          tc::tmem_st16(tmem + qlane + (uint32_t)(mat * acc_w) + 16 * c, __float_as_uint(16 * c < hn ? bv : 0.f));
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bar(kBiasReady));
    }
    // The weight row's E8M0 bytes of a stage (4 blocks; the last stage may hold
    // 2), read from global memory one stage of this group ahead of their use as
    // two 16-bit halves that are only combined at the use, so that no wait for
    // the load lands before the stage's barrier waits.
    const uint16_t* scrow[NMAT];
#pragma unroll
    for (int mat = 0; mat < NMAT; ++mat)
      scrow[mat] = reinterpret_cast<const uint16_t*>(p.w_sc[mat] + ((size_t)e * p.R + m0 + trow) * p.wrs * nbc);
    const bool sc_row = trow < rows_here;
    uint16_t sc_lo16[NMAT], sc_hi16[NMAT];
    auto sc_fetch = [&](int ks) {
#pragma unroll
      for (int mat = 0; mat < NMAT; ++mat) {
        sc_lo16[mat] = (sc_row && ks < nk) ? __ldg(scrow[mat] + 2 * ks) : (uint16_t)0x7F7F;
        sc_hi16[mat] = (sc_row && 4 * ks + 2 < nbc) ? __ldg(scrow[mat] + 2 * ks + 1) : (uint16_t)0x7F7F;
      }
    };
    sc_fetch(g);
    const int xr0 = trow >> 3, xc = trow & 7;  // expansion: chunk xc of rows xr0 + 16 i
    for (int ks = g; ks < nk; ks += 2) {
      const int rs = ks % RS, rn = ks / RS;
      const int as = ks % OSA, an = ks / OSA;
      const int bs = ks % NBS, bn = ks / NBS;
      uint16_t cur_lo[NMAT], cur_hi[NMAT];
#pragma unroll
      for (int mat = 0; mat < NMAT; ++mat) {
        cur_lo[mat] = sc_lo16[mat];
        cur_hi[mat] = sc_hi16[mat];
      }
      sc_fetch(ks + 2);
      // every lane waits (each then sees the data); the warp leaves together if any gave up
      const bool w_ok = tc::mbar_wait(bar(kRawFull + rs), rn & 1, s_abort) &&
                        (an == 0 || tc::mbar_wait(bar(kAEmpty + as), (an - 1) & 1, s_abort)) &&
                        tc::mbar_wait(bar(kBFull + bs), bn & 1, s_abort);
      if (!__all_sync(0xffffffffu, w_ok)) {
        if (lane == 0) fail();
        break;
      }
      tc::fence_after_sync();  // the slot's previous MMAs are complete
#pragma unroll
      for (int mat = 0; mat < NMAT; ++mat) {
        const uint8_t* raw = smem + L.raw + (rs * NMAT + mat) * kRawTile;
        uint8_t* at = smem + L.a + (as * NMAT + mat) * kATile;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = xr0 + 16 * i;
          // the MMA ignores the chunk's second 8 bytes: only the nibbles are written
          *reinterpret_cast<uint2*>(at + r * 128 + ((xc ^ (r & 7)) << 4)) =
              *reinterpret_cast<const uint2*>(raw + r * (BK / 2) + xc * 8);
        }
      }
      const uint32_t slot = tmem + sc0 + (uint32_t)as * kScCols;
#pragma unroll
      for (int mat = 0; mat < NMAT; ++mat)  // A row m: lane m, column m / 32
        tmem_st1(slot + qlane + 4 * mat + q, (uint32_t)cur_lo[mat] | ((uint32_t)cur_hi[mat] << 16));
      {  // stacked B row t*hn + n, for the output rows of lane quarter q: lane 32 q + n % 32,
         // column t * nchunk + n / 32
        const uint32_t* bw = reinterpret_cast<const uint32_t*>(smem + L.bsc + (uint32_t)(bs * NT) * kBScTerm);
#pragma unroll
        for (int t = 0; t < NT; ++t)
          for (int j = 0; j < nchunk; ++j)
            tmem_st1(slot + qlane + 4 * NMAT + t * nchunk + j, bw[128 * t + 32 * j + lane]);
      }
      tc::tmem_wait_st();
      tc::fence_proxy_async_smem();  // the expanded tile becomes visible to the tensor core
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(bar(kRawEmpty + rs));
        tc::mbar_arrive(bar(kAFull + as));
      }
    }
    // epilogue: TMEM -> registers -> global (warp-uniform: tcgen05.ld is warp-wide)
    __syncwarp();
    bool go = tc::mbar_wait(bar(kAccFull), 0, nullptr);
    go = __all_sync(0xffffffffu, go && (*s_abort == 0));
    if (go) {
      tc::fence_after_sync();
      const uint32_t tbase = tmem + qlane;
      for (int c = g; c < n_mma / 16; c += 2) {
        if (NMAT == 2) {
          uint32_t v0[16], v1[16];
          tc::tmem_ld16x2_wait(tbase + 16 * c, tbase + (uint32_t)acc_w + 16 * c, v0, v1);
          for (int b = 1; b < nsum; ++b) {
            uint32_t w0[16], w1[16];
            tc::tmem_ld16x2_wait(tbase + (uint32_t)(b * hn) + 16 * c, tbase + (uint32_t)(acc_w + b * hn) + 16 * c, w0, w1);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              v0[i] = __float_as_uint(__uint_as_float(v0[i]) + __uint_as_float(w0[i]));
              v1[i] = __float_as_uint(__uint_as_float(v1[i]) + __uint_as_float(w1[i]));
            }
          }
          const bool blk = (m0 + 32 * q) < p.R;  // whole 32-row blocks: R % 32 == 0
          const int col = m0 + 32 * q + mx_pos(lane);
          const size_t hterm = (size_t)p.max_rows * p.R;
          const int nks_r = (p.R / 32 + 3) / 4;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int n = 16 * c + i;
            const float h = swiglu_oai_f(__uint_as_float(v0[i]), __uint_as_float(v1[i]), p.alpha, p.limit);
            uint32_t hq[kHTerms], hs[kHTerms];
            split_terms<kHTerms>(h, hq, hs);
            if (blk && n < live) {
              const size_t row = (size_t)(tile_row0 + n);
#pragma unroll
              for (int t = 0; t < kHTerms; ++t) {
                p.out_q[t * hterm + row * p.R + col] = (uint8_t)hq[t];
                if (lane == 0)
                  p.out_sc[(((size_t)t * nks_r + m0 / BM) * p.max_rows + row) * 4 + q] = (uint8_t)hs[t];
              }
            }
          }
        } else {
          uint32_t v0[16];
          tc::tmem_ld16_wait(tbase + 16 * c, v0);
          for (int b = 1; b < nsum; ++b) {
            uint32_t w0[16];
            tc::tmem_ld16_wait(tbase + (uint32_t)(b * hn) + 16 * c, w0);
#pragma unroll
            for (int i = 0; i < 16; ++i) v0[i] = __float_as_uint(__uint_as_float(v0[i]) + __uint_as_float(w0[i]));
          }
          if (f < p.R) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int n = 16 * c + i;
              if (n < live) {
                const int a = s_rows[n];
                atomicAdd(p.y + (size_t)(a / p.k) * p.R + f, s_w[n] * __uint_as_float(v0[i]));
              }
            }
          }
        }
      }
    }
  }

  // Tensor memory goes back once every epilogue warp and the MMA thread have
  // arrived on an mbarrier, freed by warp kGrpWarp0, whose code is warp-uniform
  // throughout. (No CTA-wide barrier: it would also count warps whose lane 0 is
  // still in its role loop.) Shared memory lives until every thread has exited;
  // the producers wait for their copies in flight before they leave on an abort.
  if (warp >= kGrpWarp0) {
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(bar(kTFree));
    if (warp == kGrpWarp0) {
      tc::mbar_wait_sleep(bar(kTFree), 0, nullptr, 64);
      tc::fence_after_sync();
      tc::tmem_dealloc(tmem, kTmemCols);
    }
  }
}

// Bucket rows of x as kXTerms E4M3 terms in the MMA's K order, [kXTerms][max_rows][D],
// plus their scale words [kXTerms][D/128 rounded up][max_rows]; one warp per
// (bucket row, stage of 4 blocks). Pad rows are skipped: their MMA columns are
// never stored. Also zeroes y for the scatter-add of the down projection.
__global__ void __launch_bounds__(256) quant_rows_mx_kernel(const float* __restrict__ x, int T, int D, int k,
                                                            const int32_t* __restrict__ rows,
                                                            const int32_t* __restrict__ basep, int E, int max_rows,
                                                            uint8_t* __restrict__ q_terms,
                                                            uint32_t* __restrict__ sc_terms,
                                                            float* __restrict__ y_zero) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * 8;
  const int mpad = basep[E];
  const int nbc = D / 32, nks = (nbc + 3) / 4;
  const int pos = mx_pos(lane);
  const size_t qterm = (size_t)max_rows * D;
  const int ntask = mpad * nks;
  for (int task = blockIdx.x * 8 + (threadIdx.x >> 5); task < ntask; task += nwarps) {
    const int row = task / nks, ks = task - row * nks;
    const int a = rows[row];
    if (a < 0) continue;
    const float* src = x + (size_t)(a / k) * D + 128 * ks + lane;
    const int nb = min(4, nbc - 4 * ks);
    float v[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) v[b] = (b < nb) ? __ldg(src + 32 * b) : 0.f;  // all four loads in flight
    uint32_t w[kXTerms];
#pragma unroll
    for (int t = 0; t < kXTerms; ++t) w[t] = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int blk = 4 * ks + b;
      if (b < nb) {  // warp-uniform
        uint32_t qv[kXTerms], sv[kXTerms];
        split_terms<kXTerms>(v[b], qv, sv);
#pragma unroll
        for (int t = 0; t < kXTerms; ++t) {
          q_terms[t * qterm + (size_t)row * D + 32 * blk + pos] = (uint8_t)qv[t];
          w[t] |= sv[t] << (8 * b);
        }
      } else {
#pragma unroll
        for (int t = 0; t < kXTerms; ++t) w[t] |= 0x7Fu << (8 * b);
      }
    }
    if (lane < kXTerms) {
      uint32_t wv = w[0];
#pragma unroll
      for (int t = 1; t < kXTerms; ++t) wv = (lane == t) ? w[t] : wv;
      sc_terms[((size_t)lane * nks + ks) * max_rows + row] = wv;
    }
  }
  if (y_zero) {
    float4* y4 = reinterpret_cast<float4*>(y_zero);
    const size_t ny = (size_t)T * D / 4;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < ny; i += (size_t)gridDim.x * blockDim.x)
      y4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

}  // namespace mx

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
cudaError_t launch_quant_rows_mx(const float* x, int T, int D, int k, const int32_t* rows, const int32_t* basep,
                                 int E, int max_rows, uint8_t* q_terms, uint32_t* sc_terms, float* y_zero,
                                 Launch L) {
  const int nks = (D / 32 + 3) / 4;
  const long long tasks = (long long)max_rows * nks;
  int blocks = (int)((tasks + 7) / 8);
  const int cap = device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_kernel(mx::quant_rows_mx_kernel, dim3(blocks), dim3(256), 0, L, x, T, D, k, rows, basep, E,
                       max_rows, q_terms, sc_terms, y_zero);
}

template <int NMAT, int NT>
static cudaError_t launch_mx(const GroupedMXArgs& g, const CUtensorMap& t0, const CUtensorMap& t1,
                             const CUtensorMap& tb, const mx::Params& prm, Launch L) {
  const mx::Layout lay = mx::make_layout(NMAT, NT);
  if (lay.rs < 2 || lay.total > mx::kSmemLimit) return cudaErrorInvalidValue;
  cudaError_t err = ensure_smem_limit(mx::grouped_mx_kernel<NMAT, NT>, lay.total);
  if (err != cudaSuccess) return err;
  dim3 grid((g.R + mx::BM - 1) / mx::BM, g.max_rows / mx::BN);
  return launch_kernel(mx::grouped_mx_kernel<NMAT, NT>, grid, dim3(mx::kThreads), lay.total, L, t0, t1, tb, prm);
}

cudaError_t launch_grouped_mx(const GroupedMXArgs& g, Launch L) {
  if (g.max_rows <= 0) return cudaSuccess;
  if (g.C % 64 != 0 || g.C > 4096 || g.R % 32 != 0 || g.max_rows % mx::BN != 0) return cudaErrorInvalidValue;
  const int nt = g.nmat == 2 ? mx::kXTerms : mx::kHTerms;
  const int box_rows = g.R < mx::BM ? g.R : mx::BM;
  CUtensorMap t0, t1, tb;
  {
    const uint64_t wrs = g.rs == 2 && g.nmat == 2 ? 2 : 1;
    const uint64_t dims[3] = {(uint64_t)(g.C / 2), (uint64_t)g.R, (uint64_t)g.E};
    const uint64_t strides[2] = {wrs * (g.C / 2), wrs * g.R * (g.C / 2)};
    const uint32_t box[3] = {(uint32_t)(mx::BK / 2), (uint32_t)box_rows, 1};
    if (!encode_tiled_map(&t0, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, g.w_qs[0], dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    if (g.nmat == 2) {
      if (!encode_tiled_map(&t1, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, g.w_qs[1], dims, strides, box,
                            CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    } else {
      t1 = t0;
    }
  }
  {
    const uint64_t dims[3] = {(uint64_t)g.C, (uint64_t)g.max_rows, (uint64_t)nt};
    const uint64_t strides[2] = {(uint64_t)g.C, (uint64_t)g.max_rows * g.C};
    const uint32_t box[3] = {(uint32_t)mx::BK, 32, 1};
    if (!encode_tiled_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, g.a_terms, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  mx::Params prm{};
  prm.w_sc[0] = g.w_sc[0];
  prm.w_sc[1] = g.nmat == 2 ? g.w_sc[1] : g.w_sc[0];
  prm.bias[0] = g.bias[0];
  prm.bias[1] = g.nmat == 2 ? g.bias[1] : nullptr;
  prm.wrs = g.rs == 2 && g.nmat == 2 ? 2 : 1;
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
  prm.a_sc = g.a_sc;
  prm.max_rows = g.max_rows;
  prm.out_q = g.h_terms;
  prm.out_sc = reinterpret_cast<uint8_t*>(g.h_sc);
  prm.y = g.y;
  prm.status = g.status;
  prm.box_rows = box_rows;
  if (g.nmat == 2) return launch_mx<2, mx::kXTerms>(g, t0, t1, tb, prm, L);
  return launch_mx<1, mx::kHTerms>(g, t0, t1, tb, prm, L);
}

}  // namespace moe
