// Prefill grouped GEMMs on prepacked MXFP4 weights and the block-scaled tensor
// cores, tcgen05.mma kind::mxf4 (both operands E2M1 with E8M0 block scales):
// the bias-seeded MXFP4 gate/up and down grouped GEMMs of "dasLLAMA gpt-oss
// arc" (Metal fusion lane commit: MetalMoeMulMmMx4 over the MoeBucket CSR,
// swiglu rows past each bucket's live end skipped; the fused MoE expert chain
// commit: gate+up rows, bias, activation, then down rows, bias and the
// router-weighted sum) with neither operand dequantised.
//
// Tile of one work unit: M = the 128 rows of one bucket tile (the tokens'
// activations), N = 256 weight rows (gate/up: 128 gate rows and the same 128
// up rows; down: two 128-row tiles of D), K walked in 128-column chunks. The
// activations enter as E2M1 terms (x: six, h: three; each block of 32 on its own E8M0
// scale, each term the rounded residual of the ones before), and the terms of
// a row accumulate into the same fp32 accumulator, one MMA per term and K
// half. The weights come from the prepacked planes (one bulk copy per 128-row
// tile and chunk lands the 64-byte-swizzled image the MMA reads); the
// activation chunks of a bucket tile (all terms) and their scale atoms are
// laid out the same way by quant_rows_e2m1_kernel (x) or by the gate/up
// epilogue (h).
//
// Warps: 0..5 producers (one copy of every step each; warps 0..3, one per
// tensor-memory lane quarter, also store the previous step's scale atoms into
// tensor memory with tcgen05.st and signal the MMA thread), 6 MMA issuer,
// 7..10 epilogue (one per lane quarter; warp 7 owns tensor memory). Units are
// dealt round-robin to the CTAs; every role walks the same unit sequence. The
// accumulator is freed as soon as the epilogue has read it, so the epilogue's
// arithmetic overlaps the next unit's MMAs.
//   gate/up epilogue: bias, swiglu_oai, h as three E2M1 terms per 32-block
//     (computed by each thread over its row's 32 columns), written as the down
//     GEMM's activation chunks.
//   down epilogue: y[t] += w_a * (acc + bd) for the bucket row's assignment a
//     (float atomics, as the pages' weighted scatter).
#include <cuda.h>

#include "decode_mx.cuh"
#include "mx_terms.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace gx4 {

constexpr int kProd = 6;
constexpr int kMmaWarp = 6;
constexpr int kEpiWarp0 = 7;
constexpr int kEpiWarps = 8;  // two per tensor-memory lane quarter, each taking half of the columns
constexpr int kTmemWarp = 7;
constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;
constexpr int kChunk = 8192;  // 128 rows x 64 bytes: one term's (or one weight tile's) chunk
constexpr int kAtom = 512;
constexpr uint32_t kAccCols = 256;
constexpr uint32_t kTmemCols = 512;

// Per-kernel plan: the activation operand's terms (x: kPrefillXTerms, h:
// kPrefillHTerms), the ring depth that fits 227 KB, the stage layout
// [terms][two weight tiles][term atoms][two weight atoms] and its scale columns.
template <int KIND>
struct Plan {
  static constexpr int kTerms = KIND == 0 ? kPrefillXTerms : kPrefillHTerms;
  static constexpr uint32_t kOffB = kTerms * kChunk;
  static constexpr uint32_t kOffSfa = kOffB + 2 * kChunk;
  static constexpr uint32_t kOffSfb = kOffSfa + kTerms * kAtom;
  static constexpr uint32_t kStageBytes = ((kOffSfb + 2 * kAtom) + 1023u) & ~1023u;
  static constexpr int kStages = (int)((226u * 1024u) / kStageBytes) > 6 ? 6 : (int)((226u * 1024u) / kStageBytes);
  static constexpr uint32_t kDynSmem = kStages * kStageBytes + 1024;
  static constexpr uint32_t kSfCols = 4 * kTerms + 8;  // per stage: the term atoms, then the two weight atoms
  static constexpr int kScaleBatch = kStages - 1;
};
static_assert(Plan<0>::kStages >= 3 && Plan<1>::kStages >= 3, "ring depth");
static_assert(kAccCols + Plan<0>::kStages * Plan<0>::kSfCols <= kTmemCols, "tensor memory plan");
static_assert(kAccCols + Plan<1>::kStages * Plan<1>::kSfCols <= kTmemCols, "tensor memory plan");

struct Params {
  int E, R, C, NK, NT;  // weight matrices [R][C]: NT tiles of 128 rows, NK chunks of 128 columns
  int npair;            // N tile pairs per bucket tile
  int ntiles;           // bucket tiles (max_rows / 128)
  const uint8_t* w_qs[2];
  const uint8_t* w_sf[2];
  const float* bias[2];
  const int32_t* counts;
  const int32_t* basep;
  const int32_t* rows;
  int k;
  const float* weights;
  const uint8_t* aq;   // activation chunks [ntiles][NK][terms][8192]
  const uint8_t* asf;  // [ntiles][NK][terms][512]
  uint8_t* hq;         // gate/up: down operand chunks [ntiles][NT][kPrefillHTerms][8192]
  uint8_t* hsf;        // [ntiles][NT][kPrefillHTerms][512]
  float alpha, limit;
  float* y;  // down: [T][R], accumulated into (zeroed beforehand)
  int* status;
};

__device__ __forceinline__ uint32_t idesc_mxf4(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_mxf4(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}

// Activation chunk layout (one per bucket tile and 128-column chunk, all terms
// of its rows): 16 groups of 8 rows, each group holding the terms one after
// the other, every (group, term) the 512-byte 64-byte-swizzled image of those
// 8 rows (block kb of row n at 64*(n%8) + 16*(kb ^ ((n>>1)&3))). The live rows'
// groups are then one contiguous run for every term, and a term's rows are
// `terms` x 512 bytes apart group to group (the MMA descriptor's stride).
__host__ __device__ __forceinline__ size_t act_off(int n, int t, int terms, int kb, int i) {
  return ((size_t)(n >> 3) * terms + t) * 512 + dmx::chunk_off(n & 7, kb, i);
}

// A work unit: bucket tile b (its expert e and live rows) and N tile pair t.
struct Unit {
  int b, t, e, live;
};

// The i-th unit of this CTA that is not a ghost (past the padded end of the
// last bucket); false when there is none. `cursor` walks the unit indices.
__device__ __forceinline__ bool next_unit(const Params& p, int mpad, int& cursor, Unit& u) {
  const int nunits = p.ntiles * p.npair;
  for (; cursor < nunits; cursor += gridDim.x) {
    const int b = cursor / p.npair, t = cursor - b * p.npair;
    const int row0 = 128 * b;
    if (row0 >= mpad) continue;
    int lo = 0, hi = p.E - 1;  // basep[e] <= row0 < basep[e + 1]
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(p.basep + mid) <= row0) lo = mid; else hi = mid - 1;
    }
    const int live = min(128, __ldg(p.counts + lo) - (row0 - __ldg(p.basep + lo)));
    if (live <= 0) continue;
    u.b = b;
    u.t = t;
    u.e = lo;
    u.live = live;
    cursor += gridDim.x;
    return true;
  }
  return false;
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1) grouped_mx4_kernel(const Params p) {
  using PL = Plan<KIND>;
  constexpr int kTerms = PL::kTerms, kStages = PL::kStages, kScaleBatch = PL::kScaleBatch;
  constexpr uint32_t kOffB = PL::kOffB, kOffSfa = PL::kOffSfa, kOffSfb = PL::kOffSfb;
  constexpr uint32_t kStageBytes = PL::kStageBytes, kSfCols = PL::kSfCols;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t sfr_bar[kStages];
  __shared__ __align__(8) uint64_t accf_bar, acce_bar, drain_bar, tfree_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_bias[256];  // the epilogue's unit biases (gate/up: 128 gate, 128 up; down: 256)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == 1 && lane == 0) {
    for (int i = 0; i < kStages; ++i) {
      tc::mbar_init(tc::smem_u32(&full_bar[i]), kProd);
      tc::mbar_init(tc::smem_u32(&empty_bar[i]), 1);
      tc::mbar_init(tc::smem_u32(&sfr_bar[i]), 4);
    }
    tc::mbar_init(tc::smem_u32(&accf_bar), 1);
    tc::mbar_init(tc::smem_u32(&acce_bar), kEpiWarps);
    tc::mbar_init(tc::smem_u32(&drain_bar), 1);
    tc::mbar_init(tc::smem_u32(&tfree_bar), 5 + kEpiWarps);  // 4 scale-loading producers, the MMA thread, the epilogue warps
    s_abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == kTmemWarp) tc::tmem_alloc(tc::smem_u32(&s_tmem), kTmemCols);
  pdl_wait();  // the bucket and the activation chunks come from earlier kernels
  pdl_launch_dependents();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  const int mpad = __ldg(p.basep + p.E);
  const int NK = p.NK;
  const volatile int* abort_flag = &s_abort;
  auto fail = [&](int role, int seq) {
    s_abort = 1;
    report_timeout(p.status, 7 + KIND, role, 0, seq);
  };
  const int nbc = p.C / 32;

  if (warp < kProd) {
    // ------------------------------------------------ producers: copy `warp` of every step;
    // warps 0..3 (one per tensor-memory lane quarter) also store the scale atoms of the
    // step before into tensor memory once its data has landed, and signal the MMA thread
    const bool loader = warp < 4;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
    uint64_t pol = 0;
    if (lane == 0) pol = tc::l2_policy_evict_first();
    int cursor = blockIdx.x, i = 0, issued = 0;
    Unit u;
    bool ok = true;
    // scale atoms of step s (stage s % kStages) into this warp's lane quarter
    auto load_scales = [&](int s) -> bool {
      const int st = s % kStages, n = s / kStages;
      // (sleeping between probes: these warps share their SM sub-partitions with the epilogue warps)
      const bool okw = tc::mbar_wait_sleep(tc::smem_u32(&full_bar[st]), n & 1, abort_flag, 64);
      if (!__all_sync(0xffffffffu, okw)) {
        if (lane == 0) fail(3, s);
        return false;
      }
      const uint8_t* sbp = smem + (size_t)st * kStageBytes;
      const uint32_t sfs = lane_base + kAccCols + (uint32_t)st * kSfCols;
#pragma unroll
      for (int a = 0; a < kTerms + 2; ++a) {  // activation atoms, then the two weight atoms
        const uint8_t* atom = sbp + (a < kTerms ? kOffSfa + a * kAtom : kOffSfb + (a - kTerms) * kAtom);
        const uint4 w = *reinterpret_cast<const uint4*>(atom + 16 * lane);
        tc::tmem_st4(sfs + 4 * a, w.x, w.y, w.z, w.w);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sfr_bar[st]));
      return true;
    };
    while (ok && next_unit(p, mpad, cursor, u)) {
      const int live_groups = (u.live + 7) >> 3;
      for (int j = 0; j < NK && ok; ++j, ++i) {
        const int st = i % kStages, n = i / kStages;
        if (lane == 0) {
          if (n > 0 && !tc::mbar_wait_sleep(tc::smem_u32(&empty_bar[st]), (n - 1) & 1, abort_flag, 32)) {
            fail(0, i);
            ok = false;
          }
        }
        if (loader) ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        if (lane == 0) {
          const uint32_t fb = tc::smem_u32(&full_bar[st]);
          const uint32_t sb = tc::smem_u32(smem) + (uint32_t)st * kStageBytes;
          const size_t achunk = (size_t)u.b * NK + j;
          if (warp < 2) {  // the live rows' groups of all terms, in two runs
            const int g0 = (live_groups + 1) >> 1;
            const int ga = warp == 0 ? 0 : g0, gn = warp == 0 ? g0 : live_groups - g0;
            const uint32_t bytes = (uint32_t)(gn * kTerms * 512);
            tc::mbar_expect_tx(fb, bytes);
            if (bytes)
              tc::bulk_load(sb + (uint32_t)(ga * kTerms * 512),
                            p.aq + achunk * (size_t)(kTerms * kChunk) + (size_t)ga * kTerms * 512, bytes, fb);
          } else if (warp == 4) {  // the activation atoms of all terms
            tc::mbar_expect_tx(fb, kTerms * kAtom);
            tc::bulk_load(sb + kOffSfa, p.asf + achunk * kTerms * kAtom, kTerms * kAtom, fb);
          } else if (warp < 4) {
            // weight tile h of the pair (gate/up: matrix h of tile t; down: tile 2t + h); a
            // missing tile leaves its rows stale: they only feed accumulator columns nobody reads
            const int h = warp - 2;
            const int tile = KIND == 0 ? u.t : 2 * u.t + h;
            if (tile < p.NT) {
              const int rows_t = min(128, p.R - 128 * tile);
              const uint32_t bytes = (uint32_t)(rows_t * 64);
              const uint8_t* src = p.w_qs[KIND == 0 ? h : 0] +
                                   ((size_t)u.e * p.R + 128 * (size_t)tile) * ((size_t)NK * 64) + (size_t)rows_t * 64 * j;
              tc::mbar_expect_tx(fb, bytes);
              tc::bulk_load_stream(sb + kOffB + (uint32_t)(h * kChunk), src, bytes, fb, pol);
            } else {
              tc::mbar_expect_tx(fb, 0);
            }
          } else {  // warp 5: the weight tiles' scale atoms
            uint32_t bytes = 0;
            for (int h = 0; h < 2; ++h) bytes += (KIND == 0 || 2 * u.t + h < p.NT) ? kAtom : 0u;
            tc::mbar_expect_tx(fb, bytes);
            for (int h = 0; h < 2; ++h) {
              const int tile = KIND == 0 ? u.t : 2 * u.t + h;
              if (tile >= p.NT) continue;
              tc::bulk_load_stream(sb + kOffSfb + (uint32_t)(h * kAtom),
                                   p.w_sf[KIND == 0 ? h : 0] + (((size_t)u.e * p.NT + tile) * NK + j) * kAtom, kAtom,
                                   fb, pol);
            }
          }
          issued = i + 1;
        }
        if (loader) {
          __syncwarp();
          if (i >= 1 && !load_scales(i - 1)) ok = false;
        }
      }
    }
    if (loader) {
      issued = __shfl_sync(0xffffffffu, issued, 0);
      if (ok && issued >= 1) ok = load_scales(issued - 1);  // the last step's scales
      tc::fence_before_sync();  // this warp's tensor-memory stores are complete
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tc::smem_u32(&tfree_bar));
    }
    if (lane == 0 && *abort_flag) {  // every copy already issued lands before shared memory goes away
      for (int st = 0; st < kStages; ++st) {
        const int n = issued > st ? (issued - 1 - st) / kStages + 1 : 0;
        if (n > 0) tc::mbar_wait(tc::smem_u32(&full_bar[st]), (n - 1) & 1, nullptr);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_mxf4(128, 256);
      int cursor = blockIdx.x, i = 0, lu = 0;
      Unit u;
      bool ok = true;
      while (ok && next_unit(p, mpad, cursor, u)) {
        if (lu > 0 && !tc::mbar_wait_sleep(tc::smem_u32(&acce_bar), (lu - 1) & 1, abort_flag, 32)) {
          fail(1, i);
          break;
        }
        tc::fence_after_sync();
        for (int j = 0; j < NK; ++j, ++i) {
          const int st = i % kStages, n = i / kStages;
          if (!tc::mbar_wait(tc::smem_u32(&sfr_bar[st]), n & 1, abort_flag)) {
            fail(1, i);
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t sb = tc::smem_u32(smem) + (uint32_t)st * kStageBytes;
          const uint32_t sfs = tmem + kAccCols + (uint32_t)st * kSfCols;
          const int nkb = min(4, nbc - 4 * j);  // 32-blocks in this chunk: 2 or 4 (widths are multiples of 64)
          const uint64_t bdesc = tc::sw64_kmajor_desc(sb + kOffB);
          const uint64_t adesc = tc::sw64_kmajor_desc_sbo(sb, kTerms * 512);  // term t starts t*512 further
#pragma unroll
          for (int kh = 0; kh < 2; ++kh) {
            if (2 * kh >= nkb) continue;
            const uint32_t id = idesc | (kh ? ((2u << 4) | (2u << 29)) : 0u);
#pragma unroll
            for (int term = 0; term < kTerms; ++term)
              mma_mxf4(tmem, adesc + (uint64_t)(term * (512 >> 4) + 2 * kh), bdesc + (uint64_t)(2 * kh), id,
                       sfs + 4 * term, sfs + 4 * kTerms, (j == 0 && kh == 0 && term == 0) ? 0u : 1u);
          }
          tc::mma_commit(tc::smem_u32(&empty_bar[st]));
          if (j == NK - 1) tc::mma_commit(tc::smem_u32(&accf_bar));
        }
        ++lu;
      }
      tc::mma_commit(tc::smem_u32(&drain_bar));
      tc::mbar_wait(tc::smem_u32(&drain_bar), 0, nullptr);
      tc::fence_before_sync();
      tc::mbar_arrive(tc::smem_u32(&tfree_bar));
    }
  } else {
    // ------------------------------------------------ epilogue (warps 7..14)
    const int q = warp & 3;
    const int half = (warp - kEpiWarp0) >> 2;  // which half of the unit's columns
    const int row = 32 * q + lane;  // bucket row within the tile = tensor-memory lane
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
    int cur_epi = blockIdx.x;
    Unit ue{};
    int ldone = 0;  // units whose epilogue has run
    bool have_e = next_unit(p, mpad, cur_epi, ue);
    while (have_e) {
      // ---- the epilogue of unit ldone (ue)
      const int e = ue.e;
      const int prow = 128 * ue.b + row;  // bucket row
      // the unit's biases into shared memory (the four epilogue warps; every
      // reader of the previous unit's is past the first barrier)
      tc::named_sync(1, 32 * kEpiWarps);
      {
        const int c = 32 * q + lane;  // 128 columns per pass
        for (int h2 = half; h2 < 2; h2 += 2) {
          float bv = 0.f;
          if (KIND == 0) {
            const int f = 128 * ue.t + c;
            if (p.bias[h2] && f < p.R) bv = __ldg(p.bias[h2] + (size_t)e * p.R + f);
          } else {
            const int col = 256 * ue.t + 128 * h2 + c;
            if (p.bias[0] && col < p.R) bv = __ldg(p.bias[0] + (size_t)e * p.R + col);
          }
          s_bias[128 * h2 + c] = bv;
        }
      }
      tc::named_sync(1, 32 * kEpiWarps);
      const bool okw = tc::mbar_wait_sleep(tc::smem_u32(&accf_bar), ldone & 1, abort_flag, 128);
      if (!__all_sync(0xffffffffu, okw)) {
        if (lane == 0) fail(2, ldone);
        break;
      }
      tc::fence_after_sync();
      if constexpr (KIND == 0) {
        // ---- gate/up: bias + swiglu of all 128 columns into registers, the
        // accumulator released, then h as E2M1 terms per 32-column block
        const int F = p.R;
        uint8_t* hq = p.hq + ((size_t)ue.b * p.NT + ue.t) * (size_t)(kPrefillHTerms * kChunk);
        uint8_t* hsf = p.hsf + (((size_t)ue.b * p.NT + ue.t) * kPrefillHTerms) * kAtom;
        const bool live = row < ue.live;
        float h[2][32];  // column groups 2*half, 2*half+1
#pragma unroll
        for (int gg = 0; gg < 2; ++gg) {
          const int g = 2 * half + gg;
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            uint32_t gv[16], uv[16];
            tc::tmem_ld16x2_wait(lane_base + 32 * g + 16 * hb, lane_base + 128 + 32 * g + 16 * hb, gv, uv);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int cc = 32 * g + 16 * hb + c;
              h[gg][16 * hb + c] = (live && 128 * ue.t + cc < F)
                                      ? swiglu_oai_fast(__uint_as_float(gv[c]) + s_bias[cc],
                                                        __uint_as_float(uv[c]) + s_bias[128 + cc], p.alpha, p.limit)
                                      : 0.f;
            }
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_u32(&acce_bar));  // the next unit's MMAs may start
#pragma unroll
        for (int gg = 0; gg < 2; ++gg) {
          const int g = 2 * half + gg;
          uint4 packed[kPrefillHTerms];
          uint32_t sc[kPrefillHTerms];
          mx::split_block_e2m1<kPrefillHTerms>(h[gg], packed, sc);
#pragma unroll
          for (int term = 0; term < kPrefillHTerms; ++term) {
            *reinterpret_cast<uint4*>(hq + act_off(row, term, kPrefillHTerms, g, 0)) = packed[term];
            hsf[(size_t)term * kAtom + dmx::atom_off(row, g)] = (uint8_t)sc[term];
          }
        }
      } else {
        // ---- down: y[token] += w_a * (acc + bd) over the pair's valid columns
        const int D = p.R;
        const int a = row < ue.live ? __ldg(p.rows + prow) : -1;
        const int tok = a >= 0 ? a / p.k : 0;
        const float wa = a >= 0 ? __ldg(p.weights + a) : 0.f;
#pragma unroll 1
        for (int g = 8 * half; g < 8 * half + 8; ++g) {
          uint32_t v[16];
          tc::tmem_ld16_wait(lane_base + 16 * g, v);
          if (g == 8 * half + 7) {
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_u32(&acce_bar));
          }
          if (a >= 0) {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int col = 256 * ue.t + 16 * g + c;
              if (col < D) atomicAdd(p.y + (size_t)tok * D + col, wa * (__uint_as_float(v[c]) + s_bias[16 * g + c]));
            }
          }
        }
      }
      ++ldone;
      have_e = next_unit(p, mpad, cur_epi, ue);
    }
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(tc::smem_u32(&tfree_bar));
    if (KIND == 0) asm volatile("fence.proxy.async.global;" ::: "memory");  // read next by the copy engine
  }

  // Tensor memory goes back once the epilogue warps and the MMA thread are done
  // with it (an mbarrier: no CTA-wide barrier after role loops run by lane 0 alone).
  if (warp == kTmemWarp) {
    tc::mbar_wait_sleep(tc::smem_u32(&tfree_bar), 0, nullptr, 64);
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// x rows in bucket order as kPrefillXTerms E2M1 terms, in the activation-chunk
// layout: one warp per (bucket row, 32-block); pad rows and blocks past D are
// zero. y[0 .. T*D) is zeroed (the down GEMM accumulates into it).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quant_rows_e2m1_kernel(const float* __restrict__ x, int T, int D, int k,
                                                              const int32_t* __restrict__ rows,
                                                              const int32_t* __restrict__ basep, int E, int NK,
                                                              uint8_t* __restrict__ aq, uint8_t* __restrict__ asf,
                                                              float* __restrict__ y) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int mpad = basep[E];
  const int nbp = 4 * NK, nb = D / 32;
  for (int64_t w = gw; w < (int64_t)mpad * nbp; w += nw) {
    const int p = (int)(w / nbp), blk = (int)(w - (int64_t)p * nbp);
    const int a = rows[p];
    float v = 0.f;
    if (a >= 0 && blk < nb) v = x[(size_t)(a / k) * D + 32 * blk + lane];
    uint32_t qv[kPrefillXTerms], sv[kPrefillXTerms];
    mx::split_terms_e2m1<kPrefillXTerms>(v, qv, sv);
    const int b = p >> 7, r = p & 127, j = blk >> 2, kb = blk & 3;
    const size_t base = ((size_t)b * NK + j) * kPrefillXTerms;
#pragma unroll
    for (int term = 0; term < kPrefillXTerms; ++term) {
      const uint32_t byte = mx::pack_e2m1_block(qv[term]);
      if (lane < 16) aq[((size_t)b * NK + j) * (kPrefillXTerms * kChunk) + act_off(r, term, kPrefillXTerms, kb, lane)] =
          (uint8_t)byte;
      if (lane == 0) asf[(base + term) * kAtom + dmx::atom_off(r, kb)] = (uint8_t)sv[term];
    }
  }
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (int64_t)T * D;
       i += (int64_t)gridDim.x * blockDim.x)
    y[i] = 0.f;
  asm volatile("fence.proxy.async.global;" ::: "memory");  // read next by the copy engine
}

}  // namespace gx4

size_t prefill_operand_bytes(int max_rows, int C, int terms) {
  return (size_t)(max_rows / 128) * ((C + 127) / 128) * terms * gx4::kChunk;
}
size_t prefill_atom_bytes(int max_rows, int C, int terms) {
  return (size_t)(max_rows / 128) * ((C + 127) / 128) * terms * gx4::kAtom;
}

cudaError_t launch_quant_rows_e2m1(const float* x, int T, int D, int k, const int32_t* rows, const int32_t* basep,
                                   int E, int max_rows, uint8_t* aq, uint8_t* asf, float* y, Launch L) {
  const int NK = (D + 127) / 128;
  const int64_t warps = (int64_t)max_rows * 4 * NK;
  int64_t blocks = (warps * 32 + 255) / 256;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_kernel(gx4::quant_rows_e2m1_kernel, dim3((unsigned)blocks), dim3(256), 0, L, x, T, D, k, rows, basep,
                       E, NK, aq, asf, y);
}

cudaError_t launch_grouped_mx4(const GroupedMX4Args& a, Launch L) {
  using namespace gx4;
  if (a.max_rows <= 0) return cudaSuccess;
  if (a.R % 64 != 0 || a.C % 64 != 0 || a.max_rows % 128 != 0 || (a.kind != 0 && a.kind != 1))
    return cudaErrorInvalidValue;
  Params prm{};
  prm.E = a.E;
  prm.R = a.R;
  prm.C = a.C;
  prm.NK = (a.C + 127) / 128;
  prm.NT = (a.R + 127) / 128;
  prm.npair = a.kind == 0 ? prm.NT : (prm.NT + 1) / 2;
  prm.ntiles = a.max_rows / 128;
  for (int m = 0; m < 2; ++m) {
    prm.w_qs[m] = a.w_qs[m];
    prm.w_sf[m] = a.w_sf[m];
    prm.bias[m] = a.bias[m];
  }
  prm.counts = a.counts;
  prm.basep = a.basep;
  prm.rows = a.rows;
  prm.k = a.k;
  prm.weights = a.weights;
  prm.aq = a.aq;
  prm.asf = a.asf;
  prm.hq = a.hq;
  prm.hsf = a.hsf;
  prm.alpha = a.alpha;
  prm.limit = a.limit;
  prm.y = a.y;
  prm.status = a.status;
  const int nunits = prm.ntiles * prm.npair;
  int grid = device_sm_count();
  if (grid > nunits) grid = nunits;
  if (a.kind == 0) {
    cudaError_t err = ensure_smem_limit(grouped_mx4_kernel<0>, Plan<0>::kDynSmem);
    if (err != cudaSuccess) return err;
    return launch_kernel(grouped_mx4_kernel<0>, dim3(grid), dim3(kThreads), Plan<0>::kDynSmem, L, prm);
  }
  cudaError_t err = ensure_smem_limit(grouped_mx4_kernel<1>, Plan<1>::kDynSmem);
  if (err != cudaSuccess) return err;
  return launch_kernel(grouped_mx4_kernel<1>, dim3(grid), dim3(kThreads), Plan<1>::kDynSmem, L, prm);
}

}  // namespace moe
