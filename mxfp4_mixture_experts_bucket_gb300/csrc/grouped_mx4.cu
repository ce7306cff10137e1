// Prefill grouped GEMMs on prepacked MXFP4 weights and the block-scaled tensor
// cores, tcgen05.mma kind::mxf4 (both operands E2M1 with E8M0 block scales):
// the bias-seeded MXFP4 gate/up and down grouped GEMMs of "dasLLAMA gpt-oss
// arc" (Metal fusion lane commit: MetalMoeMulMmMx4 over the MoeBucket CSR,
// swiglu rows past each bucket's live end skipped; the fused MoE expert chain
// commit: gate+up rows, bias, activation, then down rows, bias and the
// router-weighted sum) with neither operand dequantised.
//
// Orientation: the weights are the MMA's A operand (M = 128 weight rows of one
// tile) and the bucket rows its B operand, so N follows the live rows instead
// of the 128-row padding of a bucket tile. The activations enter as E2M1 terms
// (x: six, h: four; each block of 32 on its own E8M0 scale, each term the
// rounded residual of the ones before), and m terms share one MMA: B holds
// term t's rows, then term t+1's, ... (N = m * rn), and the groups of m terms
// accumulate into the same columns, so accumulator column j * rn + n holds the
// sum over the terms congruent to j mod m for row n; the epilogue adds the m
// slots, all in the thread that owns the weight row. m is the largest divisor
// of the term count with m * rn <= 192 (the tensor memory of one accumulator).
// An MMA costs about N / 2 cycles down to a floor near N = 110, so stacking
// terms keeps small segments off that floor.
//
// A bucket tile with L live rows is one segment when L <= 96, else two (rows
// 0..63 and 64..L-1); rn = the segment's rows rounded up to 16. A work unit is
// (segment, weight tile pair): gate/up: the gate and up tiles of 128 features
// (two accumulators); down: two 128-row tiles of D.
//
// Activation chunk layout (one per bucket tile and 128-column chunk): term t's
// 8192-byte image of the tile's 128 rows (64-byte-swizzled, block kb of row n
// at 64*n + 16*(kb ^ ((n>>1)&3))), terms one after the other, so a segment's
// rows of a term are one contiguous run. Its scale atoms: one run of `terms`
// atoms per segment; term t's scales for segment row r sit in atom
// (t / m) * ceil(m * rn / 128) + (n >> 7) at row n & 127, n = (t % m) * rn + r
// (B row n of the term group's MMA). Written by quant_rows_e2m1_kernel: x from the token rows,
// h from the float rows the gate/up epilogue leaves.
//
// Warps: 0..3 scale loaders (one per tensor-memory lane quarter: each step's
// scale atoms into tensor memory with tcgen05.st once its data has landed,
// then a signal to the MMA thread), 4..5 copy issuers (activations; weights),
// 6 MMA issuer, 7..14 epilogue (two per lane quarter; warp 7 owns tensor
// memory). Units are handed out dynamically: the activation copy issuer takes
// each next unit index from a global counter per GEMM and publishes it in a
// small shared-memory ring that every other role reads in order. The
// accumulators are freed as soon as the epilogue has read them, so the
// epilogue's remaining work overlaps the next unit's MMAs.
//   gate/up epilogue: (first, while the first unit streams: y zeroed for the
//     down GEMM) bias, swiglu_oai of every (feature, row) into registers,
//     accumulators freed, then h stored as float rows (32 consecutive
//     features per warp and row).
//   down epilogue: every 16-row chunk of the accumulator read into registers,
//     accumulator freed, then y[t] += w_a * (acc + bd) for each row's
//     assignment a (float atomics over 32 consecutive outputs per warp, as the
//     pages' weighted scatter).
#include <cuda.h>

#include "decode_mx.cuh"
#include "mx_terms.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace gx4 {

constexpr int kProd = 6;
constexpr int kMmaWarp = 6;
constexpr int kEpiWarp0 = 7;
constexpr int kEpiWarps = 8;  // two per tensor-memory lane quarter
constexpr int kTmemWarp = 7;
constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;
constexpr int kTermBytes = 8192;  // one term's image of a bucket tile chunk: 128 rows x 64 bytes
constexpr int kTileBytes = 8192;  // one weight tile chunk: 128 rows x 64 bytes
constexpr int kAtom = 512;
constexpr int kSegMax = 96;          // most rows in one segment
constexpr uint32_t kAccStride = 192;  // tensor-memory columns of one accumulator: m * rn <= 192
constexpr uint32_t kSfBase = 2 * kAccStride;  // scale atoms after the two accumulators
constexpr uint32_t kTmemCols = 512;

__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }

// Per-kernel plan: the activation operand's terms (x: kPrefillXTerms, h:
// kPrefillHTerms), the stage layout [two weight tiles][terms x kSegMax rows]
// [activation atoms][two weight atoms], its scale columns, and the ring depth
// that fits both 227 KB of shared memory and the tensor memory left for scales.
template <int KIND>
struct Plan {
  static constexpr int kTerms = KIND == 0 ? kPrefillXTerms : kPrefillHTerms;
  static constexpr uint32_t kOffAct = 2 * kTileBytes;
  static constexpr uint32_t kOffSfa = kOffAct + kTerms * kSegMax * 64;
  static constexpr uint32_t kOffSfw = kOffSfa + kTerms * kAtom;
  static constexpr uint32_t kStageBytes = ((kOffSfw + 2 * kAtom) + 1023u) & ~1023u;
  static constexpr uint32_t kSfCols = 4 * kTerms + 8;  // per stage: the activation atoms, then the two weight atoms
  static constexpr int kStages =
      cmin(6, cmin((int)((226u * 1024u) / kStageBytes), (int)((kTmemCols - kSfBase) / kSfCols)));
  static constexpr uint32_t kDynSmem = kStages * kStageBytes + 512;
};
static_assert(Plan<0>::kStages >= 3 && Plan<1>::kStages >= 3, "ring depth");
static_assert(kSfBase + Plan<0>::kStages * Plan<0>::kSfCols <= kTmemCols, "tensor memory plan");
static_assert(kSfBase + Plan<1>::kStages * Plan<1>::kSfCols <= kTmemCols, "tensor memory plan");

struct Params {
  int E, R, C, NK, NT;  // weight matrices [R][C]: NT tiles of 128 rows, NK chunks of 128 columns
  int npair;            // weight tile pairs per segment (gate/up: NT; down: ceil(NT / 2))
  int ntiles;           // bucket tiles (max_rows / 128)
  const uint8_t* w_qs[2];
  const uint8_t* w_sf[2];
  const float* bias[2];
  const int32_t* counts;
  const int32_t* basep;
  const int32_t* rows;
  const int2* segs;    // the segment table: segs[0].x = count; segs[1 + i] = ((b << 1) | s, (e << 8) | live)
  int* ctr;            // units handed out so far (zeroed by the x quantiser)
  int k;
  const float* weights;
  const uint8_t* aq;   // activation chunks [ntiles][NK][terms][8192]
  const uint8_t* asf;  // [ntiles][NK][2 segments][terms][512]
  float* hf;           // gate/up: h as float rows [ntiles * 128][R]
  float alpha, limit;
  float* y;  // down: [T][R], accumulated into; gate/up: zeroed (ny floats) by the epilogue warps
  int64_t ny;
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

// Segments of a bucket tile with `live` rows: segment s's first row, row
// count, and rows rounded up to 16 (0 rows: no such segment).
struct Segment {
  int base, rows, rn;
};
__host__ __device__ __forceinline__ Segment segment_of(int live, int s) {
  Segment g{64 * s, 0, 0};
  if (live > kSegMax) g.rows = s == 0 ? 64 : live - 64;
  else g.rows = s == 0 ? live : 0;
  g.rn = (g.rows + 15) & ~15;
  return g;
}
// Terms per MMA for a segment of rn rows: the largest divisor m of `terms`
// with m * rn <= kAccStride (m = 1 always fits: rn <= 96).
template <int TERMS>
__host__ __device__ __forceinline__ int slots_of(int rn) {
  int m = 1;
#pragma unroll
  for (int d = 2; d <= TERMS; ++d)
    if (TERMS % d == 0 && d * rn <= (int)kAccStride) m = d;
  return m;
}
// Scale atoms per term group (one per 128 B rows of the group's MMA).
__host__ __device__ __forceinline__ int atoms_per_group(int m, int rn) { return (m * rn + 127) >> 7; }

// Atom (within the segment's run) and atom row of the scales of term t,
// segment row r: B row n = (t % m) * rn + r of group t / m. At most `terms`
// atoms: a group of m >= 2 terms takes at most 2 (m * rn <= 192), a single
// term 1 (rn <= 96).
__host__ __device__ __forceinline__ int atom_index(int t, int m, int rn, int r, int& n) {
  const int nn = (t % m) * rn + r;
  n = nn & 127;
  return (t / m) * atoms_per_group(m, rn) + (nn >> 7);
}

// Atoms a segment of rn rows uses: the first (terms / m) * ceil(m * rn / 128)
// of its run.
template <int TERMS>
__host__ __device__ __forceinline__ int used_atoms(int rn) {
  const int m = slots_of<TERMS>(rn);
  return (TERMS / m) * atoms_per_group(m, rn);
}

// A work unit: bucket tile b (expert e), segment s, weight tile pair t.
struct Unit {
  int b, s, t, e;
  Segment g;
};

// Unit v: segment v / npair of the segment table (every segment of every live
// bucket tile, in bucket order) and weight tile pair v % npair.
__device__ __forceinline__ void decode_unit(const Params& p, int v, Unit& u) {
  const int si = v / p.npair;
  const int2 sg = __ldg(p.segs + 1 + si);
  u.b = sg.x >> 1;
  u.s = sg.x & 1;
  u.t = v - si * p.npair;
  u.e = sg.y >> 8;
  u.g = segment_of(sg.y & 255, u.s);
}

// Units are handed out dynamically: the activation copy issuer of each CTA takes
// the next index from a global counter and publishes it in a small ring in
// shared memory; every other role reads the CTA's units from the ring in order.
constexpr int kUnitRing = 4;
constexpr int kUnitReaders = 1 + 4 + 1 + kEpiWarps;  // weight copies, scale loaders, MMA thread, epilogue warps

// 16 columns from column c0 of the accumulator at `acc` (this warp's lanes),
// summed over its m term slots (slot j at column j * rn + c0).
__device__ __forceinline__ void slot_sum16(uint32_t acc, int c0, int rn, int m, float (&out)[16]) {
  uint32_t a0[16], a1[16];
  if (m == 1) {
    tc::tmem_ld16_wait(acc + c0, a0);
#pragma unroll
    for (int k = 0; k < 16; ++k) out[k] = __uint_as_float(a0[k]);
    return;
  }
  tc::tmem_ld16x2_wait(acc + c0, acc + rn + c0, a0, a1);
#pragma unroll
  for (int k = 0; k < 16; ++k) out[k] = __uint_as_float(a0[k]) + __uint_as_float(a1[k]);
  for (int j = 2; j < m; j += 2) {
    if (j + 1 < m) {
      tc::tmem_ld16x2_wait(acc + j * rn + c0, acc + (j + 1) * rn + c0, a0, a1);
#pragma unroll
      for (int k = 0; k < 16; ++k) out[k] += __uint_as_float(a0[k]) + __uint_as_float(a1[k]);
    } else {
      tc::tmem_ld16_wait(acc + j * rn + c0, a0);
#pragma unroll
      for (int k = 0; k < 16; ++k) out[k] += __uint_as_float(a0[k]);
    }
  }
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1) grouped_mx4_kernel(const Params p) {
  using PL = Plan<KIND>;
  constexpr int kTerms = PL::kTerms, kStages = PL::kStages;
  constexpr uint32_t kOffAct = PL::kOffAct, kOffSfa = PL::kOffSfa, kOffSfw = PL::kOffSfw;
  constexpr uint32_t kStageBytes = PL::kStageBytes, kSfCols = PL::kSfCols;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 511) &
                                             ~static_cast<uintptr_t>(511));
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t sfr_bar[kStages];
  __shared__ __align__(8) uint64_t accf_bar, acce_bar, drain_bar, tfree_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_unit[kUnitRing];
  __shared__ __align__(8) uint64_t ufull_bar[kUnitRing], uempty_bar[kUnitRing];
  __shared__ float s_bias[256];  // the unit's biases (gate/up: 128 gate, 128 up; down: 256)
  __shared__ int s_tok[KIND == 1 ? kSegMax : 1];    // down: each segment row's token (-1: none)
  __shared__ float s_w[KIND == 1 ? kSegMax : 1];    // and its router weight
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == 1 && lane == 0) {
    for (int i = 0; i < kStages; ++i) {
      tc::mbar_init(tc::smem_u32(&full_bar[i]), 2);  // the two copy issuers
      tc::mbar_init(tc::smem_u32(&empty_bar[i]), 1);
      tc::mbar_init(tc::smem_u32(&sfr_bar[i]), 4);
    }
    tc::mbar_init(tc::smem_u32(&accf_bar), 1);
    tc::mbar_init(tc::smem_u32(&acce_bar), kEpiWarps);
    tc::mbar_init(tc::smem_u32(&drain_bar), 1);
    for (int i = 0; i < kUnitRing; ++i) {
      tc::mbar_init(tc::smem_u32(&ufull_bar[i]), 1);
      tc::mbar_init(tc::smem_u32(&uempty_bar[i]), kUnitReaders);
    }
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
  const int nseg = __ldg(&p.segs[0].x);
  const int NK = p.NK;
  const volatile int* abort_flag = &s_abort;
  auto fail = [&](int role, int seq) {
    s_abort = 1;
    report_timeout(p.status, 7 + KIND, role, 0, seq);
  };
  const int nbc = p.C / 32;
  const int nunits = nseg * p.npair;
  // the issuer publishes the CTA's unit n (the counter's next index, -1 once they are all
  // handed out); returns it, or -2 if the wait for the ring slot gave up
  auto publish = [&](int n) -> int {
    const int slot = n % kUnitRing;
    if (n >= kUnitRing &&
        !tc::mbar_wait_sleep(tc::smem_u32(&uempty_bar[slot]), (n / kUnitRing - 1) & 1, abort_flag, 32))
      return -2;
    int v = atomicAdd(p.ctr, 1);
    if (v >= nunits) v = -1;
    *reinterpret_cast<volatile int*>(&s_unit[slot]) = v;
    tc::mbar_arrive(tc::smem_u32(&ufull_bar[slot]));
    return v;
  };
  // a reader takes the CTA's unit n (one lane, or every lane of a warp); false at the end
  // of the units or if the wait gave up (then *abort_flag is set)
  auto take = [&](int n, Unit& u, bool warp_wide, int role) -> bool {
    const int slot = n % kUnitRing;
    bool okw = tc::mbar_wait_sleep(tc::smem_u32(&ufull_bar[slot]), (n / kUnitRing) & 1, abort_flag, 32);
    if (warp_wide) okw = __all_sync(0xffffffffu, okw);
    if (!okw) {
      if (!warp_wide || lane == 0) fail(role, n);
      return false;
    }
    const int v = *reinterpret_cast<volatile int*>(&s_unit[slot]);
    if (warp_wide) __syncwarp();
    if (!warp_wide || lane == 0) tc::mbar_arrive(tc::smem_u32(&uempty_bar[slot]));
    if (v < 0) return false;
    decode_unit(p, v, u);
    return true;
  };
  // weight tile h of unit u's pair (gate/up: matrix h of tile t; down: tile 2t + h), or -1
  auto wtile = [&](const Unit& u, int h) { return KIND == 0 ? u.t : (2 * u.t + h < p.NT ? 2 * u.t + h : -1); };

  if (warp < 4) {
    // ------------------------------------------------ scale loaders, one per tensor-memory lane
    // quarter: step by step, once a step's data has landed, its scale atoms go into this
    // warp's lane quarter (tcgen05.st) and the MMA thread is signalled. They never hold up
    // the copies, which run up to kStages steps ahead.
    const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
    int un = 0, i = 0;
    Unit u;
    bool ok = true;
    while (ok && take(un++, u, true, 4)) {
      const int na = used_atoms<kTerms>(u.g.rn);
      for (int j = 0; j < NK; ++j, ++i) {
        const int st = i % kStages, n = i / kStages;
        const bool okw = tc::mbar_wait_sleep(tc::smem_u32(&full_bar[st]), n & 1, abort_flag, 32);
        if (!__all_sync(0xffffffffu, okw)) {
          if (lane == 0) fail(3, i);
          ok = false;
          break;
        }
        const uint8_t* sbp = smem + (size_t)st * kStageBytes;
        const uint32_t sfs = lane_base + kSfBase + (uint32_t)st * kSfCols;
#pragma unroll 1
        for (int a = 0; a < na; ++a) {  // the activation atoms the segment's MMAs read
          const uint4 w = *reinterpret_cast<const uint4*>(sbp + kOffSfa + a * kAtom + 16 * lane);
          tc::tmem_st4(sfs + 4 * a, w.x, w.y, w.z, w.w);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // the two weight atoms
          const uint4 w = *reinterpret_cast<const uint4*>(sbp + kOffSfw + h * kAtom + 16 * lane);
          tc::tmem_st4(sfs + 4 * (kTerms + h), w.x, w.y, w.z, w.w);
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sfr_bar[st]));
      }
    }
    tc::fence_before_sync();  // this warp's tensor-memory stores are complete
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(tc::smem_u32(&tfree_bar));
  } else if (warp < kProd) {
    // ------------------------------------------------ copy issuers (lane 0): warp 4 the
    // segment's rows of every activation term and their atoms, warp 5 the two weight
    // tiles and their atoms
    if (lane == 0) {
      uint64_t pol = tc::l2_policy_evict_first();
      int un = 0, i = 0, issued = 0;
      Unit u;
      bool ok = true;
      while (ok) {
        if (warp == 4) {  // the scheduler
          const int v = publish(un++);
          if (v == -2) fail(5, un - 1);
          if (v < 0) break;
          decode_unit(p, v, u);
        } else if (!take(un++, u, false, 5)) {
          break;
        }
        const uint32_t run = (uint32_t)u.g.rn * 64;  // one term's rows of the segment
        for (int j = 0; j < NK; ++j, ++i) {
          const int st = i % kStages, n = i / kStages;
          if (n > 0 && !tc::mbar_wait_sleep(tc::smem_u32(&empty_bar[st]), (n - 1) & 1, abort_flag, 32)) {
            fail(0, i);
            ok = false;
            break;
          }
          const uint32_t fb = tc::smem_u32(&full_bar[st]);
          const uint32_t sb = tc::smem_u32(smem) + (uint32_t)st * kStageBytes;
          if (warp == 4) {
            const size_t achunk = (size_t)u.b * NK + j;
            const uint8_t* src = p.aq + achunk * (size_t)(kTerms * kTermBytes) + (size_t)u.g.base * 64;
            const uint32_t abytes = (uint32_t)used_atoms<kTerms>(u.g.rn) * kAtom;
            if (!MOE_IN_BOUNDS(p.status, u.b >= 0 && u.b < p.ntiles && u.g.base + u.g.rn <= 128)) {
              tc::mbar_expect_tx(fb, 0);  // the stage completes without this part
            } else {
              tc::mbar_expect_tx(fb, (uint32_t)kTerms * run + abytes);
              for (int t = 0; t < kTerms; ++t)
                tc::bulk_load(sb + kOffAct + (uint32_t)t * run, src + (size_t)t * kTermBytes, run, fb);
              tc::bulk_load(sb + kOffSfa, p.asf + (achunk * 2 + u.s) * (kTerms * kAtom), abytes, fb);
            }
          } else {
            // a tile shorter than 128 rows leaves the rest stale: those rows only feed
            // accumulator lanes nobody reads
            const bool wok = MOE_IN_BOUNDS(p.status, u.e >= 0 && u.e < p.E && wtile(u, 0) < p.NT);
            uint32_t bytes = 0;
            for (int h = 0; h < 2; ++h) {
              const int tile = wtile(u, h);
              if (tile >= 0 && wok) bytes += (uint32_t)(min(128, p.R - 128 * tile) * 64) + kAtom;
            }
            tc::mbar_expect_tx(fb, bytes);
            for (int h = 0; h < 2; ++h) {
              const int tile = wtile(u, h);
              if (tile < 0 || !wok) continue;
              const int rows_t = min(128, p.R - 128 * tile);
              const uint8_t* src = p.w_qs[KIND == 0 ? h : 0] +
                                   ((size_t)u.e * p.R + 128 * (size_t)tile) * ((size_t)NK * 64) + (size_t)rows_t * 64 * j;
              tc::bulk_load_stream(sb + (uint32_t)(h * kTileBytes), src, (uint32_t)(rows_t * 64), fb, pol);
              tc::bulk_load_stream(sb + kOffSfw + (uint32_t)(h * kAtom),
                                   p.w_sf[KIND == 0 ? h : 0] + (((size_t)u.e * p.NT + tile) * NK + j) * kAtom, kAtom,
                                   fb, pol);
            }
          }
          issued = i + 1;
        }
      }
      if (*abort_flag) {  // every copy already issued lands before shared memory goes away
        for (int st = 0; st < kStages; ++st) {
          const int n = issued > st ? (issued - 1 - st) / kStages + 1 : 0;
          if (n > 0) tc::mbar_wait(tc::smem_u32(&full_bar[st]), (n - 1) & 1, nullptr);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      int i = 0, lu = 0;
      Unit u;
      bool ok = true;
      while (ok && take(lu, u, false, 1)) {
        if (lu > 0 && !tc::mbar_wait_sleep(tc::smem_u32(&acce_bar), (lu - 1) & 1, abort_flag, 32)) {
          fail(1, i);
          break;
        }
        tc::fence_after_sync();
        const int m = slots_of<kTerms>(u.g.rn), ngrp = kTerms / m, apg = atoms_per_group(m, u.g.rn);
        const uint32_t idesc = idesc_mxf4(128, m * u.g.rn);
        const bool two = wtile(u, 1) >= 0;
        const uint32_t grp_step = (uint32_t)(m * u.g.rn * 64) >> 4;  // descriptor units between term groups
        for (int j = 0; j < NK; ++j, ++i) {
          const int st = i % kStages, n = i / kStages;
          if (!tc::mbar_wait(tc::smem_u32(&sfr_bar[st]), n & 1, abort_flag)) {
            fail(1, i);
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t sb = tc::smem_u32(smem) + (uint32_t)st * kStageBytes;
          const uint32_t sfs = tmem + kSfBase + (uint32_t)st * kSfCols;
          const int nkb = min(4, nbc - 4 * j);  // 32-blocks in this chunk: 2 or 4 (widths are multiples of 64)
          const uint64_t adesc0 = tc::sw64_kmajor_desc(sb);
          const uint64_t adesc1 = tc::sw64_kmajor_desc(sb + kTileBytes);
          const uint64_t bdesc = tc::sw64_kmajor_desc(sb + kOffAct);
#pragma unroll
          for (int kh = 0; kh < 2; ++kh) {
            if (2 * kh >= nkb) continue;
            const uint32_t id = idesc | (kh ? ((2u << 4) | (2u << 29)) : 0u);
#pragma unroll 1
            for (int q = 0; q < ngrp; ++q) {
              const uint64_t bq = bdesc + (uint64_t)(q * grp_step + 2 * kh);
              const uint32_t sfb = sfs + 4 * q * apg;
              const uint32_t acc = (j == 0 && kh == 0 && q == 0) ? 0u : 1u;
              mma_mxf4(tmem, adesc0 + (uint64_t)(2 * kh), bq, id, sfs + 4 * kTerms, sfb, acc);
              if (two) mma_mxf4(tmem + kAccStride, adesc1 + (uint64_t)(2 * kh), bq, id, sfs + 4 * kTerms + 4, sfb, acc);
            }
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
    const int hh = (warp - kEpiWarp0) >> 2;  // gate/up: which row chunks; down: which tile of the pair
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
    const int et = threadIdx.x - kEpiWarp0 * 32;  // 0..255
    if (KIND == 0 && p.y) {
      // the down GEMM's output, zeroed while the first unit's MMAs run (the down
      // kernel starts after this one has completed)
      const int64_t n4 = p.ny >> 2, stride = (int64_t)gridDim.x * 32 * kEpiWarps;
      float4* y4 = reinterpret_cast<float4*>(p.y);
      for (int64_t i = (int64_t)blockIdx.x * 32 * kEpiWarps + et; i < n4; i += stride)
        y4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int64_t i = 4 * n4 + (int64_t)blockIdx.x * 32 * kEpiWarps + et; i < p.ny; i += stride) p.y[i] = 0.f;
    }
    Unit ue{};
    int ldone = 0;  // units whose epilogue has run
    bool have_e = take(0, ue, true, 2);
    while (have_e) {
      // ---- the epilogue of unit ldone (ue)
      const int e = ue.e;
      const Segment g = ue.g;
      // the unit's biases (and, down, its rows' tokens) into shared memory; every
      // reader of the previous unit's is past the first barrier
      tc::named_sync(1, 32 * kEpiWarps);
      {
        float bv = 0.f;
        if (KIND == 0) {
          const int h2 = et >> 7, f = 128 * ue.t + (et & 127);
          if (p.bias[h2] && f < p.R && MOE_IN_BOUNDS(p.status, e >= 0 && e < p.E)) bv = __ldg(p.bias[h2] + (size_t)e * p.R + f);
        } else {
          const int col = 256 * ue.t + et;
          if (p.bias[0] && col < p.R && MOE_IN_BOUNDS(p.status, e >= 0 && e < p.E)) bv = __ldg(p.bias[0] + (size_t)e * p.R + col);
          if (et < kSegMax) {
            const int a = et < g.rows ? __ldg(p.rows + 128 * ue.b + g.base + et) : -1;
            s_tok[et] = a >= 0 ? a / p.k : -1;
            s_w[et] = a >= 0 ? __ldg(p.weights + a) : 0.f;
          }
        }
        s_bias[et] = bv;
      }
      tc::named_sync(1, 32 * kEpiWarps);
      const bool okw = tc::mbar_wait_sleep(tc::smem_u32(&accf_bar), ldone & 1, abort_flag, 128);
      if (!__all_sync(0xffffffffu, okw)) {
        if (lane == 0) fail(2, ldone);
        break;
      }
      tc::fence_after_sync();
      if constexpr (KIND == 0) {
        // ---- gate/up: this lane's feature f; rows in 16-row chunks hh, hh + 2, hh + 4
        const int m = slots_of<kPrefillXTerms>(g.rn);
        const int fl = 32 * q + lane, f = 128 * ue.t + fl;
        const bool fvalid = f < p.R;
        const float bg = s_bias[fl], bu = s_bias[128 + fl];
        float hv[3][16];
#pragma unroll
        for (int ci = 0; ci < 3; ++ci) {
          const int c = hh + 2 * ci;
          if (16 * c < g.rn) {
            float gs[16], us[16];
            slot_sum16(lane_base, 16 * c, g.rn, m, gs);
            slot_sum16(lane_base + kAccStride, 16 * c, g.rn, m, us);
#pragma unroll
            for (int k = 0; k < 16; ++k) hv[ci][k] = swiglu_oai_fast(gs[k] + bg, us[k] + bu, p.alpha, p.limit);
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_u32(&acce_bar));  // the next unit's MMAs may start
        // h rows: 32 consecutive features per warp and row
        float* hrow = p.hf + (size_t)(128 * ue.b + g.base) * p.R + f;
#pragma unroll
        for (int ci = 0; ci < 3; ++ci) {
          const int c = hh + 2 * ci;
          if (16 * c >= g.rows) continue;
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int r = 16 * c + k;
            if (fvalid && r < g.rows && MOE_IN_BOUNDS(p.status, 128 * ue.b + g.base + r < 128 * p.ntiles))
              hrow[(size_t)r * p.R] = hv[ci][k];
          }
        }
      } else {
        // ---- down: output d of tile hh; y[token] += w_a * (acc + bd) for the segment's rows
        const int m = slots_of<kPrefillHTerms>(g.rn);
        const int D = p.R;
        const int dl = 128 * hh + 32 * q + lane, d = 256 * ue.t + dl;
        const bool has = wtile(ue, hh) >= 0;
        const bool dvalid = has && d < D;
        const float bd = s_bias[dl];
        const uint32_t acc = lane_base + kAccStride * hh;
        const int nch = (g.rows + 15) >> 4;
        if (!has) {
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(tc::smem_u32(&acce_bar));
        } else {
          // every chunk is read out before the accumulator goes back, so the next
          // unit's MMAs need not wait for this unit's scatter
          float v[kSegMax / 16][16];
#pragma unroll
          for (int c = 0; c < kSegMax / 16; ++c)
            if (c < nch) slot_sum16(acc, 16 * c, g.rn, m, v[c]);
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(tc::smem_u32(&acce_bar));
#pragma unroll
          for (int c = 0; c < kSegMax / 16; ++c) {
            if (c >= nch) break;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const int r = 16 * c + k;
              const int tok = r < g.rows ? s_tok[r] : -1;
              if (dvalid && tok >= 0 && MOE_IN_BOUNDS(p.status, (int64_t)tok * D + d < p.ny))
                atomicAdd(p.y + (size_t)tok * D + d, s_w[r] * (v[c][k] + bd));
            }
          }
        }
      }
      ++ldone;
      have_e = take(ldone, ue, true, 2);
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
// Bucket rows as NT E2M1 terms, in the activation-chunk layout: each 32-block
// is loaded (128 bytes) and split (split_half_block_e2m1_term) by a lane pair,
// each lane storing its 8 bytes of every term, one lane the scale bytes into
// the segment's atoms.
// GATHER (x, the gate/up operand): a lane pair per (token, 32-block) splits the
// block once and stores it into each of the token's k bucket rows (inv); pad
// rows up to each segment's rounded end are zeroed; y[0 .. T*C) is zeroed
// unless null (the down GEMM accumulates into it) and block 0 writes the
// segment table. Else (h, the down operand): a lane pair per (bucket row,
// 32-block) of src's own rows, pad rows zero. Blocks past C are zero; rows
// past a segment's rounded end are never read and not written.
// ---------------------------------------------------------------------------
// Stores a row's NT terms of one 32-block: the codes at `row` (the row's 16
// bytes of block kb in term 0's image; term t sits t * kTermBytes further) and
// the scale codes into the segment's atoms (segment of rn rows, segment row r;
// atom_index's placement, the term groups walked in order instead of divided).
template <int NT>
__device__ __forceinline__ void store_terms(uint8_t* row, uint8_t* atoms, int rn, int r, int kb,
                                            const uint4 (&packed)[NT], const uint32_t (&sc)[NT]) {
  const int m = slots_of<NT>(rn), apg = atoms_per_group(m, rn);
  int slot = 0, grp = 0;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    *reinterpret_cast<uint4*>(row + (size_t)t * kTermBytes) = packed[t];
    const int nn = slot * rn + r;  // B row of the group's MMA
    atoms[(size_t)(grp * apg + (nn >> 7)) * kAtom + dmx::atom_off(nn & 127, kb)] = (uint8_t)sc[t];
    if (++slot == m) {
      slot = 0;
      ++grp;
    }
  }
}

// The same for a lane pair's half of the block: this lane's 8 bytes of each
// term at `row` (already offset to the lane's half); the scale codes only if
// `scales` (one lane of the pair).
template <int NT>
__device__ __forceinline__ void store_half_terms(uint8_t* row, uint8_t* atoms, int rn, int r, int kb, bool scales,
                                                 const uint2 (&packed)[NT], const uint32_t (&sc)[NT]) {
  const int m = slots_of<NT>(rn), apg = atoms_per_group(m, rn);
  int slot = 0, grp = 0;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    *reinterpret_cast<uint2*>(row + (size_t)t * kTermBytes) = packed[t];
    const int nn = slot * rn + r;
    if (scales) atoms[(size_t)(grp * apg + (nn >> 7)) * kAtom + dmx::atom_off(nn & 127, kb)] = (uint8_t)sc[t];
    if (++slot == m) {
      slot = 0;
      ++grp;
    }
  }
}

template <int NT, bool GATHER>
__global__ void __launch_bounds__(256, 3) quant_rows_e2m1_kernel(const float* __restrict__ src, int T, int C, int k,
                                                              const int32_t* __restrict__ rows,
                                                              const int32_t* __restrict__ counts,
                                                              const int32_t* __restrict__ basep, int E, int NK,
                                                              uint8_t* __restrict__ aq, uint8_t* __restrict__ asf,
                                                              float* __restrict__ y, int2* __restrict__ segs,
                                                              const int32_t* __restrict__ inv, int* __restrict__ ctr,
                                                              int* status) {
  pdl_launch_dependents();
  pdl_wait();
  if (GATHER && blockIdx.x == 0 && threadIdx.x == 32) {  // the GEMMs' unit counters
    ctr[0] = 0;
    ctr[1] = 0;
  }
  if (GATHER && blockIdx.x == 0 && threadIdx.x < 32) {
    // the segment table: one lane per expert, a warp prefix over the experts' segment counts
    const int lane = threadIdx.x;
    int total = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int cnt = e < E ? counts[e] : 0;
      const int t0 = e < E ? (basep[e] >> 7) : 0;
      const int ntl = (cnt + 127) >> 7;
      int ns = 0;
      for (int i = 0; i < ntl; ++i) ns += min(128, cnt - 128 * i) > kSegMax ? 2 : 1;
      int incl = ns;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int pos = total + incl - ns;
      for (int i = 0; i < ntl; ++i) {
        const int live = min(128, cnt - 128 * i);
        for (int sg = 0; sg < (live > kSegMax ? 2 : 1); ++sg)
          segs[1 + pos++] = make_int2(((t0 + i) << 1) | sg, (e << 8) | live);
      }
      total += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) segs[0] = make_int2(total, 0);
  }
  // every bucket tile's live rows, once per block: each expert's tiles follow
  // one another from its padded base
  extern __shared__ int s_live[];
  const int mpad = basep[E];
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int cnt = counts[e], b0 = basep[e] >> 7;
    for (int i = 0; 128 * i < cnt; ++i) s_live[b0 + i] = min(128, cnt - 128 * i);
  }
  __syncthreads();
  const int tid = blockIdx.x * blockDim.x + threadIdx.x;
  const int nthr = gridDim.x * blockDim.x;
  const int nbp = 4 * NK, nb = C / 32;
  uint4 zq[NT];  // a zero row: every code 0, every scale code 0
  uint32_t zs[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    zq[t] = make_uint4(0u, 0u, 0u, 0u);
    zs[t] = 0u;
  }
  if constexpr (GATHER) {
    // the tokens: each block split once by a lane pair (both lanes of a pair take the
    // same item: nthr and tid keep their parity), its terms stored into the token's
    // k bucket rows
    const int hf = threadIdx.x & 1;
    const uint32_t pair = 3u << (threadIdx.x & 30);
    for (int64_t w2 = tid; w2 < 2 * (int64_t)T * nbp; w2 += nthr) {
      const int w = (int)(w2 >> 1);
      const int t = w / nbp, blk = w - t * nbp, j = blk >> 2, kb = blk & 3;
      float v[16];
      if (blk < nb) {
        const float4* s4 = reinterpret_cast<const float4*>(src + (size_t)t * C + 32 * blk + 8 * hf);
        const float4 f0 = __ldg(s4), f1 = __ldg(s4 + 1), f2 = __ldg(s4 + 4), f3 = __ldg(s4 + 5);
        v[0] = f0.x; v[1] = f0.y; v[2] = f0.z; v[3] = f0.w; v[4] = f1.x; v[5] = f1.y; v[6] = f1.z; v[7] = f1.w;
        v[8] = f2.x; v[9] = f2.y; v[10] = f2.z; v[11] = f2.w; v[12] = f3.x; v[13] = f3.y; v[14] = f3.z; v[15] = f3.w;
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.f;
      }
      uint2 packed[NT];
      uint32_t sc[NT];
#pragma unroll
      for (int term = 0; term < NT; ++term)
        mx::split_half_block_e2m1_term(v, term + 1 == NT, pair, packed[term], sc[term]);
      for (int jj = 0; jj < k; ++jj) {
        const int p = __ldg(inv + (size_t)t * k + jj);
        if (p < 0) continue;  // an invalid expert id: the assignment has no bucket row
        if (!MOE_IN_BOUNDS(status, p < mpad)) continue;
        const int b = p >> 7, rt = p & 127;
        const int live = s_live[b];
        const int s = live > kSegMax ? (rt >> 6) : 0;
        const Segment g = segment_of(live, s);
        store_half_terms<NT>(aq + ((size_t)b * NK + j) * (NT * kTermBytes) + dmx::chunk_off(rt, kb, 8 * hf),
                             asf + (((size_t)b * NK + j) * 2 + s) * (NT * kAtom), g.rn, rt - g.base, kb, hf == 0,
                             packed, sc);
      }
    }
    // the pad rows of every segment, up to its rounded end: zero terms, scale code 0
    for (int w = tid; w < (mpad >> 7) * 16 * nbp; w += nthr) {
      const int b = w / (16 * nbp), rem = w - b * (16 * nbp), pr = rem / nbp, blk = rem - pr * nbp;
      const int live = s_live[b];
      const int s = live > kSegMax ? 1 : 0;
      const Segment g = segment_of(live, s);
      const int rt = live + pr;
      if (rt >= g.base + g.rn) continue;
      const int j = blk >> 2, kb = blk & 3;
      store_terms<NT>(aq + ((size_t)b * NK + j) * (NT * kTermBytes) + dmx::chunk_off(rt, kb, 0),
                      asf + (((size_t)b * NK + j) * 2 + s) * (NT * kAtom), g.rn, rt - g.base, kb, zq, zs);
    }
  } else {
    // a lane pair per (bucket row, 32-block): both lanes of a pair always take
    // the same item (nthr and tid keep their parity), so they skip or split it together
    const int hf = threadIdx.x & 1;
    const uint32_t pair = 3u << (threadIdx.x & 30);
    const int64_t nitem = 2 * (int64_t)mpad * nbp;
    for (int64_t w2 = tid; w2 < nitem; w2 += nthr) {
      const int w = (int)(w2 >> 1);
      const int p = w / nbp, blk = w - p * nbp;
      const int b = p >> 7, rt = p & 127, j = blk >> 2, kb = blk & 3;
      const int live = s_live[b];
      const int s = live > kSegMax ? (rt >> 6) : 0;
      const Segment g = segment_of(live, s);
      const int r = rt - g.base;
      if (r >= g.rn) continue;  // rows past the segment's rounded end are never read
      const int a = rows[p];
      const int m = slots_of<NT>(g.rn);
      uint8_t* chunk = aq + ((size_t)b * NK + j) * (NT * kTermBytes) + dmx::chunk_off(rt, kb, 8 * hf);
      uint8_t* atoms = asf + (((size_t)b * NK + j) * 2 + s) * (NT * kAtom);
      float v[16];
      if (a >= 0 && blk < nb) {
        const float4* s4 = reinterpret_cast<const float4*>(src + (size_t)p * C + 32 * blk + 8 * hf);
        const float4 f0 = __ldg(s4), f1 = __ldg(s4 + 1), f2 = __ldg(s4 + 4), f3 = __ldg(s4 + 5);
        v[0] = f0.x; v[1] = f0.y; v[2] = f0.z; v[3] = f0.w; v[4] = f1.x; v[5] = f1.y; v[6] = f1.z; v[7] = f1.w;
        v[8] = f2.x; v[9] = f2.y; v[10] = f2.z; v[11] = f2.w; v[12] = f3.x; v[13] = f3.y; v[14] = f3.z; v[15] = f3.w;
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.f;
      }
#pragma unroll
      for (int term = 0; term < NT; ++term) {  // each term stored as soon as it is split
        uint2 packed;
        uint32_t sc;
        mx::split_half_block_e2m1_term(v, term + 1 == NT, pair, packed, sc);
        *reinterpret_cast<uint2*>(chunk + (size_t)term * kTermBytes) = packed;
        if (hf == 0) {
          int n;
          const int ai = atom_index(term, m, g.rn, r, n);
          atoms[(size_t)ai * kAtom + dmx::atom_off(n, kb)] = (uint8_t)sc;
        }
      }
    }
  }
  if (GATHER && y) {
    const int64_t n4 = (int64_t)T * C / 4;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
    float4* y4 = reinterpret_cast<float4*>(y);
    for (int64_t i = tid; i < n4; i += nthr) y4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t i = 4 * n4 + tid; i < (int64_t)T * C; i += nthr) y[i] = 0.f;
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");  // read next by the copy engine
}

}  // namespace gx4

size_t prefill_operand_bytes(int max_rows, int C, int terms) {
  return (size_t)(max_rows / 128) * ((C + 127) / 128) * terms * gx4::kTermBytes;
}
size_t prefill_atom_bytes(int max_rows, int C, int terms) {
  return (size_t)(max_rows / 128) * ((C + 127) / 128) * 2 * terms * gx4::kAtom;
}

namespace {
// Blocks of the row quantiser; 0 when its 32-bit item index would overflow.
// Blocks for the row quantisers: one thread per item of the h operand, at
// most eight blocks per SM (about three are resident; later waves hide the
// per-item load and split latency better than longer grid-stride loops).
int quant_blocks(int max_rows, int C) {
  const int64_t threads = (int64_t)max_rows * 4 * ((C + 127) / 128);
  if (threads > 0x7fffffffLL) return 0;
  int64_t blocks = (threads + 255) / 256;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}
}  // namespace

cudaError_t launch_quant_rows_e2m1(const float* x, int T, int D, int k, const int32_t* rows, const int32_t* inv,
                                   const int32_t* counts, const int32_t* basep, int E, int max_rows, uint8_t* aq,
                                   uint8_t* asf, float* y, int2* segs, int* ctr, int* status, Launch L) {
  const auto kern = gx4::quant_rows_e2m1_kernel<kPrefillXTerms, true>;
  const int blocks = quant_blocks(2 * max_rows, D);  // a lane pair per item
  if (blocks == 0) return cudaErrorInvalidValue;
  return launch_kernel(kern, dim3(blocks), dim3(256),
                       (size_t)(max_rows / 128) * sizeof(int), L, x, T, D, k, rows, counts, basep, E, (D + 127) / 128, aq,
                       asf, y, segs, inv, ctr, status);
}

cudaError_t launch_quant_h_e2m1(const float* hf, int F, const int32_t* rows, const int32_t* counts,
                                const int32_t* basep, int E, int max_rows, uint8_t* hq, uint8_t* hsf, int* status,
                                Launch L) {
  const auto kern = gx4::quant_rows_e2m1_kernel<kPrefillHTerms, false>;
  const int blocks = quant_blocks(2 * max_rows, F);  // a lane pair per item
  if (blocks == 0) return cudaErrorInvalidValue;
  return launch_kernel(kern, dim3(blocks), dim3(256),
                       (size_t)(max_rows / 128) * sizeof(int), L, hf, 0, F, 1, rows, counts, basep, E, (F + 127) / 128, hq,
                       hsf, nullptr, nullptr, nullptr, nullptr, status);
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
  prm.segs = a.segs;
  prm.ctr = a.ctr;
  prm.k = a.k;
  prm.weights = a.weights;
  prm.aq = a.aq;
  prm.asf = a.asf;
  prm.hf = a.hf;
  prm.alpha = a.alpha;
  prm.limit = a.limit;
  prm.y = a.y;
  prm.ny = a.ny;
  prm.status = a.status;
  const int nunits = prm.ntiles * 2 * prm.npair;
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
