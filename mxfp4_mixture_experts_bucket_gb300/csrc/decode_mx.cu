// Decode rail on the block-scaled tensor cores (T <= 8 tokens, prepacked
// MXFP4 weights): the fused routed-expert chain of "dasLLAMA gpt-oss arc"
// (fused MoE expert chain commit: stage 0 = gate+up rows + bias + activation,
// stage 1 = down rows + bias + router-weighted sum) as two kernels after the
// decode prologue (router logits and the x operand).
//
// The MXFP4 weights enter tcgen05.mma kind::mxf4.block_scale as stored: the
// E2M1 codes (prepacked so that each 128-row tile arrives with one contiguous
// bulk copy as the 64-byte-swizzled image the MMA reads) and their E8M0 bytes (one 512-byte
// atom per tile and 128 columns, written into tensor memory by the epilogue
// warps while they wait for their accumulators),
// so no weight is decoded by a thread; the
// routed-expert GEMV of "dasLLAMA: dig the last two board reds green" (section
// "gpt-oss: mx4 kernels to the lab-winning shape") becomes a 128-row MMA whose
// N columns are the tokens' activation terms. Each activation is a sum of
// kDecTerms E2M1 terms, each block of 32 on its own E8M0 scale (the MXFP4
// format itself; eight terms leave ~1e-7 of the block's largest value), and
// the products accumulate in fp32 in tensor memory.
//
// Work split: the weight tiles of the routed experts are cut into steps of one
// 128-row x 128-K tile (gate/up: both matrices) and the steps are dealt out in
// equal contiguous ranges to every CTA of the grid, across tile boundaries, so
// all SMs stream the same number of bytes. A tile whose steps span several
// CTAs is finished by the last CTA to arrive: each writes its partial sums,
// bumps the tile's counter, and the last one adds the partials in CTA order
// (deterministic) and runs the epilogue. Nothing ever waits for another CTA.
//   gate/up unit = (routed expert, 128-row tile of F); epilogue: bias, swiglu_oai,
//     the router weight, and the down operand: w*h as E2M1 terms, written in
//     the operand-chunk layout of decode_mx.cuh (one chunk per tile).
//   down unit = 128-row tile of D, steps over (routed expert, chunk of F): all
//     experts of a token accumulate into the same columns (w is folded into the
//     operand), epilogue: + sum_j w_j bd[e_j] in slot order, y stored.
//
// Warps: 0..5 = producers (warp 0 also builds the routing table), 6 = MMA
// issuer, 7..10 = scale loaders and epilogue (one per tensor-memory lane
// quarter; warp 7 also allocates and frees tensor memory). The scale atoms go from shared memory into
// tensor memory through the epilogue warps' registers (tcgen05.st): a
// tcgen05.cp would take ~80 tensor-pipe cycles per atom, and a step's six
// atoms cost as much pipe time as its eight MMAs (measured). The copy engine serves the bulk copies one issuing thread makes in
// order, each taking at least ~0.4 us (measured), so every copy of a step has
// a producer warp of its own and the weight copies are large (two 128-column
// chunks of a 128-row tile, 16 KB): each warp walks all steps in order and
// issues its one copy, which also keeps every barrier wait in phase.
// (Tiled tensor copies of 64-byte rows were measured at about 22 GB/s per SM;
// contiguous bulk copies from several warps reach the HBM rate.)
#include <cuda.h>

#include "decode_mx.cuh"
#include "decode_routing.cuh"
#include "mx_terms.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace dmx {

constexpr int kProd = 6;  // producer warps 0..5, one copy of each step apiece
constexpr int kMmaWarp = 6;
constexpr int kTmemWarp = 7;  // the first epilogue warp allocates and frees tensor memory
constexpr int kThreads = 11 * 32;
constexpr int kMaxStages = 6;
constexpr int kMaxAccSlots = 4;
constexpr int kScaleBatch = 4;  // steps whose scales one tensor-memory store wait covers (< stages)
constexpr int kATile = 8192;    // one 128-row x 128-column tile of E2M1 codes (64 bytes a row)
constexpr int kAtom = 512;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDynSmem = 222 * 1024;

struct Params {
  int E, R, C, NK, NT;  // matrices [R][C]; NK chunks of 128 along C, NT tiles of 128 rows
  int T, k, npad;
  int SC;               // chunks per step
  int acc_slots;        // tensor-memory accumulators (a unit each), 2 or 4
  const uint8_t* a_qs[2];  // prepacked planes
  const uint8_t* a_sf[2];
  const float* bias[2];
  const uint8_t* b_q;   // activation chunks: gate/up x [NK][npad*64]; down w*h [T*k][NK][npad*64]
  const uint8_t* b_sf;  // gate/up: [NK][512]; down: [T*k][NK][512]
  const float* logits;
  int32_t* ids_out;
  float* w_out;
  float alpha, limit;
  uint8_t* hq;    // gate/up: down operand chunks [T*k][NT][npad][64]
  uint8_t* hsf;   // gate/up: [T*k][NT][512]
  float* h_out;   // gate/up, optional: swiglu outputs [T*k][R]
  float* y;       // down: [T][R]
  float* part;    // [grid][2][NMAT][T][128]
  int* cnt;       // arrival counter per unit and lane quarter (zeroed by the prologue, reset after use)
  int* status;
  int nstages;
  uint32_t stage_bytes, off_b, off_sfa, off_sfb;
};

// Instruction descriptor of tcgen05.mma kind::mxf4: A and B E2M1, E8M0 scales, M x N.
__device__ __forceinline__ uint32_t idesc_mxf4(int M, int N) {
  return (1u << 7)                      // A: E2M1
         | (1u << 10)                   // B: E2M1
         | ((uint32_t)(N >> 3) << 17)   // N / 8
         | (1u << 23)                   // scales are E8M0
         | ((uint32_t)(M >> 4) << 24);  // M / 16
}

// K = 64 per instruction (two 32-blocks); the scale-factor id (bits 4-5 and
// 29-30 of the descriptor, 0 or 2) picks the pair of bytes of each 32-bit
// scale cell that the two blocks use.
__device__ __forceinline__ void mma_mxf4(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}

// Owner of step x when `total` steps are dealt to G CTAs in contiguous ranges
// [ceil(c*total/G), ceil((c+1)*total/G)).
__device__ __forceinline__ int step_owner(long long x, long long total, int G) { return (int)(x * G / total); }
__device__ __forceinline__ long long range_lo(int c, long long total, int G) {
  return ((long long)c * total + G - 1) / G;
}

// The accumulator columns of one unit (npad <= 64 columns per matrix), summed
// over the E2M1 terms of each token: v[t] for t < T.
__device__ __forceinline__ void load_token_sums(uint32_t taddr, int npad, int T, float (&v)[8]) {
  float col[64];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    uint32_t a[16];
    if (16 * g < npad) tc::tmem_ld16_wait(taddr + 16 * g, a);  // warp-uniform
#pragma unroll
    for (int i = 0; i < 16; ++i) col[16 * g + i] = 16 * g < npad ? __uint_as_float(a[i]) : 0.f;
  }
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < kDecTerms; ++q) s += col[t * kDecTerms + q];
    v[t] = t < T ? s : 0.f;
  }
}

// The walk over a CTA's steps: unit u, step s within it, and what the step covers.
struct StepPos {
  int u, s;
};

template <int KIND>
__device__ __forceinline__ void step_cover(const StepPos& sp, int NT, int NK, int nkc, int SC, int& ai, int& tile,
                                           int& j0, int& nch) {
  int jj;
  if (KIND == 0) {
    ai = sp.u / NT;
    tile = sp.u - ai * NT;
    jj = sp.s;
  } else {
    tile = sp.u;
    ai = sp.s / nkc;
    jj = sp.s - ai * nkc;
  }
  j0 = jj * SC;
  nch = min(SC, NK - j0);
}

// Chunks per step: gate/up two (a 16 KB copy per matrix), down four (two 16 KB copies).
template <int KIND>
__host__ __device__ constexpr int steps_chunks() { return KIND == 0 ? 2 : 4; }
// Copies of a step, one per producer warp: the weight parts (gate/up: gate, up;
// down: the two halves of the tile's chunks), the weight scale atoms (one per
// matrix), the activation chunks, the activation scale atoms.
template <int KIND>
__host__ __device__ constexpr int step_copies() { return KIND == 0 ? 6 : 5; }

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    decode_mx_kernel(const Params p) {
  constexpr int NMAT = KIND == 0 ? 2 : 1;
  constexpr int SCMAX = steps_chunks<KIND>();
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ DecodeRouting Rt;
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t sfr_bar[kMaxStages];  // a stage's scales are in tensor memory
  __shared__ __align__(8) uint64_t accf_bar[kMaxAccSlots];
  __shared__ __align__(8) uint64_t acce_bar[kMaxAccSlots];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ __align__(8) uint64_t tfree_bar;  // the epilogue warps and the MMA thread are done with tensor memory
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = p.nstages;
  const int AS = p.acc_slots;
  const int T = p.T, k = p.k, E = p.E, R = p.R;

  // The down kernel may start once every gate/up CTA has passed its wait for
  // the prologue, so the routing inputs (prologue output) are complete by then
  // and the down kernel routes, and streams its weights, before its own wait.
  if (KIND == 1) pdl_launch_dependents();
  if (warp == 1 && lane == 0) {
    for (int i = 0; i < NS; ++i) {
      tc::mbar_init(tc::smem_u32(&full_bar[i]), kProd);
      tc::mbar_init(tc::smem_u32(&empty_bar[i]), 1);
      tc::mbar_init(tc::smem_u32(&sfr_bar[i]), 4);
    }
    for (int i = 0; i < AS; ++i) {
      tc::mbar_init(tc::smem_u32(&accf_bar[i]), 1);
      tc::mbar_init(tc::smem_u32(&acce_bar[i]), 4);
    }
    tc::mbar_init(tc::smem_u32(&drain_bar), 1);
    tc::mbar_init(tc::smem_u32(&tfree_bar), 5);
    s_abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == kTmemWarp) tc::tmem_alloc(tc::smem_u32(&s_tmem), kTmemCols);
  if (KIND == 0) {
    pdl_wait();  // logits, the activation operand and the zeroed counters come from the prologue
    pdl_launch_dependents();
  }
  if (warp == 0) {
    routing_inputs(Rt, T, k, E, lane, p.logits, nullptr, nullptr);
    build_routing(Rt, T * k, E, lane, KIND == 0 ? p.status : nullptr);
    if (KIND == 0 && blockIdx.x == 0 && p.ids_out)
      for (int a = lane; a < T * k; a += 32) {
        p.ids_out[a] = Rt.ids[a];
        if (p.w_out) p.w_out[a] = Rt.w[a];
      }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  const int nact = Rt.nact;
  const int NK = p.NK, NT = p.NT;
  constexpr int SC = SCMAX;  // the host planned the stages with the same count
  const int nkc = (NK + SC - 1) / SC;                          // steps along K
  const long long spu = KIND == 0 ? nkc : (long long)nact * nkc;  // steps per unit
  const long long nunits = KIND == 0 ? (long long)nact * NT : NT;
  const long long total = spu * nunits;
  const int G = (int)(total < (long long)gridDim.x ? total : (long long)gridDim.x);
  const int cta = blockIdx.x;
  const volatile int* abort_flag = &s_abort;
  const uint32_t acc_cols = (uint32_t)(NMAT * p.npad);
  const uint32_t sf0 = AS * acc_cols;
  const uint32_t sf_chunk = 4 * (NMAT + 1), sfw = (uint32_t)SC * sf_chunk;

  if (total == 0) {
    // no valid assignment: y = 0 (the down kernel owes it, after the gate/up
    // kernel, so that the grid still ends after its predecessor)
    if (KIND == 1) pdl_wait();
    if (KIND == 1)
      for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < T * R; i += gridDim.x * blockDim.x) p.y[i] = 0.f;
  } else if (cta < G) {
    const long long lo = range_lo(cta, total, G), hi = range_lo(cta + 1, total, G);
    const int nsteps = (int)(hi - lo);
    const StepPos sp0 = {(int)(lo / spu), (int)(lo % spu)};
    auto advance = [&](StepPos& sp) {
      if (++sp.s == spu) {
        sp.s = 0;
        ++sp.u;
      }
    };
    auto fail = [&](int role, int seq) {
      s_abort = 1;
      report_timeout(p.status, 5 + KIND, role, 0, seq);
    };

    // Down kernel: the weight producers (warps 0 .. 1 + NMAT) stream before the
    // gate/up kernel has finished; every other role reads its output (the
    // activation operand) or follows those that do.
    if (KIND == 1 && warp >= 2 + NMAT) pdl_wait();
    if (warp < kProd) {
      // ------------------------------------------------ producers
      if (lane == 0) {
        const uint64_t pol = tc::l2_policy_evict_first();
        StepPos sp = sp0;
        int issued = 0;
        for (int i = 0; i < nsteps; ++i, advance(sp)) {
          const int st = i % NS, n = i / NS;
          if (n > 0 && !tc::mbar_wait_sleep(tc::smem_u32(&empty_bar[st]), (n - 1) & 1, abort_flag, 32)) {
            fail(0, i);
            break;
          }
          int ai, tile, j0, nch;
          step_cover<KIND>(sp, NT, NK, nkc, SC, ai, tile, j0, nch);
          const int e = Rt.act_e[ai];
          const uint32_t fb = tc::smem_u32(&full_bar[st]);
          const uint32_t sb = tc::smem_u32(smem) + (uint32_t)st * p.stage_bytes;
          const size_t bi = KIND == 0 ? (size_t)j0 : (size_t)ai * NK + j0;
          // copy c of the step goes to producer warp c % kProd: A boxes, A scale atoms, B chunks, B atoms
          // (the boxes count in full: chunks past NK are zero-filled)
          // the weight chunks j0 .. j0+nch-1 of the tile: rows_t * 64 bytes per chunk
          const int rows_t = min(128, R - 128 * tile);
          const size_t a_off = ((size_t)e * R + 128 * (size_t)tile) * ((size_t)NK * 64) + (size_t)rows_t * 64 * j0;
          const int c = warp;  // this warp's copy of the step
          uint32_t dst = 0, bytes = 0;
          const uint8_t* src = nullptr;
          bool stream = true;
          if (KIND == 0 && c < 2) {  // gate or up chunks
            bytes = (uint32_t)(rows_t * 64 * nch);
            dst = sb + c * SC * kATile;
            src = p.a_qs[c] + a_off;
          } else if (KIND == 1 && c < 2) {  // down chunks, in two halves of SC/2 chunks
            const int h0 = c * (SC / 2), hn = min(SC / 2, nch - h0);
            if (hn > 0) {
              bytes = (uint32_t)(rows_t * 64 * hn);
              dst = sb + (uint32_t)(rows_t * 64 * h0);
              src = p.a_qs[0] + a_off + (size_t)rows_t * 64 * h0;
            }
          } else if (c < 2 + NMAT) {  // weight scale atoms
            const int m = c - 2;
            bytes = (uint32_t)(nch * kAtom);
            dst = sb + p.off_sfa + m * SC * kAtom;
            src = p.a_sf[m] + (((size_t)e * NT + tile) * NK + j0) * kAtom;
          } else if (c == 2 + NMAT) {  // activation chunks
            bytes = (uint32_t)(nch * p.npad * 64);
            dst = sb + p.off_b;
            src = p.b_q + bi * p.npad * 64;
            stream = false;
          } else if (c == 3 + NMAT) {  // activation scale atoms
            bytes = (uint32_t)(nch * kAtom);
            dst = sb + p.off_sfb;
            src = p.b_sf + bi * kAtom;
            stream = false;
          }
          tc::mbar_expect_tx(fb, bytes);  // a warp without a copy this step still arrives
          if (bytes) {
            if (stream) tc::bulk_load_stream(dst, src, bytes, fb, pol);
            else tc::bulk_load(dst, src, bytes, fb);
          }
          issued = i + 1;
        }
        if (*abort_flag) {  // every copy already issued lands before shared memory goes away
          for (int st = 0; st < NS; ++st) {
            const int n = issued > st ? (issued - 1 - st) / NS + 1 : 0;
            if (n > 0) tc::mbar_wait(tc::smem_u32(&full_bar[st]), (n - 1) & 1, nullptr);
          }
        }
      }
    } else if (warp == kMmaWarp) {
      // ------------------------------------------------ MMA issuer
      if (lane == 0) {
        const uint32_t idesc = idesc_mxf4(128, p.npad);
        const int nbc = p.C / 32;
        StepPos sp = sp0;
        int lu = -1;
        for (int i = 0; i < nsteps; ++i, advance(sp)) {
          const int st = i % NS, n = i / NS;
          const bool first = (i == 0) || (sp.s == 0);
          const bool last = (i == nsteps - 1) || (sp.s == spu - 1);
          if (first) {
            ++lu;
            if (lu >= AS &&
                !tc::mbar_wait(tc::smem_u32(&acce_bar[lu % AS]), ((lu / AS) - 1) & 1, abort_flag)) {
              fail(1, i);
              break;
            }
          }
          // the stage's data has landed and its scales are in tensor memory
          if (!tc::mbar_wait(tc::smem_u32(&sfr_bar[st]), n & 1, abort_flag)) {
            fail(1, i);
            break;
          }
          tc::fence_after_sync();
          int ai, tile, j0, nch;
          step_cover<KIND>(sp, NT, NK, nkc, SC, ai, tile, j0, nch);
          const int slot = lu % AS;
          const uint32_t sb = tc::smem_u32(smem) + (uint32_t)st * p.stage_bytes;
          const uint32_t sfs = tmem + sf0 + (uint32_t)st * sfw;
          // 64-byte-swizzled operands; a chunk's K halves are 32 bytes apart. The
          // issue loop stays compact (one K half of every matrix per pass, the
          // descriptors advanced by adding to their start-address field, which
          // holds shared-memory address / 16 and cannot carry out of its 14
          // bits below 256 KB).
          const int rows_t = min(128, R - 128 * tile);
          const uint32_t dacc = tmem + (uint32_t)slot * acc_cols;
          const int nkb_last = min(4, nbc - 4 * (j0 + nch - 1));  // even: widths are multiples of 64
          const int nkh = 2 * (nch - 1) + nkb_last / 2;
          const uint64_t adesc0 = tc::sw64_kmajor_desc(sb);
          const uint64_t bdesc0 = tc::sw64_kmajor_desc(sb + p.off_b);
          const uint32_t a_c16 = (uint32_t)(rows_t * 64) >> 4, b_c16 = (uint32_t)(p.npad * 64) >> 4;
          constexpr uint32_t kAMat16 = (uint32_t)(SCMAX * kATile) >> 4;
#pragma unroll 1
          for (int x = 0; x < nkh; ++x) {
            const uint32_t c = (uint32_t)x >> 1, kh = (uint32_t)x & 1u;
            const uint64_t ad = adesc0 + (c * a_c16 + 2u * kh);
            const uint64_t bd = bdesc0 + (c * b_c16 + 2u * kh);
            const uint32_t id = idesc | (kh ? ((2u << 4) | (2u << 29)) : 0u);  // scale bytes 2kh, 2kh+1
            const uint32_t sfc = sfs + c * sf_chunk;
            const uint32_t acc = (first && x == 0) ? 0u : 1u;
#pragma unroll
            for (int m = 0; m < NMAT; ++m)
              mma_mxf4(dacc + (uint32_t)(m * p.npad), ad + (uint64_t)(m * kAMat16), bd, id, sfc + 4 * m,
                       sfc + 4 * NMAT, acc);
          }
          tc::mma_commit(tc::smem_u32(&empty_bar[st]));
          if (last) tc::mma_commit(tc::smem_u32(&accf_bar[slot]));
        }
        // every MMA issued above completes before tensor memory is released
        tc::mma_commit(tc::smem_u32(&drain_bar));
        tc::mbar_wait(tc::smem_u32(&drain_bar), 0, nullptr);
        tc::fence_before_sync();
        tc::mbar_arrive(tc::smem_u32(&tfree_bar));
      }
    } else {
      // ------------------------------------------------ epilogue (warps 5..8)
      const int q = warp & 3;            // tensor-memory lane quarter
      const int row = 32 * q + lane;     // row of the 128-row tile
      const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
      // One loop serves both duties of these warps, in an order that cannot
      // deadlock: the scales of every step (32 rows of 16 bytes per atom, row =
      // lane, stored into the stage's tensor-memory columns of this warp's lane
      // quarter, which repeats them in all four quarters as the MMA expects), and
      // the epilogue of each unit, run once the MMA needs its accumulator slot
      // back (before the scales of the first step of unit lu + AS) or when no
      // step is left.
      const int ufirst = (int)(lo / spu);
      const int nunits_cta = (int)((hi - 1) / spu) - ufirst + 1;
      StepPos sp = sp0;
      int i = 0, lu_steps = -1, ldone = 0;
      while (ldone < nunits_cta) {
        const bool step_left = i < nsteps;
        int next_lu = lu_steps + ((step_left && (i == 0 || sp.s == 0)) ? 1 : 0);
        if (step_left && next_lu < ldone + AS) {
          // ---- the scales of step i, and of the steps after it whose data has
          // landed too (up to kScaleBatch, each allowed by the rule above): one
          // wait for the tensor-memory stores per batch
          uint32_t st_mask = 0;
          bool failed = false;
          for (int nbat = 0;;) {
            lu_steps = next_lu;
            const int st = i % NS, n = i / NS;
            if (nbat == 0) {
              bool ok = tc::mbar_wait(tc::smem_u32(&full_bar[st]), n & 1, abort_flag);
              if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) fail(3, i);
                failed = true;
                break;
              }
            }
            int ai, tile, j0, nch;
            step_cover<KIND>(sp, NT, NK, nkc, SC, ai, tile, j0, nch);
            const uint8_t* sbp = smem + (size_t)st * p.stage_bytes;
            const uint32_t sfs = lane_base + sf0 + (uint32_t)st * sfw;
#pragma unroll
            for (int c = 0; c < SCMAX; ++c)
              if (c < nch) {
#pragma unroll
                for (int m = 0; m <= NMAT; ++m) {  // weight atoms, then the activation atom
                  const uint8_t* atom = sbp + (m < NMAT ? p.off_sfa + (m * SC + c) * kAtom : p.off_sfb + c * kAtom);
                  const uint4 w = *reinterpret_cast<const uint4*>(atom + 16 * lane);
                  tc::tmem_st4(sfs + c * sf_chunk + 4 * m, w.x, w.y, w.z, w.w);
                }
              }
            st_mask |= 1u << st;
            ++i;
            advance(sp);
            if (++nbat == kScaleBatch || i >= nsteps) break;
            next_lu = lu_steps + (sp.s == 0 ? 1 : 0);
            if (next_lu >= ldone + AS) break;
            if (!__all_sync(0xffffffffu, tc::mbar_peek(tc::smem_u32(&full_bar[i % NS]), (i / NS) & 1))) break;
          }
          if (failed) break;
          tc::tmem_wait_st();
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0)
            for (int st = 0; st < NS; ++st)
              if (st_mask >> st & 1u) tc::mbar_arrive(tc::smem_u32(&sfr_bar[st]));
          continue;
        }
        // ---- the epilogue of unit ldone
        const int lu = ldone++;
        const int u = ufirst + lu;
        const long long u0 = (long long)u * spu, u1 = u0 + spu;
        const int slot = lu % AS;
        // inputs of the epilogue that do not depend on the MMAs, fetched before the wait
        float bias0 = 0.f, bias1 = 0.f;
        float bsum[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) bsum[t] = 0.f;
        if constexpr (KIND == 0) {
          const int ai = u / NT, tile = u - ai * NT, e = Rt.act_e[ai], f = tile * 128 + row;
          if (f < R) {
            if (p.bias[0]) bias0 = __ldg(p.bias[0] + (size_t)e * R + f);
            if (p.bias[1]) bias1 = __ldg(p.bias[1] + (size_t)e * R + f);
          }
        } else {
          const int c = u * 128 + row;
          if (c < R && p.bias[0]) {
#pragma unroll
            for (int t = 0; t < 8; ++t)
              if (t < T)
                for (int jj = 0; jj < k; ++jj) {  // slot order
                  const int a = t * k + jj, ej = Rt.ids[a];
                  if (ej >= 0 && ej < E) bsum[t] = fmaf(Rt.w[a], __ldg(p.bias[0] + (size_t)ej * R + c), bsum[t]);
                }
          }
        }
        bool ok = tc::mbar_wait_sleep(tc::smem_u32(&accf_bar[slot]), (lu / AS) & 1, abort_flag, 256);
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) fail(2, lu);
          break;
        }
        tc::fence_after_sync();
        float v[NMAT][8];
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
          load_token_sums(lane_base + (uint32_t)slot * acc_cols + (uint32_t)(m * p.npad), p.npad, T, v[m]);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_u32(&acce_bar[slot]));

        const int cf = step_owner(u0, total, G), cl = step_owner(u1 - 1, total, G);
        if (cf != cl) {
          // Partial sums (slot 0 for the CTA's first unit, 1 for its last). Each
          // warp arrives on its own lane quarter's counter and the last warp of a
          // quarter to arrive finishes those 32 rows: no warp waits for another.
          const int ps = (u == ufirst) ? 0 : 1;
          float* pp = p.part + (size_t)(cta * 2 + ps) * NMAT * T * 128;
#pragma unroll
          for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int t = 0; t < 8; ++t)
              if (t < T) pp[(m * T + t) * 128 + row] = v[m][t];
          __threadfence();
          __syncwarp();
          int last = 0;
          if (lane == 0) last = (atomicAdd(p.cnt + 4 * u + q, 1) == cl - cf) ? 1 : 0;
          if (__shfl_sync(0xffffffffu, last, 0) == 0) continue;
          __threadfence();
          if (lane == 0) p.cnt[4 * u + q] = 0;  // every contributor has arrived: ready for the next call
#pragma unroll
          for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int t = 0; t < 8; ++t) v[m][t] = 0.f;
          // the partials of PB CTAs are loaded together, then added in CTA order
          constexpr int PB = KIND == 0 ? 2 : 4;
          for (int c0 = cf; c0 <= cl; c0 += PB) {
            float pv[PB][NMAT][8];
#pragma unroll
            for (int b = 0; b < PB; ++b) {
              const int cc = c0 + b;
              const float* src = nullptr;
              if (cc <= cl) {
                const int pc = (u == (int)(range_lo(cc, total, G) / spu)) ? 0 : 1;
                src = p.part + (size_t)(cc * 2 + pc) * NMAT * T * 128;
              }
#pragma unroll
              for (int m = 0; m < NMAT; ++m)
#pragma unroll
                for (int t = 0; t < 8; ++t) pv[b][m][t] = (src && t < T) ? __ldcg(src + (m * T + t) * 128 + row) : 0.f;
            }
#pragma unroll
            for (int b = 0; b < PB; ++b)
#pragma unroll
              for (int m = 0; m < NMAT; ++m)
#pragma unroll
                for (int t = 0; t < 8; ++t) v[m][t] += pv[b][m][t];
          }
        }

        if constexpr (KIND == 0) {
          // ---- gate/up: bias, swiglu, router weight, down operand chunk
          const int ai = u / NT, tile = u - ai * NT;
          const int e = Rt.act_e[ai];
          const int f = tile * 128 + row;
          const bool valid = f < R;
          uint8_t* chunk = p.hq + ((size_t)ai * NT + tile) * p.npad * 64;
          uint8_t* atom = p.hsf + ((size_t)ai * NT + tile) * kAtom;
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            if (t < T) {  // warp-uniform
              int slot_j = -1;
              for (int jj = 0; jj < k; ++jj)
                if (Rt.ids[t * k + jj] == e) slot_j = jj;
              float hw = 0.f;
              if (slot_j >= 0 && valid) {
                const float h = swiglu_oai_f(v[0][t] + bias0, v[1][t] + bias1, p.alpha, p.limit);
                if (p.h_out) p.h_out[(size_t)(t * k + slot_j) * R + f] = h;
                hw = h * Rt.w[t * k + slot_j];
              }
              uint32_t qv[kDecTerms], sv[kDecTerms];
              mx::split_terms_e2m1<kDecTerms>(hw, qv, sv);
#pragma unroll
              for (int term = 0; term < kDecTerms; ++term) {
                const int n = t * kDecTerms + term;
                const uint32_t byte = mx::pack_e2m1_block(qv[term]);
                if (lane < 16) chunk[chunk_off(n, q, lane)] = (uint8_t)byte;
                if (lane == 0) atom[atom_off(n, q)] = (uint8_t)sv[term];
              }
            }
          }
          for (int n = T * kDecTerms; n < p.npad; ++n) {  // rows past the tokens' terms: zero on a scale of 1
            if (lane < 4) reinterpret_cast<uint32_t*>(chunk + chunk_off(n, q, 0))[lane] = 0u;
            if (lane == 0) atom[atom_off(n, q)] = 127;
          }
        } else {
          // ---- down: + sum_j w_j bd[e_j] in slot order, y stored
          const int c = u * 128 + row;
          if (c < R) {
#pragma unroll
            for (int t = 0; t < 8; ++t)
              if (t < T) p.y[(size_t)t * R + c] = v[0][t] + bsum[t];
          }
        }
      }
      tc::fence_before_sync();  // this warp's tensor-memory reads are complete
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tc::smem_u32(&tfree_bar));
      // the down operand written above is read next by the copy engine
      if (KIND == 0) asm volatile("fence.proxy.async.global;" ::: "memory");
    }
  }

  // Tensor memory goes back when the epilogue warps and the MMA thread have
  // arrived on an mbarrier, freed by warp kTmemWarp, whose code is warp-uniform
  // throughout. (No CTA-wide barrier here: it would also count warps whose lane
  // 0 is still in its role loop.) Shared memory lives until every thread has
  // exited, and every copy issued has landed by then: each is consumed by the
  // MMAs, or waited for by its producer on abort.
  if (warp == kTmemWarp) {
    if (total > 0 && cta < G) tc::mbar_wait_sleep(tc::smem_u32(&tfree_bar), 0, nullptr, 64);
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace dmx

cudaError_t launch_decode_mx(const DecodeMXArgs& a, Launch L) {
  using namespace dmx;
  const int nmat = a.kind == 0 ? 2 : 1;
  if (a.T < 1 || a.T > 8 || a.T * a.k > kMaxAssign || a.R % 64 != 0 || a.C % 64 != 0) return cudaErrorInvalidValue;
  Params prm{};
  prm.E = a.E;
  prm.R = a.R;
  prm.C = a.C;
  prm.NK = (a.C + 127) / 128;
  prm.NT = (a.R + 127) / 128;
  prm.T = a.T;
  prm.k = a.k;
  prm.npad = npad_for(a.T);
  for (int m = 0; m < 2; ++m) {
    prm.a_qs[m] = a.w_qs[m];
    prm.a_sf[m] = a.w_sf[m];
    prm.bias[m] = a.bias[m];
  }
  prm.b_q = a.b_q;
  prm.b_sf = a.b_sf;
  prm.logits = a.logits;
  prm.ids_out = a.ids_out;
  prm.w_out = a.w_out;
  prm.alpha = a.alpha;
  prm.limit = a.limit;
  prm.hq = a.hq;
  prm.hsf = a.hsf;
  prm.h_out = a.h_out;
  prm.y = a.y;
  prm.part = a.part;
  prm.cnt = a.cnt;
  prm.status = a.status;
  // A step is SC chunks of a 128-row tile: one weight copy of up to SC * 8 KB per
  // matrix. Gate/up: 2 chunks (two 16 KB copies a step); down: 4 chunks (one 32 KB copy).
  const int sc = a.kind == 0 ? steps_chunks<0>() : steps_chunks<1>();
  prm.SC = sc;
  prm.off_b = (uint32_t)(nmat * sc * kATile);
  prm.off_sfa = prm.off_b + (uint32_t)(sc * prm.npad * 64);
  prm.off_sfb = prm.off_sfa + (uint32_t)(nmat * sc * kAtom);
  prm.stage_bytes = (prm.off_sfb + (uint32_t)(sc * kAtom) + 1023u) & ~1023u;
  int ns = (int)((kDynSmem - 1024) / prm.stage_bytes);
  if (ns > kMaxStages) ns = kMaxStages;
  const int sf_cols = ns * sc * 4 * (nmat + 1);
  int slots = kMaxAccSlots;
  while (slots > 2 && slots * nmat * prm.npad + sf_cols > (int)kTmemCols) slots /= 2;
  if (ns < 2 || slots * nmat * prm.npad + sf_cols > (int)kTmemCols) return cudaErrorInvalidValue;
  prm.nstages = ns;
  prm.acc_slots = slots;
  const size_t smem = (size_t)ns * prm.stage_bytes + 1024;

  int grid = device_sm_count();
  if (grid > kDecodeMxMaxGrid) grid = kDecodeMxMaxGrid;
  if (a.kind == 0) {
    cudaError_t err = ensure_smem_limit(decode_mx_kernel<0>, smem);
    if (err != cudaSuccess) return err;
    return launch_kernel(decode_mx_kernel<0>, dim3(grid), dim3(kThreads), smem, L, prm);
  }
  cudaError_t err = ensure_smem_limit(decode_mx_kernel<1>, smem);
  if (err != cudaSuccess) return err;
  return launch_kernel(decode_mx_kernel<1>, dim3(grid), dim3(kThreads), smem, L, prm);
}

}  // namespace moe
