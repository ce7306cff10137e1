// Decode rail: the fused routed-expert chain for T <= 8 tokens, two kernels
// after the router logits.
//
// Stage 0 (gate/up + bias + swiglu) and stage 1 (down + bias + router-weighted
// combine in slot order) follow the fused decode expert chain of "dasLLAMA
// gpt-oss arc" (fused MoE expert chain commit) and the routed-expert GEMV
// MetalMoeGemvMx4 of "dasLLAMA: dig the last two board reds green" (section
// "gpt-oss: mx4 kernels to the lab-winning shape"): every weight byte of a
// touched expert is read from HBM once with wide loads, the E8M0 exponent is
// built in the ALU, products accumulate in fp32 and partial sums reduce with
// warp shuffles.
//
// GB300 organisation:
//  * One CTA per SM: a producer warp streams weight rows with TMA bulk copies
//    into a ring of shared-memory stages; twelve consumer warps form teams of
//    TW = ceil(C/1024) warps, and each lane of a team owns one 32-column MXFP4
//    block of the row (16 bytes = one 128-bit shared load per row).
//  * Gate/up with the split vectors in shared memory (always at T = 1): each
//    warp of a team takes a third of the row's blocks and runs the products on
//    the tensor pipe, mma.sync m16n8k16 with the sub-task's 8 gate and 8 up
//    rows (decoded to f16 by the hardware conversion) as A and up to four
//    tokens' high and low f16 parts as the B columns; each block's two k16
//    products are scaled by the activation and weight block factors and added
//    in fp32, and the team adds its warps' partials.
//  * Otherwise (and always in the down kernel, whose 8-row sub-tasks would
//    leave half of each m16 product unused) the CUDA cores:
//    the input vector's block stays in the lane's registers, split into f16
//    high and low parts under a power-of-two block factor. The E2M1 pairs go
//    through the hardware e2m1x2 -> f16x2 conversion and meet the high part in
//    mixed-precision f16 x f16 + f32 FMAs (no f16 -> f32 conversions, which run
//    at half rate on sm_103a), the low part in packed f16 FMAs. Products of
//    the high part are exact in fp32; the low part carries the vector's bits
//    beyond f16 (22 significant bits in all), so results match an fp32 GEMV to
//    well under the 1e-4 decode tolerance.
//  * Work is split evenly: every team of every CTA is a worker with a
//    contiguous range of rows, cut into sub-tasks of at most kDecRows rows per
//    matrix; each team owns its stages, so a stage is only ever waited on by
//    the team that consumed its previous fills.
//  * The weight streams carry an L2 evict-first hint: they are read once, and
//    must not push out code, activations and tables that the next kernels use.
#include "decode_routing.cuh"
#include "tcgen05.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Split vectors. Block b of a length-C vector v (columns 32b..32b+31) is held
// as a factor f = 2^e and 32 words: XH[i] = (hi(v[32b+i]/f), hi(v[32b+16+i]/f))
// and XL[i] = (lo(v[32b+i]/f), lo(v[32b+16+i]/f)) as f16x2 (first element in
// the low half, the order of an MXFP4 byte's nibbles), i = 0..15, with
// hi(z) = f16(z) and lo(z) = f16(z - hi(z)). e puts the block's largest
// magnitude in [128, 256), so neither part overflows or loses bits to f16
// subnormals except for elements 2^-22 below the block's largest.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int split_exponent(float absmax) {
  const int ex = (int)(__float_as_uint(absmax) >> 23);  // absmax >= 0: no sign bit
  if (ex == 255) return 0;                                // inf / NaN: propagate unscaled
  if (ex == 0) return absmax == 0.f ? 0 : -126;
  int e = ex - 127 - 7;
  return e < -126 ? -126 : e;
}
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

__device__ __forceinline__ void split_pair(float a, float b, uint32_t& xh, uint32_t& xl) {
  const __half2 hi = __floats2half2_rn(a, b);
  const float2 back = __half22float2(hi);
  const __half2 lo = __floats2half2_rn(a - back.x, b - back.y);
  xh = *reinterpret_cast<const uint32_t*>(&hi);
  xl = *reinterpret_cast<const uint32_t*>(&lo);
}

// One lane splits block b of a vector in global memory (32 floats from src,
// 16-byte aligned; read through L2).
__device__ __forceinline__ void split_block_lane(const float* __restrict__ src, uint32_t (&XH)[16],
                                                 uint32_t (&XL)[16], float& xf) {
  float z[32];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(src) + c);
    z[4 * c + 0] = v.x;
    z[4 * c + 1] = v.y;
    z[4 * c + 2] = v.z;
    z[4 * c + 3] = v.w;
  }
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) m = fmaxf(m, fabsf(z[i]));
  const int e = split_exponent(m);
  const float inv = pow2f(-e);
  xf = pow2f(e);
#pragma unroll
  for (int i = 0; i < 16; ++i) split_pair(z[i] * inv, z[i + 16] * inv, XH[i], XL[i]);
}

// Shared-memory copy of split vectors: block (v, b) is 8 chunks of 16 bytes
// (words 4c..4c+3; XH = words 0..15, XL = words 16..31), chunk c stored at
// position c ^ (b & 7) so that eight lanes reading eight consecutive blocks hit
// distinct banks; factors in a separate float array. Threads [0, nthr) (index
// t) take float4 pieces, an aligned group of eight lanes per block, with four
// pieces in flight per thread.
__device__ __forceinline__ void stage_split_vectors(const float* __restrict__ src, int nvec, int C,
                                                    uint32_t* __restrict__ words,
                                                    float* __restrict__ fac, int t, int nthr) {
  const int nb = C >> 5;
  const int total = nvec * nb * 8;  // float4 pieces
  const int q = t & 7;              // piece within the block
  constexpr int U = 4;
  for (int p0 = t - (t & 31); p0 < total; p0 += U * nthr) {  // warp-uniform bound
    float4 z[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int p = p0 + (t & 31) + u * nthr;
      z[u] = p < total ? __ldcg(reinterpret_cast<const float4*>(src) + p) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int p = p0 + (t & 31) + u * nthr;
      float m = fmaxf(fmaxf(fabsf(z[u].x), fabsf(z[u].y)), fmaxf(fabsf(z[u].z), fabsf(z[u].w)));
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      const int e = split_exponent(m);
      const float inv = pow2f(-e);
      const float4 zs = make_float4(z[u].x * inv, z[u].y * inv, z[u].z * inv, z[u].w * inv);
      float4 zp;  // lane q < 4 gets the piece of q + 4: elements 16 + 4q .. 16 + 4q + 3
      zp.x = __shfl_down_sync(0xffffffffu, zs.x, 4);
      zp.y = __shfl_down_sync(0xffffffffu, zs.y, 4);
      zp.z = __shfl_down_sync(0xffffffffu, zs.z, 4);
      zp.w = __shfl_down_sync(0xffffffffu, zs.w, 4);
      if (p < total && q < 4) {
        const int vb = p >> 3, bb = vb % nb, sw = bb & 7;
        uint4 xh, xl;
        split_pair(zs.x, zp.x, xh.x, xl.x);
        split_pair(zs.y, zp.y, xh.y, xl.y);
        split_pair(zs.z, zp.z, xh.z, xl.z);
        split_pair(zs.w, zp.w, xh.w, xl.w);
        uint4* blk = reinterpret_cast<uint4*>(words + (size_t)vb * 32);
        blk[q ^ sw] = xh;
        blk[(4 + q) ^ sw] = xl;
        if (q == 0) fac[vb] = pow2f(e);
      }
    }
  }
}

__device__ __forceinline__ void load_split_smem(const uint32_t* __restrict__ words,
                                                const float* __restrict__ fac, int vb, int b,
                                                uint32_t (&XH)[16], uint32_t (&XL)[16], float& xf) {
  const uint4* blk = reinterpret_cast<const uint4*>(words + (size_t)vb * 32);
  const int sw = b & 7;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 q = blk[c ^ sw];
    uint32_t* dst = (c < 4) ? &XH[4 * c] : &XL[4 * (c - 4)];
    dst[0] = q.x;
    dst[1] = q.y;
    dst[2] = q.z;
    dst[3] = q.w;
  }
  xf = fac[vb];
}

// ---------------------------------------------------------------------------
// One MXFP4 block (16 bytes) against a split vector block: returns the sum of
// E2M1 value x (v/f) over the 32 columns, without the E8M0 scale.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mix_fma2(uint32_t w, uint32_t x, float& a0, float& a1) {
  asm("{\n .reg .b16 w0, w1, x0, x1;\n mov.b32 {w0, w1}, %2;\n mov.b32 {x0, x1}, %3;\n"
      " fma.rn.f32.f16 %0, w0, x0, %0;\n fma.rn.f32.f16 %1, w1, x1, %1;\n}"
      : "+f"(a0), "+f"(a1)
      : "r"(w), "r"(x));
}
__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t hadd2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// a + both halves of an f16x2, in fp32.
__device__ __forceinline__ float add_f16x2_f32(uint32_t l, float a) {
  float d;
  asm("{\n .reg .b16 l0, l1;\n mov.b32 {l0, l1}, %1;\n add.rn.f32.f16 %0, l0, %2;\n"
      " add.rn.f32.f16 %0, l1, %0;\n}"
      : "=f"(d)
      : "r"(l), "f"(a));
  return d;
}

__device__ __forceinline__ float block_dot_split(uint4 q, const uint32_t (&XH)[16], const uint32_t (&XL)[16]) {
  const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
  float h0 = 0.f, h1 = 0.f, h2 = 0.f, h3 = 0.f;
  uint32_t lo0 = 0u, lo1 = 0u;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    uint32_t w[4];
    e2m1x8_to_f16x2x4(w4[m], w);  // byte 4m+i -> w[i] = (col 32b+4m+i, col 32b+16+4m+i)
    mix_fma2(w[0], XH[4 * m + 0], h0, h1);
    mix_fma2(w[1], XH[4 * m + 1], h2, h3);
    mix_fma2(w[2], XH[4 * m + 2], h0, h1);
    mix_fma2(w[3], XH[4 * m + 3], h2, h3);
    lo0 = hfma2_u32(w[0], XL[4 * m + 0], lo0);
    lo1 = hfma2_u32(w[1], XL[4 * m + 1], lo1);
    lo0 = hfma2_u32(w[2], XL[4 * m + 2], lo0);
    lo1 = hfma2_u32(w[3], XL[4 * m + 3], lo1);
  }
  return add_f16x2_f32(hadd2_u32(lo0, lo1), (h0 + h1) + (h2 + h3));
}

// One m16n8k16 tensor-core product (f16 operands, fp32 accumulators, d += a b)
// with the register fragments of mma.sync: lane (g, q) = (lane / 4, lane % 4)
// holds A rows g and g + 8 at k = 2q, 2q + 1 (a0, a1) and k = 2q + 8, 2q + 9
// (a2, a3), B column g at the same k (b0, b1), and D rows g, g + 8 at columns
// 2q, 2q + 1.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^(s-127) with s = 0 -> 2^-127 and s = 255 -> NaN, as an fp32 bit pattern.
__device__ __forceinline__ float e8m0_scale(uint32_t s) {
  const uint32_t special = (((s + 1u) & 0xFEu) == 0u) ? 0x00400000u : 0u;
  return __uint_as_float((s << 23) | special);
}

// Sum over the warp of NV values per lane; lane l ends with the total of value
// (l >> (5 - log2 NV)). NV - 1 + 5 - log2 NV shuffles in all.
template <int NV>
__device__ __forceinline__ float transpose_reduce(float (&v)[NV], int lane) {
#pragma unroll
  for (int half = NV / 2, mask = 16; half >= 1; half >>= 1, mask >>= 1) {
    const bool upper = (lane & mask) != 0;
#pragma unroll
    for (int j = 0; j < half; ++j) {
      const float send = upper ? v[j] : v[j + half];
      const float keep = upper ? v[j + half] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
    }
  }
#pragma unroll
  for (int mask = 16 / NV; mask >= 1; mask >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], mask);
  return v[0];
}

// ---------------------------------------------------------------------------
// Kernel arguments and the sub-task walk shared by producer and consumers.
// ---------------------------------------------------------------------------
constexpr int kDecConsumers = 12;
constexpr int kDecThreads = (kDecConsumers + 1) * 32;
constexpr int kDecMaxStages = 48;
constexpr int kDecRows = 8;  // rows per matrix per sub-task

struct DecodeArgs {
  const uint8_t* qs[2];
  const uint8_t* sc[2];
  const float* bias[2];
  int E, R, C;  // per-expert matrices [R][C]: gate/up R = F, C = D; down R = D, C = F
  int T, k;
  const float* vec;  // gate/up: x [T][D]; down: h [T*k][F]
  const float* logits;
  const int32_t* ids_in;
  const float* w_in;
  int32_t* ids_out;
  float* w_out;
  float alpha, limit;
  float* out;  // gate/up: h [T*k][F]; down: y [T][D]
  int tw;      // warps per team
  int spt;     // stages per team
  int staged;  // vectors split into shared memory once per CTA
  int vec_wait;  // gate/up: x is written by the previous kernel (read it after the wait)
  int rs;        // gate/up rows: 1 = separate planes; 2 = one plane, rows interleaved (gate f = row 2f,
                 // up f = row 2f+1; qs[1], sc[1], bias[1] point one row or one element further)
  uint32_t stage_bytes;
  int* status;
};

// Bytes of one matrix's slice of a stage: kDecRows rows of nibbles, then an
// E8M0 window of kDecRows rows rounded out to 16-byte bounds.
__host__ __device__ __forceinline__ uint32_t dec_qs_bytes(int C) { return (uint32_t)kDecRows * (C / 2); }
__host__ __device__ __forceinline__ uint32_t dec_sc_bytes(int C) { return (uint32_t)kDecRows * (C / 32) + 32; }

// Walk of a worker's rows. Gate/up: units are (active expert, row) pairs in
// expert-major order, a sub-task is <= kDecRows rows of one expert. Down: units
// are output rows, a chunk is <= kDecRows rows and a sub-task one active
// expert of the chunk (expert-minor order).
struct SubWalk {
  int u, u1;  // next unit, end of range
  int ai;     // down: next expert of the current chunk
};
struct SubTask {
  int ai, r0, nr;
  bool last;  // down: last expert of its chunk
};

template <int KIND>
__device__ __forceinline__ bool sub_next(SubWalk& s, int R, int nact, SubTask& t) {
  if (s.u >= s.u1) return false;
  if (KIND == 0) {
    t.ai = s.u / R;
    t.r0 = s.u - t.ai * R;
    int nr = s.u1 - s.u;
    if (nr > kDecRows) nr = kDecRows;
    if (nr > R - t.r0) nr = R - t.r0;
    t.nr = nr;
    t.last = true;
    s.u += nr;
  } else {
    t.ai = s.ai;
    t.r0 = s.u;
    int nr = s.u1 - s.u;
    if (nr > kDecRows) nr = kDecRows;
    t.nr = nr;
    t.last = (s.ai == nact - 1);
    if (t.last) {
      s.ai = 0;
      s.u += nr;
    } else {
      ++s.ai;
    }
  }
  return true;
}

template <int KIND>
__device__ __forceinline__ SubWalk sub_init(int worker, int nworkers, int R, int nact) {
  // U * (worker + 1) < 2^32: U <= 64 * 4096 units, workers <= a few thousand
  const uint32_t U = (KIND == 0) ? (uint32_t)nact * (uint32_t)R : (nact > 0 ? (uint32_t)R : 0u);
  SubWalk s;
  s.u = (int)(U * (uint32_t)worker / (uint32_t)nworkers);
  s.u1 = (int)(U * (uint32_t)(worker + 1) / (uint32_t)nworkers);
  s.ai = 0;
  return s;
}

// ---------------------------------------------------------------------------
// The two expert kernels. KIND 0: h[a][f] = swiglu(Wg[e] x_t + bg, Wu[e] x_t + bu)
// for every assignment a = t*k + j of expert e. KIND 1: y[t][c] = sum_j w[t][j]
// (Wd[e_j][c] . h[t*k+j] + bd[e_j][c]) in slot order.
// ---------------------------------------------------------------------------
template <int KIND>
__global__ void __launch_bounds__(kDecThreads, 1) decode_expert_kernel(const DecodeArgs A) {
  constexpr int NMAT = (KIND == 0) ? 2 : 1;
  constexpr int NV = NMAT * kDecRows;  // row results per lane per (sub-task, vector)
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ DecodeRouting Rt;
  __shared__ __align__(8) uint64_t full_bar[kDecMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kDecMaxStages];
  __shared__ float s_part[2][kDecConsumers][64];  // per warp: 16 row results, or 4 assignments x 8 rows x 2
  __shared__ __align__(8) uint64_t xfull_bar[kDecConsumers][2];  // per team and buffer: partials written
  __shared__ __align__(8) uint64_t xfree_bar[kDecConsumers][2];  // per team and buffer: leader done with them
  __shared__ SubWalk s_walk[kDecConsumers];
  __shared__ int s_last[kDecMaxStages];
  __shared__ int s_abort;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int C = A.C, R = A.R, T = A.T, k = A.k, E = A.E;
  const int TK = T * k;
  const int nb = C >> 5;
  const int tw = A.tw;
  const int nteams = kDecConsumers / tw;
  const int nstages = nteams * A.spt;
  const int nvec = (KIND == 0) ? T : TK;
  uint8_t* ring = dsm;
  uint32_t* vwords = reinterpret_cast<uint32_t*>(dsm + (size_t)nstages * A.stage_bytes);
  float* vfac = reinterpret_cast<float*>(vwords + (A.staged ? (size_t)nvec * nb * 32 : 0));
  float* s_o = vfac + (A.staged ? nvec * nb : 0);  // down: [team][TK][kDecRows]

  // The down kernel releases its dependents at once; the gate/up kernel only
  // after its wait for the router, so that a down kernel that starts early
  // finds the router logits complete: it routes and streams its weights
  // before its own wait (only the split vectors, h, come from gate/up).
  if (KIND == 1) pdl_launch_dependents();
  if (warp == 0) {
    if (lane == 0) {
      for (int i = 0; i < nstages; ++i) {
        tc::mbar_init(tc::smem_u32(&full_bar[i]), 1);
        tc::mbar_init(tc::smem_u32(&empty_bar[i]), tw);
        s_last[i] = -1;
      }
      for (int tm = 0; tm < nteams; ++tm)
        for (int bf = 0; bf < 2; ++bf) {
          tc::mbar_init(tc::smem_u32(&xfull_bar[tm][bf]), tw);
          tc::mbar_init(tc::smem_u32(&xfree_bar[tm][bf]), 1);
        }
      s_abort = 0;
      tc::fence_mbar_init();
    }
    if (KIND == 0 || !A.logits) pdl_wait();  // gate/up: router logits come from the previous kernel
    routing_inputs(Rt, T, k, E, lane, A.logits, A.ids_in, A.w_in);
    build_routing(Rt, TK, E, lane, KIND == 0 ? A.status : nullptr);
    if (KIND == 0 && blockIdx.x == 0 && A.ids_out)
      for (int a = lane; a < TK; a += 32) {
        A.ids_out[a] = Rt.ids[a];
        if (A.w_out) A.w_out[a] = Rt.w[a];
      }
  }
  __syncthreads();
  if (KIND == 0) pdl_launch_dependents();
  const int nact = Rt.nact;
  if (nact == 0) {
    // No valid assignment: the down kernel still owes y = 0.
    if (KIND == 1) {
      pdl_wait();
      for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < T * R; i += gridDim.x * blockDim.x)
        A.out[i] = 0.f;
    }
    return;
  }
  const int nworkers = gridDim.x * nteams;
  const volatile int* abort_flag = &s_abort;
  const uint32_t qsb = dec_qs_bytes(C), scb = dec_sc_bytes(C);

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane < nteams) s_walk[lane] = sub_init<KIND>(blockIdx.x * nteams + lane, nworkers, R, nact);
    __syncwarp();
    if (lane == 0) {
      const uint64_t stream_policy = tc::l2_policy_evict_first();
      bool any = true;
      for (int j = 0; any && !*abort_flag; ++j) {
        any = false;
        for (int tm = 0; tm < nteams; ++tm) {
          SubTask st;
          if (!sub_next<KIND>(s_walk[tm], R, nact, st)) continue;
          any = true;
          const int s = tm * A.spt + j % A.spt, n = j / A.spt;
          if (n > 0 && !tc::mbar_wait(tc::smem_u32(&empty_bar[s]), (n - 1) & 1, abort_flag)) {
            s_abort = 1;
            report_timeout(A.status, 1 + KIND, 0, s, j);
            break;
          }
          const int e = Rt.act_e[st.ai];
          const uint32_t fb = tc::smem_u32(&full_bar[s]);
          uint8_t* stage = ring + (size_t)s * A.stage_bytes;
          const size_t row0 = (size_t)e * R + st.r0;
          if (!MOE_IN_BOUNDS(A.status, e >= 0 && e < E && st.r0 >= 0 && st.nr >= 1 && st.r0 + st.nr <= R)) {
            tc::mbar_expect_tx(fb, 0);  // the stage completes without data
          } else if (KIND == 0 && A.rs == 2) {
            // interleaved gate/up: the sub-task's gate and up rows are one run of 2*nr rows,
            // one copy for the nibbles and one for the scale window
            const size_t sc0 = 2 * row0 * nb, sc1 = sc0 + 2 * (size_t)st.nr * nb;
            const size_t w0 = sc0 & ~(size_t)15, w1 = (sc1 + 15) & ~(size_t)15;
            const uint32_t qbytes = 2u * (uint32_t)st.nr * (C / 2);
            tc::mbar_expect_tx(fb, qbytes + (uint32_t)(w1 - w0));
            tc::bulk_load_stream(tc::smem_u32(stage), A.qs[0] + 2 * row0 * (C / 2), qbytes, fb, stream_policy);
            tc::bulk_load_stream(tc::smem_u32(stage + NMAT * qsb), A.sc[0] + w0, (uint32_t)(w1 - w0), fb,
                                 stream_policy);
          } else {
            const size_t sc0 = row0 * nb, sc1 = sc0 + (size_t)st.nr * nb;
            const size_t w0 = sc0 & ~(size_t)15, w1 = (sc1 + 15) & ~(size_t)15;
            const uint32_t qbytes = (uint32_t)st.nr * (C / 2);
            tc::mbar_expect_tx(fb, NMAT * (qbytes + (uint32_t)(w1 - w0)));
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
              tc::bulk_load_stream(tc::smem_u32(stage + m * qsb), A.qs[m] + row0 * (C / 2), qbytes, fb,
                                   stream_policy);
              tc::bulk_load_stream(tc::smem_u32(stage + NMAT * qsb + m * scb), A.sc[m] + w0, (uint32_t)(w1 - w0),
                                   fb, stream_policy);
            }
          }
          s_last[s] = n;
        }
      }
      // After an abort, let every copy already issued land before shared memory
      // goes away. A fill is only issued once its stage's previous fill was
      // consumed, so each stage has at most one copy in flight: its last.
      if (*abort_flag)
        for (int i = 0; i < nstages; ++i)
          if (s_last[i] >= 0) tc::mbar_wait(tc::smem_u32(&full_bar[i]), s_last[i] & 1, nullptr);
    }
    return;
  }

  // ---------------- consumers ----------------
  // x is the layer's input (unless the router copies it there); h (down) comes
  // from the previous kernel. The split vectors go to shared memory for all
  // consumer warps (a named barrier over them: the producer is already streaming).
  if (KIND == 1 || A.vec_wait) pdl_wait();
  if (A.staged) {
    stage_split_vectors(A.vec, nvec, C, vwords, vfac, threadIdx.x - 32, kDecThreads - 32);
    tc::named_sync(1, kDecThreads - 32);
  }
  const int cw = warp - 1;
  const int team = cw / tw, wt = cw - team * tw;
  if (team >= nteams) return;
  const int bpw = (nb + tw - 1) / tw;
  const int b = wt * bpw + lane;
  const bool active = lane < bpw && b < nb;
  SubWalk walk = sub_init<KIND>(blockIdx.x * nteams + team, nworkers, R, nact);
  SubTask st;
  bool dead = false;
  int it = 0;  // exchange iteration: one per (sub-task, assignment), the same for every warp of the team
  float* so = s_o + (size_t)team * TK * kDecRows;
  uint32_t XH[16], XL[16];
  float xf = 0.f;
  // Bounded wait on a team barrier; a failed wait turns this warp's remaining work into no-ops.
  auto team_wait = [&](uint64_t* bar, int parity, int site) {
    if (!dead && !tc::mbar_wait(tc::smem_u32(bar), parity, abort_flag)) {
      dead = true;
      s_abort = 1;
      report_timeout(A.status, 1 + KIND, site, team, it);
    }
  };

  for (int j = 0; sub_next<KIND>(walk, R, nact, st); ++j) {
    const int s = team * A.spt + j % A.spt, n = j / A.spt;
    const int e = Rt.act_e[st.ai];
    // biases of the sub-task's rows, in flight during the products
    float bias0 = 0.f, bias1 = 0.f;
    const int rsv = (KIND == 0) ? A.rs : 1;
    if (lane < st.nr && MOE_IN_BOUNDS(A.status, e >= 0 && e < E)) {
      const size_t ro = ((size_t)e * R + st.r0 + lane) * rsv;
      if (A.bias[0]) bias0 = __ldg(A.bias[0] + ro);
      if (KIND == 0 && A.bias[1]) bias1 = __ldg(A.bias[1] + ro);
    }
    team_wait(&full_bar[s], n & 1, 1);
    const uint8_t* stage = ring + (size_t)s * A.stage_bytes;
    const int sc_skew = (int)((((size_t)e * R + st.r0) * rsv * nb) & 15);
    // stage strides: between a matrix's consecutive rows, and between the two matrices' row r
    const uint32_t q_rs = (uint32_t)rsv * (C / 2), q_ms = rsv == 2 ? (uint32_t)(C / 2) : qsb;
    const uint32_t s_rs = (uint32_t)(rsv * nb), s_ms = rsv == 2 ? (uint32_t)nb : scb;
    if (KIND == 0 && A.staged) {
      // Tensor cores (mma.sync m16n8k16, f16 in, fp32 out): A = the sub-task's rows
      // (gate/up: gate rows 0..7, up rows 8..15; down: rows 0..7 twice), each lane
      // decoding one 32-bit word of two rows per block; B = up to four
      // assignments' split vectors (column 2j: high part of assignment j, 2j + 1:
      // its low part), read as stored; per block the two k16 products are scaled
      // by the block factors and added in fp32. This warp takes blocks
      // [kb0, kb1) of the row; the team adds its warps' partials as below.
      const int g = lane >> 2, tq = lane & 3;
      const int kbw = (nb + tw - 1) / tw, kb0 = wt * kbw, kb1 = min(nb, kb0 + kbw);
      const uint8_t* qa = stage + g * q_rs + 4 * tq;
      const uint8_t* qb = qa + (KIND == 0 ? q_ms : 0u);
      const uint8_t* sa = stage + NMAT * qsb + sc_skew + g * s_rs;
      const uint8_t* sb = sa + (KIND == 0 ? s_ms : 0u);
      // biases of the rows the leader's lanes finish: row lane % 8
      float lb0 = 0.f, lb1 = 0.f;
      if ((lane & 7) < st.nr && MOE_IN_BOUNDS(A.status, e >= 0 && e < E)) {
        const size_t ro = ((size_t)e * R + st.r0 + (lane & 7)) * rsv;
        if (A.bias[0]) lb0 = __ldg(A.bias[0] + ro);
        if (KIND == 0 && A.bias[1]) lb1 = __ldg(A.bias[1] + ro);
      }
      const int l0 = Rt.act_off[st.ai], nas = Rt.act_off[st.ai + 1] - l0;
      for (int g0 = 0; g0 < nas; g0 += 4, ++it) {
        const int ng = min(4, nas - g0);
        const int ab = Rt.lst[l0 + g0 + ((g >> 1) < ng ? (g >> 1) : 0)];  // this lane's B column
        const int ac = Rt.lst[l0 + g0 + (tq < ng ? tq : 0)];              // its D columns
        const uint32_t* xw = vwords + (size_t)((KIND == 0) ? ab / k : ab) * nb * 32;
        const int cx = 4 * (g & 1) + tq;  // the 16-byte piece: high (g even) or low words 4q .. 4q + 3
        const float* xfa = vfac + (size_t)((KIND == 0) ? ac / k : ac) * nb;
        float acc0 = 0.f, acc1 = 0.f;
        if (!__any_sync(0xffffffffu, dead)) {  // mma.sync wants the whole warp
#pragma unroll 2
          for (int blk = kb0; blk < kb1; ++blk) {
            uint32_t ha[4], hb[4];
            e2m1x8_to_f16x2x4(*reinterpret_cast<const uint32_t*>(qa + 16 * blk), ha);
            if (KIND == 0) e2m1x8_to_f16x2x4(*reinterpret_cast<const uint32_t*>(qb + 16 * blk), hb);
            const uint4 xq = *reinterpret_cast<const uint4*>(xw + 32 * blk + 4 * (cx ^ (blk & 7)));
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            if (KIND == 0) {
              mma_f16_16816(d, ha[0], hb[0], ha[1], hb[1], xq.x, xq.y);
              mma_f16_16816(d, ha[2], hb[2], ha[3], hb[3], xq.z, xq.w);
            } else {
              mma_f16_16816(d, ha[0], ha[0], ha[1], ha[1], xq.x, xq.y);
              mma_f16_16816(d, ha[2], ha[2], ha[3], ha[3], xq.z, xq.w);
            }
            const float xf = xfa[blk];
            acc0 = fmaf(d[0] + d[1], xf * e8m0_scale(sa[blk]), acc0);
            if (KIND == 0) acc1 = fmaf(d[2] + d[3], xf * e8m0_scale(sb[blk]), acc1);
          }
        }
        // exchange: lane (g, q) holds row g of assignment g0 + q
        const int buf = it & 1, ph = it >> 1;
        if (it >= 2) team_wait(&xfree_bar[team][buf], (ph - 1) & 1, 2);
        s_part[buf][cw][16 * tq + 2 * g] = acc0;
        s_part[buf][cw][16 * tq + 2 * g + 1] = acc1;
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_u32(&xfull_bar[team][buf]));
        if (wt == it % tw) {
          team_wait(&xfull_bar[team][buf], ph & 1, 3);
          const int jj = lane >> 3, r = lane & 7;  // the leader's lane: assignment g0 + jj, row r
          if (jj < ng && r < st.nr) {
            const int a = Rt.lst[l0 + g0 + jj];
            const int c0 = team * tw;
            float v0 = 0.f, v1 = 0.f;
            for (int w2 = 0; w2 < tw; ++w2) {
              v0 += s_part[buf][c0 + w2][16 * jj + 2 * r];
              v1 += s_part[buf][c0 + w2][16 * jj + 2 * r + 1];
            }
            if (!MOE_IN_BOUNDS(A.status, a >= 0 && a < TK && st.r0 + r < R)) {
            } else if (KIND == 0) {
              A.out[(size_t)a * R + st.r0 + r] = swiglu_oai_f(v0 + lb0, v1 + lb1, A.alpha, A.limit);
            } else {
              so[a * kDecRows + r] = v0 + lb0;
            }
          }
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(tc::smem_u32(&xfree_bar[team][buf]));
        }
      }
    } else
    for (int li = Rt.act_off[st.ai]; li < Rt.act_off[st.ai + 1]; ++li, ++it) {
      const int a = Rt.lst[li];
      const int v = (KIND == 0) ? a / k : a;
      float acc[NV];
#pragma unroll
      for (int r = 0; r < NV; ++r) acc[r] = 0.f;
      if (active && !dead) {
        if (A.staged)
          load_split_smem(vwords, vfac, v * nb + b, b, XH, XL, xf);
        else
          split_block_lane(A.vec + (size_t)v * C + 32 * b, XH, XL, xf);
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
          const uint8_t* qrow = stage + m * q_ms + b * 16;
          const uint8_t* srow = stage + NMAT * qsb + m * s_ms + sc_skew + b;
#pragma unroll
          for (int r = 0; r < kDecRows; ++r) {
            if (r < st.nr) {
              const uint4 q = *reinterpret_cast<const uint4*>(qrow + r * q_rs);
              const float sc = e8m0_scale(srow[r * s_rs]);
              acc[m * kDecRows + r] = (block_dot_split(q, XH, XL) * xf) * sc;
            }
          }
        }
      }
      const float part = transpose_reduce<NV>(acc, lane);
      // Exchange through s_part[buf]: every warp of the team publishes its row
      // partials, the iteration's leader (rotating) adds them up; the others
      // go straight on. A buffer is reused two iterations later, once its
      // leader has released it.
      const int buf = it & 1, ph = it >> 1;
      if (it >= 2) team_wait(&xfree_bar[team][buf], (ph - 1) & 1, 2);
      constexpr int SHIFT = (NV == 16) ? 1 : 2;
      if ((lane & ((1 << SHIFT) - 1)) == 0) s_part[buf][cw][lane >> SHIFT] = part;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tc::smem_u32(&xfull_bar[team][buf]));
      if (wt == it % tw) {
        team_wait(&xfull_bar[team][buf], ph & 1, 3);
        if (lane < st.nr) {
          const int c0 = team * tw;
          if (KIND == 0) {
            float g = 0.f, u = 0.f;
            for (int w2 = 0; w2 < tw; ++w2) {
              g += s_part[buf][c0 + w2][lane];
              u += s_part[buf][c0 + w2][kDecRows + lane];
            }
            if (MOE_IN_BOUNDS(A.status, a >= 0 && a < TK && st.r0 + lane < R))
              A.out[(size_t)a * R + st.r0 + lane] = swiglu_oai_f(g + bias0, u + bias1, A.alpha, A.limit);
          } else {
            float d = 0.f;
            for (int w2 = 0; w2 < tw; ++w2) d += s_part[buf][c0 + w2][lane];
            if (MOE_IN_BOUNDS(A.status, a >= 0 && a < TK)) so[a * kDecRows + lane] = d + bias0;
          }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_u32(&xfree_bar[team][buf]));
      }
    }
    __syncwarp();
    // This warp is done with the stage. A warp whose wait failed never releases:
    // the producer then stalls, sees the abort flag and stops.
    if (lane == 0 && !dead) tc::mbar_arrive(tc::smem_u32(&empty_bar[s]));
    // Down: the leader of the chunk's last iteration combines the chunk's rows
    // once the leader of the iteration before it is done too.
    if (KIND == 1 && st.last && wt == (it - 1) % tw) {
      if (it >= 2) team_wait(&xfree_bar[team][(it - 2) & 1], ((it - 2) >> 1) & 1, 4);
      for (int idx = lane; idx < T * st.nr; idx += 32) {
        const int t = idx / st.nr, r = idx - t * st.nr;
        float yv = 0.f;
        for (int jj = 0; jj < k; ++jj) {  // slot order
          const int a = t * k + jj;
          const int ej = Rt.ids[a];
          if (ej < 0 || ej >= E) continue;
          yv = fmaf(Rt.w[a], so[a * kDecRows + r], yv);
        }
        if (MOE_IN_BOUNDS(A.status, st.r0 + r < R)) A.out[(size_t)t * R + st.r0 + r] = yv;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
// Shared memory: stages (an equal number per team, 1..4) first, then the split
// vectors if they still fit (gate/up: with as little as one stage per team),
// then the down kernel's per-team row results.
static cudaError_t decode_plan(int KIND, int C, int nvec, int TK, DecodeArgs& A, size_t& smem) {
  constexpr size_t kBudget = 216 * 1024;  // with the kernel's static shared memory, under 227 KB
  const int nb = C >> 5;
  const int tw = (nb + 31) / 32;
  if (tw < 1 || tw > 4) return cudaErrorInvalidValue;
  const int nteams = kDecConsumers / tw;
  const int nmat = KIND == 0 ? 2 : 1;
  const size_t stage = (((size_t)nmat * (dec_qs_bytes(C) + dec_sc_bytes(C))) + 127) & ~(size_t)127;
  const size_t vec = (size_t)nvec * nb * (128 + 4);
  const size_t so = KIND == 1 ? (size_t)nteams * TK * kDecRows * 4 : 0;
  int spt = 0, staged = 0;
  // staged split vectors first (down to one stage per team for gate/up), else per-lane splits
  for (int s = 4; s >= (KIND == 0 ? 1 : 2) && !spt; --s)
    if ((size_t)nteams * s * stage + vec + so <= kBudget) spt = s, staged = 1;
  for (int s = 4; s >= 2 && !spt; --s)
    if ((size_t)nteams * s * stage + so <= kBudget) spt = s;
  if (!spt || nteams * spt > kDecMaxStages) return cudaErrorInvalidValue;
  A.tw = tw;
  A.spt = spt;
  A.staged = staged;
  A.stage_bytes = (uint32_t)stage;
  smem = (size_t)nteams * spt * stage + (staged ? vec : 0) + so;
  return cudaSuccess;
}

template <int KIND>
static cudaError_t launch_decode(DecodeArgs& A, int nvec, Launch L) {
  size_t smem = 0;
  cudaError_t err = decode_plan(KIND, A.C, nvec, A.T * A.k, A, smem);
  if (err != cudaSuccess) return err;
  if ((err = ensure_smem_limit(decode_expert_kernel<KIND>, smem)) != cudaSuccess) return err;
  const int per_sm = resident_blocks_per_sm(decode_expert_kernel<KIND>, kDecThreads, smem);
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const dim3 grid(device_sm_count() * per_sm);
  return launch_kernel(decode_expert_kernel<KIND>, grid, dim3(kDecThreads), smem, L, A);
}

cudaError_t launch_gemv_gateup(const uint8_t* g_qs, const uint8_t* g_sc, const float* bg,
                               const uint8_t* u_qs, const uint8_t* u_sc, const float* bu, int E,
                               int F, int D, int T, int k, const float* x, const float* logits,
                               const int32_t* ids_in, int32_t* ids_out, float* w_out, float alpha,
                               float limit, float* h, int* status, bool x_from_prev, Launch L, int rs) {
  if (T <= 0) return cudaSuccess;
  if (T * k > kMaxAssign || (rs != 1 && rs != 2)) return cudaErrorInvalidValue;
  DecodeArgs A = {};
  A.vec_wait = x_from_prev ? 1 : 0;
  A.rs = rs;
  A.qs[0] = g_qs;
  A.qs[1] = u_qs;
  A.sc[0] = g_sc;
  A.sc[1] = u_sc;
  A.bias[0] = bg;
  A.bias[1] = bu;
  A.E = E;
  A.R = F;
  A.C = D;
  A.T = T;
  A.k = k;
  A.vec = x;
  A.logits = logits;
  A.ids_in = ids_in;
  A.ids_out = ids_out;
  A.w_out = w_out;
  A.alpha = alpha;
  A.limit = limit;
  A.out = h;
  A.status = status;
  return launch_decode<0>(A, T, L);
}

cudaError_t launch_gemv_down(const uint8_t* d_qs, const uint8_t* d_sc, const float* bd, int E,
                             int D, int F, int T, int k, const float* h, const float* logits,
                             const int32_t* ids_in, const float* w_in, float* y, int* status,
                             Launch L) {
  if (T <= 0) return cudaSuccess;
  if (T * k > kMaxAssign) return cudaErrorInvalidValue;
  DecodeArgs A = {};
  A.rs = 1;
  A.qs[0] = d_qs;
  A.sc[0] = d_sc;
  A.bias[0] = bd;
  A.E = E;
  A.R = D;
  A.C = F;
  A.T = T;
  A.k = k;
  A.vec = h;
  A.logits = logits;
  A.ids_in = ids_in;
  A.w_in = w_in;
  A.out = y;
  A.status = status;
  return launch_decode<1>(A, T * k, L);
}

}  // namespace moe
