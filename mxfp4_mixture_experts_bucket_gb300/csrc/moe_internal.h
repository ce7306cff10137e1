// Internal (non-exported) launchers shared between the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace moe {

// Epilogue ids of the grouped GEMM (same values as the public MOE_EPI_* macros).
constexpr int MOE_EPI_STORE_BF16_ID = 0;
constexpr int MOE_EPI_SWIGLU_BF16_ID = 1;
constexpr int MOE_EPI_SCATTER_WEIGHTED_ID = 2;

struct Launch {
  cudaStream_t stream = nullptr;
  bool pdl = false;  // programmatic dependent launch on the previous kernel in the stream
};

// Counts every kernel the library enqueues (defined in abi.cu).
void count_launch();
// Records a cudaError_t for moe_last_cuda_error in the calling thread (abi.cu).
void set_last_cuda_error(int err);
int device_sm_count();

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, Launch L,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  cfg.numAttrs = 0;
  if (L.pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  count_launch();
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Raises a kernel's dynamic shared-memory limit to at least `bytes` (static
// plus dynamic may exceed the 48 KB default even when `bytes` alone does not).
// Remembered per (kernel, device); defined in abi.cu.
cudaError_t ensure_smem_limit_fn(const void* kern, size_t bytes);
// Resident blocks per SM of a kernel at a block size and dynamic shared memory,
// remembered per (kernel, device, threads, bytes); defined in abi.cu.
int resident_blocks_per_sm_fn(const void* kern, int threads, size_t smem);

template <typename K>
cudaError_t ensure_smem_limit(K kern, size_t bytes) {
  return ensure_smem_limit_fn(reinterpret_cast<const void*>(kern), bytes);
}
template <typename K>
int resident_blocks_per_sm(K kern, int threads, size_t smem) {
  return resident_blocks_per_sm_fn(reinterpret_cast<const void*>(kern), threads, smem);
}

// ---- route_bucket.cu ----
// x_copy (T <= 8 only, may be null): receives a copy of x [T][D] written by the kernel.
cudaError_t launch_router_logits(const float* x, int T, int D, const float* wr, const float* br,
                                 int E, float* logits, float* x_copy, Launch L);
cudaError_t launch_topk_softmax(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                                Launch L);
// Router and top-k-then-softmax in one call. T > 8 with `part` given: the
// router split over D (partial dots in part, kRouterMaxSplits x T x E floats at
// most), the slices added in order by the top-k kernel, which also writes
// logits. Else the single-pass router and topk_softmax.
constexpr int kRouterMaxSplits = 32;
size_t router_partials_bytes(int T, int E);
cudaError_t launch_route_topk(const float* x, int T, int D, const float* wr, const float* br, int E, int k,
                              float* logits, float* part, int32_t* ids, float* w, Launch L);
cudaError_t launch_bucket(const int32_t* ids, int T, int k, int E, int tile, int max_rows,
                          int32_t* counts, int32_t* basep, int32_t* rows, int32_t* inv,
                          int* status, Launch L);
cudaError_t launch_gather_bf16(const float* x, int T, int D, int k, const int32_t* rows,
                               const int32_t* basep, int E, int max_rows, uint16_t* xg,
                               uint16_t* xg_lo, float* y_zero, bool zero_pads, Launch L);

// ---- gemv.cu ----
cudaError_t launch_mxfp4_gemv(const uint8_t* qs, const uint8_t* sc, int E, int R, int C,
                              const int32_t* experts, int n, const float* x, int64_t x_stride,
                              const float* bias, float* out, int* status, Launch L);
cudaError_t launch_selftest_wait_timeout(const uint8_t* src, int* status, Launch L);
cudaError_t launch_quant_q8(const float* v, int64_t rows, int C, int8_t* q, float* d, Launch L);
cudaError_t launch_gemv_q8(const uint8_t* qs, const uint8_t* sc, int E, int R, int C, const int32_t* experts,
                           int n, int act_div, const int8_t* aq, const float* ad, const float* bias, float* out,
                           int* status, Launch L, int wrs = 1);
cudaError_t launch_combine_slots(const float* o, const float* w, const int32_t* ids, int T, int k, int D, int E,
                                 float* y, Launch L);
cudaError_t launch_rms_renorm(const float* x, int T, int D, float* y, Launch L);
cudaError_t launch_swiglu(const float* g, const float* u, void* h, int64_t n, int h_dtype,
                          float alpha, float limit, Launch L);

// ---- decode.cu ----
// Decode rail, stage 0: gate/up projections + bias + swiglu for every routed
// assignment. Routing comes from `logits` (top-k + softmax inside the kernel)
// when not NULL, else from `ids_in`; CTA 0 writes it to ids_out / w_out if not
// NULL. h: [T*k][F] floats, row per assignment.
// x_from_prev: x is written by the previous kernel in the stream (wait before reading it).
cudaError_t launch_gemv_gateup(const uint8_t* g_qs, const uint8_t* g_sc, const float* bg,
                               const uint8_t* u_qs, const uint8_t* u_sc, const float* bu, int E,
                               int F, int D, int T, int k, const float* x, const float* logits,
                               const int32_t* ids_in, int32_t* ids_out, float* w_out, float alpha,
                               float limit, float* h, int* status, bool x_from_prev, Launch L, int rs = 1);
// Decode rail, stage 1: down projection + bias + router-weighted combine in slot
// order. Routing from `logits` when not NULL, else from ids_in / w_in.
cudaError_t launch_gemv_down(const uint8_t* d_qs, const uint8_t* d_sc, const float* bd, int E,
                             int D, int F, int T, int k, const float* h, const float* logits,
                             const int32_t* ids_in, const float* w_in, float* y, int* status,
                             Launch L);

// ---- prepack.cu ----
// Prepacked MXFP4 planes of the block-scaled rails (layout in prepack.cu).
size_t packed_qs_bytes(int E, int R, int C);
size_t packed_sf_bytes(int E, int R, int C);
cudaError_t launch_prepack(const uint8_t* qs, const uint8_t* sc, int E, int R, int C, uint8_t* qs_p,
                           uint8_t* sf_p, Launch L, int rs = 1);

// ---- route_bucket.cu: prologue of the block-scaled decode rail ----
// Router logits, x as E4M3 operand chunks xq [NK][npad][128] + atoms xsf [NK][512],
// and zero[0 .. nzero) = 0.
cudaError_t launch_decode_prologue(const float* x, int T, int D, const float* wr, const float* br, int E,
                                   float* logits, uint8_t* xq, uint8_t* xsf, int npad, int* zero, int nzero,
                                   Launch L);

// ---- decode_mx.cu ----
constexpr int kDecodeMxMaxGrid = 256;  // partial-sum slots are sized for this many CTAs
struct DecodeMXArgs {
  int kind;  // 0: gate/up + swiglu (two matrices), 1: down + combine
  const uint8_t* w_qs[2];  // prepacked planes
  const uint8_t* w_sf[2];
  const float* bias[2];
  int E, R, C, T, k;
  const uint8_t* b_q;   // activation operand chunks
  const uint8_t* b_sf;
  const float* logits;
  int32_t* ids_out;
  float* w_out;
  float alpha, limit;
  uint8_t* hq;
  uint8_t* hsf;
  float* h_out;
  float* y;
  float* part;
  int* cnt;
  int* status;
};
cudaError_t launch_decode_mx(const DecodeMXArgs& a, Launch L);

// ---- grouped_mx4.cu: prefill grouped GEMMs on prepacked planes (kind::mxf4) ----
constexpr int kPrefillXTerms = 6;  // E2M1 terms of x (the gate/up operand)
constexpr int kPrefillHTerms = 4;  // E2M1 terms of h (the down operand)
struct GroupedMX4Args {
  int kind;                 // 0: gate/up + swiglu -> h rows; 1: down + weighted scatter into y
  const uint8_t* w_qs[2];   // prepacked planes (gate, up; or down, down)
  const uint8_t* w_sf[2];
  const float* bias[2];
  int E, R, C;              // per-expert matrices [R][C]
  const int32_t* counts;
  const int32_t* basep;
  const int32_t* rows;
  const int2* segs;         // segment table written by launch_quant_rows_e2m1 (2 * max_rows / 128 + 1 entries)
  int* ctr;                 // this GEMM's unit counter (zeroed by launch_quant_rows_e2m1)
  int max_rows, k;
  const float* weights;     // router weights [T*k] (down)
  const uint8_t* aq;        // activation chunks [max_rows/128][ceil(C/128)][terms][8192] (x: 6 terms, h: 4)
  const uint8_t* asf;       // their scale atoms [max_rows/128][ceil(C/128)][2 segments][terms][512]
  float* hf;                // gate/up output: h as float rows [max_rows][R]
  float alpha, limit;
  float* y;                 // down: [T][R], accumulated into; gate/up: zeroed (ny floats) while its first unit streams
  int64_t ny;
  int* status;
};
size_t prefill_operand_bytes(int max_rows, int C, int terms);
size_t prefill_atom_bytes(int max_rows, int C, int terms);
// x's token rows in bucket order as kPrefillXTerms E2M1 terms (each token split once, stored into
// its k bucket rows via inv), y zeroed unless null, and
// the segment table of the bucket (segs: 2 * max_rows / 128 + 1 entries); ctr[0..1] (the GEMMs'
// unit counters) zeroed
cudaError_t launch_quant_rows_e2m1(const float* x, int T, int D, int k, const int32_t* rows, const int32_t* inv,
                                   const int32_t* counts, const int32_t* basep, int E, int max_rows, uint8_t* aq,
                                   uint8_t* asf, float* y, int2* segs, int* ctr, int* status, Launch L);
// h's bucket rows (float [max_rows][F]) as kPrefillHTerms E2M1 terms
cudaError_t launch_quant_h_e2m1(const float* hf, int F, const int32_t* rows, const int32_t* counts,
                                const int32_t* basep, int E, int max_rows, uint8_t* hq, uint8_t* hsf, int* status,
                                Launch L);
cudaError_t launch_grouped_mx4(const GroupedMX4Args& a, Launch L);

// ---- grouped_mm.cu ----
struct GroupedMMArgs {
  const uint8_t* w_qs[2];
  const uint8_t* w_sc[2];
  const float* bias[2];
  int nmat;  // 1 or 2
  int E, R, C;
  const uint16_t* a;     // bf16 [max_rows][C]
  const uint16_t* a_lo;  // optional bf16 [max_rows][C]: low parts, the operand is a + a_lo
  const int32_t* counts;
  const int32_t* basep;
  const int32_t* rows;
  int max_rows;
  int k;
  const float* weights;
  int epilogue;
  float alpha, limit;
  void* out;
  int64_t out_ld;
  int64_t out_rows = 0;  // rows of out (scatter: tokens; row stores: max_rows), for the checked build; 0: unknown
  int* status;
  int rs = 1;  // nmat 2: 1 = separate planes; 2 = gate/up rows interleaved in one plane (w_qs[1], w_sc[1],
               // bias[1] point one row or one element past w_qs[0], w_sc[0], bias[0])
};
// Returns cudaErrorInvalidValue for unsupported shapes (checked by the caller first).
cudaError_t launch_grouped_mm(const GroupedMMArgs& args, Launch L);
// Tiled tensor map through the driver's encoder (no fill for out-of-range
// elements, 256-byte L2 promotion); false if the encoder is missing or refuses.
bool encode_tiled_map(CUtensorMap* tm, CUtensorMapDataType dtype, int rank, const void* base,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      CUtensorMapSwizzle swizzle);

// ---- grouped_mx.cu ----
// Gate/up (nmat 2) or down (nmat 1) on the block-scaled tensor cores. The
// activation operand is a sum of E4M3 terms (gate/up: 3, down: 2), each
// [max_rows][C] in the MMA's per-block K order, terms back to back, with scale
// words [terms][C/128 rounded up][max_rows].
struct GroupedMXArgs {
  const uint8_t* w_qs[2];
  const uint8_t* w_sc[2];
  const float* bias[2];
  int nmat;
  int E, R, C;
  const uint8_t* a_terms;
  const uint32_t* a_sc;
  const int32_t* counts;
  const int32_t* basep;
  const int32_t* rows;
  int max_rows;
  int k;
  const float* weights;
  float alpha, limit;
  uint8_t* h_terms;  // nmat 2: swiglu output in the down operand's format, [2][max_rows][R]
  uint32_t* h_sc;    // nmat 2: [2][R/128 rounded up][max_rows]
  float* y;          // nmat 1: [T][R], accumulated into (zeroed beforehand)
  int* status;
  int rs = 1;        // as GroupedMMArgs::rs
};
constexpr int kMxXTerms = 3;
constexpr int kMxHTerms = 2;
cudaError_t launch_grouped_mx(const GroupedMXArgs& args, Launch L);
// x rows in bucket order -> kMxXTerms E4M3 terms + scale words; zeroes y_zero [T][D] if given.
cudaError_t launch_quant_rows_mx(const float* x, int T, int D, int k, const int32_t* rows, const int32_t* basep,
                                 int E, int max_rows, uint8_t* q_terms, uint32_t* sc_terms, float* y_zero,
                                 Launch L);

}  // namespace moe
