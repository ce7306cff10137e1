/*
 * moe_mxfp4.h -- C ABI of the GB300 (sm_103a) MXFP4 routed mixture-of-experts
 * expert chain: router top-k, expert bucketing, MXFP4 projections with the
 * gpt-oss swiglu, and the router-weighted combine.
 *
 * The method follows three dasLLAMA pull-request pages:
 *  - "dasLLAMA gpt-oss arc: idot dot migrations, Metal fusion lane, fused MoE
 *    expert chain, fleet boards": the Metal fusion-lane commit (bias-seeded
 *    MetalMoeMulMmMx4, the MetalSwigluOaiPf ghost-row exit, the prefix folded
 *    into MetalMoeBucket) and the fused MoE expert chain commit (gate+up rows,
 *    bias, activation, then down rows, bias and the weighted sum in slot order).
 *  - "dasLLAMA: dig the last two board reds green -- lcpp-shape mx4 kernels +
 *    GPU PLE pre-step", section "gpt-oss: mx4 kernels to the lab-winning
 *    shape": the routed-expert MXFP4 GEMV (MetalMoeGemvMx4), the 16-value
 *    E2M1 table and the ALU E8M0 decode.
 *  - "dasLLAMA: M5 pp deep-dense - board v8", section "Claims - stated, not
 *    tested": 128-row tiles for the MoE tensor pair.
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers owned by the caller unless stated otherwise.
 *    The library allocates no memory and keeps no state except one status
 *    word per device (moe_get_status).
 *  - Work is enqueued on `stream` and the call returns without waiting for it.
 *    No call below synchronises the host except moe_get_status.
 *  - Return value: MOE_OK, or a negative code. MOE_EINVAL means an argument
 *    was rejected on the host before anything was enqueued. MOE_ECUDA means a
 *    CUDA runtime call failed (moe_last_cuda_error gives its cudaError_t).
 *    MOE_EUNSUPPORTED means the shape or the device is outside what the
 *    kernels handle (the kernels are built for sm_103a only).
 *  - Data errors found on the device (an expert id outside [0, E), a pipeline
 *    wait that timed out) never trap: they set bits in the device status word.
 *
 * MXFP4 storage: a matrix W[R][C] (C a multiple of 32) is two planes, both
 * row-major: the nibble plane qs[R][C/2] (uint8) and the exponent plane
 * sc[R][C/32] (uint8, E8M0). Block b of a row covers columns 32b..32b+31 and
 * is held in bytes 16b..16b+15 of the row; byte i holds column 32b+i in its
 * low nibble and column 32b+16+i in its high nibble. The value is
 * E2M1[q] * 2^(s-127), E2M1 = {0, .5, 1, 1.5, 2, 3, 4, 6, -0, -.5, -1, -1.5,
 * -2, -3, -4, -6}; s = 255 decodes to NaN. Expert matrices are stacked:
 * qs[E][R][C/2], sc[E][R][C/32]. Planes must be 16-byte aligned.
 */
#ifndef MOE_MXFP4_H
#define MOE_MXFP4_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ---- */
#define MOE_OK 0
#define MOE_EINVAL (-1)
#define MOE_ECUDA (-2)
#define MOE_EUNSUPPORTED (-3)
#define MOE_ESCRATCH (-4) /* the shape needs more scratch than MOE_DECODE_SCRATCH_BYTES */

/* ---- device status bits (moe_get_status) ---- */
#define MOE_STATUS_BAD_EXPERT_ID 0x1 /* an id outside [0, E) reached a kernel */
#define MOE_STATUS_WAIT_TIMEOUT 0x2  /* a pipeline wait gave up; outputs are invalid */
#define MOE_STATUS_OUT_OF_BOUNDS 0x4 /* checked build only: an index a kernel formed fell outside its
                                        buffer; that access was skipped, outputs are invalid */

/* ---- activation element types ---- */
#define MOE_DTYPE_F32 0
#define MOE_DTYPE_BF16 1

/* ---- grouped-GEMM epilogues ---- */
#define MOE_EPI_STORE_BF16 0       /* out[p][r] = bf16(acc)                       */
#define MOE_EPI_SWIGLU_BF16 1      /* out[p][r] = bf16(swiglu_oai(acc1, acc2))     */
#define MOE_EPI_SCATTER_WEIGHTED 2 /* out[t][r] += weights[a] * acc, a = rows[p]   */

/* ---- layer rails ---- */
#define MOE_RAIL_AUTO 0       /* by T: see MOE_AUTO_GEMV_MAX_T and MOE_AUTO_MX_MAX_T */
#define MOE_RAIL_GEMV 1
#define MOE_RAIL_GROUPED_MM 2
#define MOE_RAIL_GROUPED_MX 3 /* grouped GEMM on the block-scaled (MXFP4 x E4M3) tensor cores */
#define MOE_RAIL_DECODE_MX 4  /* T <= MOE_GEMV_MAX_T on the block-scaled tensor cores (prepacked weights) */
#define MOE_RAIL_GEMV_Q8 5    /* T <= MOE_GEMV_MAX_T: x and h requantised to Q8, integer MXFP4 x Q8 dots */
#define MOE_RAIL_GROUPED_MX4 6 /* prepacked weights, any T: grouped GEMMs on tcgen05.mma kind::mxf4 */
#define MOE_GEMV_MAX_T 8
/*
 * MOE_RAIL_AUTO on the canonical planes (moe_ffn_layer and friends) takes the
 * rail measured fastest on GB300 for the gpt-oss shape (E=32, k=4,
 * D=F=2880): the GEMV rail for T <= MOE_AUTO_GEMV_MAX_T (its whole range:
 * 135 us against 158 us for the next rail at T = 4, 217 against 233 at T = 8),
 * the block-scaled grouped GEMM for T <= MOE_AUTO_MX_MAX_T, the bf16 grouped
 * GEMM beyond. The rails differ in precision: the GEMV rail is held to 1e-4 of a
 * float64 reference (row-normwise), the grouped rails to 2e-2; a caller that
 * needs the tighter bound names MOE_RAIL_GEMV. On prepacked planes
 * (moe_ffn_layer_packed) MOE_RAIL_AUTO is MOE_RAIL_DECODE_MX for
 * T <= MOE_AUTO_DECODE_MX_MAX_T and MOE_RAIL_GROUPED_MX4 beyond (measured:
 * at T = 2 the decode rail leads by about 6%, from T = 4 the grouped rail
 * leads, 72 us against 84 us per layer step, 183 us at T = 512).
 */
#define MOE_AUTO_GEMV_MAX_T 8
#define MOE_AUTO_MX_MAX_T 320
#define MOE_AUTO_DECODE_MX_MAX_T 2

/* Bucket tile height of the grouped-GEMM rail (rows per tensor-core tile). */
#define MOE_MM_TILE 128

/*
 * moe_bucket_max_rows -- length of the `rows` array of moe_bucket: the
 * worst-case padded row count T*k + E*(tile-1), rounded up to a whole tile.
 * Returns 0 for invalid arguments. Host only.
 */
size_t moe_bucket_max_rows(int T, int k, int E, int tile);

/*
 * moe_ffn_workspace_bytes -- bytes of device workspace moe_ffn_layer needs
 * for the given shape and rail (MOE_RAIL_AUTO resolves as moe_ffn_layer
 * does). Returns 0 for invalid arguments. Host only.
 */
size_t moe_ffn_workspace_bytes(int T, int D, int F, int E, int k, int rail);

/*
 * moe_route_topk -- router logits, top-k, softmax over the k selected.
 *   logits[t][e] = sum_i x[t][i] * w_router[e][i] + b_router[e]   (fp32)
 *   ids[t][0..k-1]: the k largest logits of token t in descending order,
 *                   lower expert index first on equal logits (slot order)
 *   weights[t][j] = exp(l_j - l_0) / sum_m exp(l_m - l_0) over the k selected
 * x: float [T][D]; w_router: float [E][D]; b_router: float [E] or NULL;
 * logits: float [T][E] (output); ids: int32 [T][k]; weights: float [T][k].
 * Requires 1 <= k <= E <= 256, D a multiple of 4, T >= 0 (T = 0 is a no-op).
 * The selection on the pages is implicit (the router produces the "ids" that
 * the MoE kernels consume, E = 32, k = 4); top-k then softmax over the k is
 * the gpt-oss router.
 */
int moe_route_topk(const float* x, int T, int D, const float* w_router, const float* b_router,
                   int E, int k, float* logits, int32_t* ids, float* weights, cudaStream_t stream);

/*
 * moe_bucket -- CSR of the T*k (token, slot) assignments grouped by expert,
 * with each expert's row range padded to `tile` rows (MetalMoeBucket with
 * MetalMoePrefix folded in: each expert's block computes its own padded
 * base in-block; "dasLLAMA gpt-oss arc", Metal fusion lane commit, third
 * bullet). One kernel; the result is deterministic and bit-exact:
 *   counts[e]  = number of assignments with ids == e                 int32 [E]
 *   basep[e]   = sum_{e' < e} ceil(counts[e']/tile)*tile; basep[E] = mpad   int32 [E+1]
 *   rows[p]    = t*k + j for p in [basep[e], basep[e]+counts[e]), ascending;
 *                -1 at every other p < moe_bucket_max_rows(T, k, E, tile)
 *   inv[t*k+j] = the row p holding that assignment, -1 if its id is invalid int32 [T*k]
 * ids: int32 [T][k]. Ids outside [0, E) are skipped and set
 * MOE_STATUS_BAD_EXPERT_ID. Requires 1 <= k, 1 <= E <= 1024, 1 <= tile <= 1024.
 */
int moe_bucket(const int32_t* ids, int T, int k, int E, int tile, int32_t* counts, int32_t* basep,
               int32_t* rows, int32_t* inv, cudaStream_t stream);

/*
 * moe_mxfp4_gemv -- n independent MXFP4 matrix-vector products with bias
 * (the routed-expert GEMV, MetalMoeGemvMx4, of "dasLLAMA: dig the last two
 * board reds green", section "gpt-oss: mx4 kernels to the lab-winning shape").
 *   out[i][r] = sum_c W[experts[i]][r][c] * x_i[c] + bias[experts[i]][r]
 * W: stacked MXFP4 planes w_qs [E][R][C/2], w_sc [E][R][C/32]; experts: int32
 * [n]; x_i = x + i * x_stride (floats; x_stride = 0 uses one vector for all
 * i); bias: float [E][R] or NULL; out: float [n][R]. fp32 accumulation.
 * Requires C a multiple of 32, x_stride a multiple of 4. An expert id outside
 * [0, E) gives a zero row and sets MOE_STATUS_BAD_EXPERT_ID.
 */
int moe_mxfp4_gemv(const uint8_t* w_qs, const uint8_t* w_sc, int E, int R, int C,
                   const int32_t* experts, int n, const float* x, int64_t x_stride,
                   const float* bias, float* out, cudaStream_t stream);

/*
 * moe_quantize_q8 -- activations requantised in blocks of 32 (the 32-block
 * requant of the first stage of the fused MoE expert chain, "dasLLAMA gpt-oss
 * arc", fused MoE expert chain commit): for every block of 32 consecutive
 * values of the rows x [rows][C], with amax its largest magnitude,
 *   d = amax / 127,  q[c] = round(x[c] * (127 / amax))  (nearest, ties to even),
 * each division and product rounded to float32; an all-zero block gives d = 0
 * and zero codes. q: int8 [rows][C], d: float [rows][C/32], both device memory
 * owned by the caller. Finite inputs. Requires C a multiple of 32; x and q
 * 16-byte aligned. Deterministic, bit-exact.
 */
int moe_quantize_q8(const float* x, int64_t rows, int C, int8_t* q, float* d, cudaStream_t stream);

/*
 * moe_mxfp4_gemv_q8 -- n MXFP4 x Q8 matrix-vector products with bias, taken
 * in integers (the dot_mx4q8 template of "dasLLAMA gpt-oss arc", commit
 * "dot_mx4q8_template rewritten in plain das": the weight block's nibbles go
 * through a table, the low one masked with 15, the high one shifted by 4, and
 * four-lane integer dots accumulate):
 *   isum[b] = sum_{i<32} T2[code(r, 32b+i)] * q_a[32b+i]       (exact, int32)
 *   out[i][r] = sum_b isum[b] * (d_a[b] * 2^(s[r][b] - 128)) + bias[e][r]
 * with T2 the E2M1 table doubled (integers in [-12, 12]), a = i / act_div the
 * activation row (act_div = k: one row per token for the k slots of a token;
 * 1: one row per output), e = experts[i], s the weight block's E8M0 byte (255:
 * NaN). The float32 sum has a fixed order: lane l of 32 adds blocks l, l+32,
 * ... in ascending order (each product and sum rounded to float32), then the
 * 32 lane sums meet in a butterfly over lane distances 16, 8, 4, 2, 1, then the
 * bias is added: the result is bit-exact and deterministic. W: w_qs
 * [E][R][C/2], w_sc [E][R][C/32]; q: int8 [rows][C], d: float [rows][C/32]
 * from moe_quantize_q8; bias float [E][R] or NULL; out float [n][R].
 * Requires C a multiple of 32 and at most 4096 (MOE_EUNSUPPORTED beyond),
 * act_div >= 1, q and w_qs 16-byte aligned. An expert id outside [0, E) gives
 * a zero row and sets MOE_STATUS_BAD_EXPERT_ID.
 */
int moe_mxfp4_gemv_q8(const uint8_t* w_qs, const uint8_t* w_sc, int E, int R, int C, const int32_t* experts,
                      int n, int act_div, const int8_t* q, const float* d, const float* bias, float* out,
                      cudaStream_t stream);

/*
 * moe_swiglu_oai -- h = min(g, limit) * sigmoid(alpha * min(g, limit))
 *                       * (clamp(u, -limit, limit) + 1)
 * elementwise over n floats (gpt-oss uses alpha = 1.702, limit = 7). h is
 * float (h_dtype MOE_DTYPE_F32) or bfloat16 (MOE_DTYPE_BF16, rounded to
 * nearest even). The sigmoid is evaluated without overflow for any g.
 * The pages name this activation as the MetalSwigluOaiPf kernel of the prefill
 * chain ("dasLLAMA gpt-oss arc", Metal fusion lane commit, second bullet: the
 * swiglu rows past each bucket's live end exit early) and as the activation of
 * stage 0 of the fused MoE expert chain commit; its constants and the one-sided
 * gate clamp are those of gpt-oss.
 */
int moe_swiglu_oai(const float* g, const float* u, void* h, int64_t n, int h_dtype, float alpha,
                   float limit, cudaStream_t stream);

/*
 * moe_rms_renorm -- y[t][c] = x[t][c] / sqrt(mean over c of x[t][c]^2) for
 * t < T, c < D (a row of zeros stays zero): the renormalisation between the
 * layers of a stack of MoE layers, which keeps the hidden state of a deep
 * stack bounded. It is not a step of the MoE layer: gpt-oss puts an RMSNorm
 * before each MoE block (its learned gain is not modelled here). x, y: float
 * [T][D] in device memory, owned by the caller; in place (y == x) is allowed.
 * The sum of squares is added in a fixed order, so the result is
 * deterministic. Returns MOE_EINVAL for T < 0, D < 1 or a NULL pointer with
 * T > 0.
 */
int moe_rms_renorm(const float* x, int T, int D, float* y, cudaStream_t stream);

/*
 * moe_gather_rows_bf16 -- activation rows of the grouped GEMM in bucket order:
 *   xg[p][:] = bf16(x[rows[p] / k][:]) for p < basep[E] with rows[p] >= 0,
 *   xg[p][:] = 0 for pad rows p < basep[E]; rows p >= basep[E] are not written.
 * If xg_lo is not NULL it receives the rounding remainders in the same rows,
 * xg_lo[p][c] = bf16(x - float(xg[p][c])), so that xg + xg_lo carries 16
 * significant bits of x (the layer uses this split for its gate/up GEMM: with
 * weights of large E8M0 scale, rounding x alone to bf16 moves g and u by whole
 * units near the swiglu clamp knees). Rounding is to nearest even.
 * x: float [T][D]; rows/basep from moe_bucket; xg, xg_lo: bf16 [max_rows][D].
 * If y_zero is not NULL, y_zero[0 .. T*D) is also set to 0 (the scatter
 * epilogue accumulates into it). Requires D a multiple of 8.
 */
int moe_gather_rows_bf16(const float* x, int T, int D, int k, const int32_t* rows,
                         const int32_t* basep, int E, int max_rows, uint16_t* xg, uint16_t* xg_lo,
                         float* y_zero, cudaStream_t stream);

/*
 * moe_mxfp4_grouped_mm -- per-expert MXFP4 GEMM over the bucket rows on the
 * tcgen05 tensor cores (MetalMoeMulMmMx4; "dasLLAMA gpt-oss arc", Metal
 * fusion lane commit). For every expert e and every live bucket row p in
 * [basep[e], basep[e] + counts[e]):
 *   acc[p][r]  = bias[e][r] + sum_c W[e][r][c] * a[p][c]       (r < R)
 *   acc2[p][r] = bias2[e][r] + sum_c W2[e][r][c] * a[p][c]     (MOE_EPI_SWIGLU_BF16 only)
 * where a[p][c] is the bf16 row, or a[p][c] + a_lo[p][c] when a_lo is not NULL
 * (a second MMA per step on the low parts, accumulating into the same tensor
 * memory). bf16 x bf16 products, fp32 accumulation in tensor memory; the bias seeds
 * the accumulator (NULL bias: the accumulator starts at zero). Then:
 *   MOE_EPI_STORE_BF16:        out (bf16 [max_rows][out_ld]) row p = bf16(acc[p])
 *   MOE_EPI_SWIGLU_BF16:       out row p = bf16(swiglu_oai(acc[p], acc2[p]; alpha, limit))
 *   MOE_EPI_SCATTER_WEIGHTED:  out (float [T][out_ld]) row rows[p]/k += weights[rows[p]] * acc[p]
 *                              (atomic adds: the order of the k contributions is not fixed)
 * Pad rows and rows past basep[E] are neither computed nor written; tiles
 * past basep[E] exit at once. a: bf16 [max_rows][C] in bucket order (see
 * moe_gather_rows_bf16), max_rows = moe_bucket_max_rows(., ., E, MOE_MM_TILE);
 * basep must be padded to MOE_MM_TILE. Requires C a multiple of 64 with
 * C <= 4096, R a multiple of 8, out_ld >= R and a multiple of 8.
 */
int moe_mxfp4_grouped_mm(const uint8_t* w_qs, const uint8_t* w_sc, const float* bias,
                         const uint8_t* w2_qs, const uint8_t* w2_sc, const float* bias2, int E,
                         int R, int C, const uint16_t* a, const uint16_t* a_lo,
                         const int32_t* counts, const int32_t* basep, const int32_t* rows,
                         int max_rows, int k, const float* weights, int epilogue, float alpha,
                         float limit, void* out, int64_t out_ld, cudaStream_t stream);

/*
 * moe_expert_gateup_swiglu -- stage 0 of the fused decode expert chain ("dasLLAMA
 * gpt-oss arc", fused MoE expert chain commit: gate+up rows + bias + activation
 * per expert row span), the GEMV rail's first expert kernel (the routed-expert
 * GEMV MetalMoeGemvMx4 takes the router's expert ids the same way). For every
 * assignment a = t*k + j with e = ids[a] in [0, E):
 *   h[a] = swiglu_oai(Wg[e] x_t + bg[e], Wu[e] x_t + bu[e]; alpha, limit)
 * Each weight row is streamed from HBM once for all of the tokens routed to
 * its expert. x: float [T][D]; ids: int32 [T][k]; gate/up planes [E][F][D/2],
 * [E][F][D/32]; bg, bu [E][F] or NULL; h: float [T*k][F], row a = h[a] (rows
 * of assignments with an invalid id are left as they were). x and h must be
 * 16-byte aligned. Ids outside [0, E) are skipped and set
 * MOE_STATUS_BAD_EXPERT_ID.
 * Requires 1 <= T <= MOE_GEMV_MAX_T, k <= 8, D and F multiples of 64, <= 4096.
 */
int moe_expert_gateup_swiglu(const uint8_t* g_qs, const uint8_t* g_sc, const float* bg,
                             const uint8_t* u_qs, const uint8_t* u_sc, const float* bu, int E,
                             int F, int D, int T, int k, const float* x, const int32_t* ids,
                             float alpha, float limit, float* h, cudaStream_t stream);

/*
 * moe_expert_down_combine -- stage 1 of the fused decode expert chain: every
 * expert's down rows, bias, and the router-weighted sum in slot order, per
 * output row span:
 *   y[t][c] = sum_{j=0..k-1} weights[t][j] * (Wd[ids[t][j]][c] . h[t*k+j] + bd[ids[t][j]][c])
 * summed for j = 0, 1, ..., k-1 in that order (deterministic). h: output of
 * moe_expert_gateup_swiglu; ids int32 [T][k], weights float [T][k]; down
 * planes [E][D][F/2], [E][D][F/32]; bd [E][D] or NULL; y: float [T][D],
 * overwritten. Same limits as moe_expert_gateup_swiglu.
 */
int moe_expert_down_combine(const uint8_t* d_qs, const uint8_t* d_sc, const float* bd, int E, int D,
                            int F, int T, int k, const float* h, const int32_t* ids,
                            const float* weights, float* y, cudaStream_t stream);

/*
 * moe_ffn_layer -- the whole routed-expert chain for T tokens:
 *   route (moe_route_topk) -> bucket -> gate/up projections with bias and
 *   swiglu_oai -> down projection with bias -> router-weighted combine in
 *   slot order.
 * This is the chain of "dasLLAMA gpt-oss arc": the Metal fusion lane commit
 * for prefill (MetalMoeBucket with the prefix folded in, bias-seeded
 * MetalMoeMulMmMx4 for gate/up and down, MetalSwigluOaiPf between them, ghost
 * rows exiting early) and the fused MoE expert chain commit for decode (stage 0:
 * gate+up rows, bias, activation; stage 1: down rows, bias and the weighted sum
 * in slot order), with the routed-expert GEMV of "dasLLAMA: dig the last two
 * board reds green", section "gpt-oss: mx4 kernels to the lab-winning shape".
 *   y[t] = sum_j weights[t][j] * (Wd[e] h_j + bd[e]),  e = ids[t][j],
 *   h_j  = swiglu_oai(Wg[e] x_t + bg[e], Wu[e] x_t + bu[e])  (alpha 1.702, limit 7)
 * Rails: MOE_RAIL_GEMV (T <= MOE_GEMV_MAX_T) streams the touched experts'
 * weights through fused GEMVs with fp32 accumulation (gate/up + swiglu, its
 * inner products on the tensor pipe with mma.sync when the activations fit in
 * shared memory; down + bias + slot-order combine on the CUDA cores;
 * deterministic); its two expert kernels take the
 * top-k of the router logits themselves, so a decode step is three kernels. MOE_RAIL_GROUPED_MM runs the
 * tcgen05 grouped GEMM with bf16 MMAs (x enters gate/up split into bf16 high
 * and low parts, h enters down rounded to bf16), the swiglu fused into the
 * gate/up epilogue and the weighted scatter fused into the down epilogue.
 * MOE_RAIL_GROUPED_MX has the same structure on the block-scaled tensor cores:
 * the MXFP4 weights enter the MMA as stored (no dequantisation); x enters as
 * a sum of three E4M3 blocks and h as two (each block of 32 on its own E8M0
 * scale, each term carrying the rounding residual of the ones before: about
 * 12 and 8 significant bits). Both grouped rails accumulate in fp32 and
 * scatter with float atomics (order not deterministic).
 * MOE_RAIL_GEMV_Q8 (T <= MOE_GEMV_MAX_T, k <= 8) is the Q8 variant of the
 * decode rail: x and h are requantised in blocks of 32 (moe_quantize_q8) and
 * each projection is moe_mxfp4_gemv_q8 (integer block dots), then the
 * slot-order combine; nine kernels, deterministic. It computes the layer on
 * the requantised operands to float32 rounding; its distance from the float64
 * layer is the requant's own (each activation rounded to 1/254 of its block's
 * largest: large where a block of h spans several orders of magnitude).
 * MOE_RAIL_AUTO picks by T (MOE_AUTO_GEMV_MAX_T, MOE_AUTO_MX_MAX_T above).
 * x: float [T][D]; w_router [E][D]; b_router [E] or NULL; gate/up planes
 * [E][F][D/2], [E][F][D/32]; down planes [E][D][F/2], [E][D][F/32]; biases
 * bg, bu [E][F], bd [E][D] (each may be NULL); y: float [T][D], overwritten.
 * ids_out [T][k] and weights_out [T][k] receive the routing if not NULL.
 * workspace: device memory of at least moe_ffn_workspace_bytes(T, D, F, E, k,
 * rail) bytes, 256-byte aligned; its contents on entry do not matter.
 * Requires D, F multiples of 64 (grouped rail: also <= 4096), 1 <= k <= E <= 256.
 */
int moe_ffn_layer(const float* x, int T, int D, int F, int E, int k, const float* w_router,
                  const float* b_router, const uint8_t* g_qs, const uint8_t* g_sc, const float* bg,
                  const uint8_t* u_qs, const uint8_t* u_sc, const float* bu, const uint8_t* d_qs,
                  const uint8_t* d_sc, const float* bd, int rail, void* workspace,
                  size_t workspace_bytes, float* y, int32_t* ids_out, float* weights_out,
                  cudaStream_t stream);

/*
 * moe_ffn_layer_gu -- moe_ffn_layer with gate and up stored as gpt-oss stores
 * them: one MXFP4 plane per expert of 2F rows, gate row f at row 2f and up row
 * f at row 2f+1 (the pages' decode stage reads "gate+up rows" together:
 * "dasLLAMA gpt-oss arc", fused MoE expert chain commit, stage 0). gu_qs
 * [E][2F][D/2], gu_sc [E][2F][D/32], gu_b [E][2F] (interleaved the same way)
 * or NULL; every other argument, the workspace (moe_ffn_workspace_bytes) and
 * the results are those of moe_ffn_layer on the separated planes, bit for bit
 * on the deterministic rails (GEMV, GEMV_Q8). The GEMV rail streams a
 * sub-task's gate and up rows as one run of 2*8 rows (one copy for the
 * nibbles, one for the scales); the grouped rails read the plane through
 * strided tensor maps. Requires gu_qs 16-byte aligned and gu_sc 16-byte
 * aligned; other requirements as moe_ffn_layer.
 */
int moe_ffn_layer_gu(const float* x, int T, int D, int F, int E, int k, const float* w_router,
                     const float* b_router, const uint8_t* gu_qs, const uint8_t* gu_sc, const float* gu_b,
                     const uint8_t* d_qs, const uint8_t* d_sc, const float* bd, int rail, void* workspace,
                     size_t workspace_bytes, float* y, int32_t* ids_out, float* weights_out, cudaStream_t stream);

/*
 * moe_ffn_args_t -- every argument of moe_ffn_layer that stays fixed from one
 * step to the next, plus two device staging buffers x_dev and y_dev of T*D
 * floats (16-byte aligned). Filled once by the caller; the library neither
 * keeps nor frees anything it points to.
 */
typedef struct {
  int T, D, F, E, k, rail;
  const float* w_router;
  const float* b_router;
  const uint8_t* g_qs;
  const uint8_t* g_sc;
  const float* bg;
  const uint8_t* u_qs;
  const uint8_t* u_sc;
  const float* bu;
  const uint8_t* d_qs;
  const uint8_t* d_sc;
  const float* bd;
  void* workspace;
  size_t workspace_bytes;
  float* x_dev;
  float* y_dev;
} moe_ffn_args_t;

/*
 * moe_ffn_layer_hostio -- moe_ffn_layer for tokens that live in host memory:
 * on `stream` it copies x_host [T][D] to args->x_dev, runs moe_ffn_layer with
 * the fixed arguments in *args (same definition, rails, limits and workspace
 * contract), and copies args->y_dev back to y_host [T][D], all enqueued from C
 * so that a serving loop passes four arguments per step. x_host and y_host
 * should be pinned (page-locked) for the copies to be asynchronous. The call
 * returns once the work is enqueued: y_host holds the result after the stream
 * has been synchronised. Errors as moe_ffn_layer; a failed copy returns
 * MOE_ECUDA.
 * On the GEMV rail with pinned x_host and y_host no copy is enqueued: the
 * router kernel reads x from host memory through the pinned mapping and
 * writes the device copy into x_dev (the expert kernels read that), and the
 * down kernel writes y straight into y_host (y_dev is not touched). Other
 * rails, and pageable buffers, copy through x_dev and y_dev as described.
 */
int moe_ffn_layer_hostio(const moe_ffn_args_t* args, const float* x_host, float* y_host,
                         cudaStream_t stream);

/*
 * ---- Prepacked weights for the block-scaled tensor-core rails ----
 *
 * The same MXFP4 values (E2M1 codes and E8M0 exponents, nothing decoded or
 * rounded), placed so that one contiguous copy brings a 128-row weight tile
 * into shared memory in the operand order of tcgen05.mma kind::mxf4:
 *   qs_p: tile by tile, NK = ceil(C/128) chunks of 64 bytes per row. Expert e,
 *        128-row tile t (rows_t = 128, or R - 128t for the last tile) starts at
 *        byte (e*R + 128t) * NK*64; inside it the 128-column chunk j starts at
 *        rows_t*64*j and is the 64-byte-swizzled image of its rows: block kb of
 *        tile row m at m*64 + 16*(kb ^ ((m >> 1) & 3)) (its 16 bytes as stored;
 *        blocks past C/32 are zero). moe_mxfp4_packed_qs_bytes(E, R, C) =
 *        E*R*NK*64.
 *   sf_p [E][ceil(R/128)][NK][512] bytes, NK = ceil(C/128): byte
 *        16*(m%32) + 4*(m/32) + kb of an atom is the exponent of tile row m,
 *        block 4j+kb (127 where the row or block does not exist).
 *        moe_mxfp4_packed_sf_bytes(E, R, C).
 */
size_t moe_mxfp4_packed_qs_bytes(int E, int R, int C);
size_t moe_mxfp4_packed_sf_bytes(int E, int R, int C);

/*
 * moe_mxfp4_prepack -- canonical planes qs [E][R][C/2], sc [E][R][C/32] ->
 * prepacked planes qs_p, sf_p (layout above). Run once per weight matrix
 * stack, e.g. at load time. Requires R a multiple of 64 and C a multiple of
 * 32; qs, sc, sf_p 16-byte aligned, qs_p 32-byte aligned. The layer kernels
 * further require C a multiple of 64.
 */
int moe_mxfp4_prepack(const uint8_t* qs, const uint8_t* sc, int E, int R, int C, uint8_t* qs_p,
                      uint8_t* sf_p, cudaStream_t stream);

/*
 * moe_mxfp4_prepack_gu -- moe_mxfp4_prepack of the gate and the up matrices
 * straight from one interleaved gate/up plane (gu_qs [E][2F][D/2], gu_sc
 * [E][2F][D/32]: gate row f at row 2f, up row f at row 2f+1, as
 * moe_ffn_layer_gu takes them) into the two prepacked pairs (g_qs_p, g_sf_p)
 * and (u_qs_p, u_sf_p), each sized moe_mxfp4_packed_*_bytes(E, F, D). The
 * packed planes equal those of moe_mxfp4_prepack on the separated planes.
 * Requires F a multiple of 64, D of 32; gu_qs 16-byte aligned, *_qs_p 32, *_sf_p 16.
 */
int moe_mxfp4_prepack_gu(const uint8_t* gu_qs, const uint8_t* gu_sc, int E, int F, int D, uint8_t* g_qs_p,
                         uint8_t* g_sf_p, uint8_t* u_qs_p, uint8_t* u_sf_p, cudaStream_t stream);

/*
 * moe_packed_layer_t -- one layer's device weights with the three expert
 * matrix stacks prepacked (gate/up [E][F][D], down [E][D][F]); biases and the
 * router as in moe_ffn_layer (b_router, bg, bu, bd may be NULL).
 */
typedef struct {
  int D, F, E, k;
  const float* w_router;
  const float* b_router;
  const uint8_t* g_qs;
  const uint8_t* g_sf;
  const float* bg;
  const uint8_t* u_qs;
  const uint8_t* u_sf;
  const float* bu;
  const uint8_t* d_qs;
  const uint8_t* d_sf;
  const float* bd;
} moe_packed_layer_t;

/*
 * moe_ffn_packed_workspace_bytes -- device workspace of moe_ffn_layer_packed
 * (MOE_RAIL_AUTO resolves as there). Returns 0 for invalid arguments or a
 * rail the packed layer does not run. Host only.
 */
size_t moe_ffn_packed_workspace_bytes(int T, int D, int F, int E, int k, int rail);

/*
 * moe_ffn_layer_packed -- moe_ffn_layer (same definition of y, routing and
 * combine) on prepacked weights. Rails: MOE_RAIL_DECODE_MX (MOE_RAIL_AUTO for
 * T <= MOE_GEMV_MAX_T) runs the decode step as three kernels: a prologue
 * (router logits; x as a sum of eight MXFP4 terms per value, each block of 32
 * E2M1 codes on its own E8M0 scale, the residual left ~1e-7 of the block's
 * largest value), gate/up + bias + swiglu on the block-scaled tensor cores
 * (tcgen05.mma kind::mxf4) with the MXFP4 weights as stored, and down on the
 * same tensor cores with the router weights folded into the operand (w*h as
 * eight MXFP4 terms) so that all k experts of a token accumulate in one fp32
 * accumulator, plus sum_j w_j bd[e_j] in slot order. Every SM streams an
 * equal share of the routed experts' weight tiles; tiles shared by several
 * CTAs are summed in a fixed order, so results are deterministic.
 * h_out (may be NULL): receives the swiglu outputs h[t*k+j][F] of the
 * assignments (decode rail only). Other arguments and limits as in
 * moe_ffn_layer; D and F multiples of 64; k*T <= 64 on the decode rail.
 * MOE_RAIL_GROUPED_MX4 (MOE_RAIL_AUTO for T > MOE_AUTO_DECODE_MX_MAX_T) runs the prefill
 * chain of "dasLLAMA gpt-oss arc" (Metal fusion lane commit: router, the
 * MoeBucket CSR with the prefix folded in, the MXFP4 grouped mul_mm for
 * gate/up with bias and swiglu, then down with bias and the router-weighted
 * scatter) on the same prepacked planes: x enters as six E2M1 terms per value
 * in bucket order; on tcgen05.mma kind::mxf4 each 128-row weight tile is the A
 * operand and a bucket segment of at most 96 live rows (as many of its terms
 * stacked per MMA as fit 192 columns) the B operand, so the MMA work follows
 * the live rows, not the 128-row padding; h leaves the gate/up epilogue as
 * float rows split into four E2M1 terms, and the down
 * epilogue scatters w*(acc + bd) into y with float atomics (summation order not
 * deterministic).
 */
int moe_ffn_layer_packed(const moe_packed_layer_t* layer, const float* x, int T, int rail, void* workspace,
                         size_t workspace_bytes, float* y, int32_t* ids_out, float* weights_out, float* h_out,
                         cudaStream_t stream);

/* Stages of the block-scaled decode rail (moe_ffn_layer_packed_stage, a bit mask). */
#define MOE_STAGE_PROLOGUE 1 /* router logits, x as E2M1 operand terms, counters zeroed */
#define MOE_STAGE_GATEUP 2   /* gate/up + bias + swiglu, the down operand written to the workspace */
#define MOE_STAGE_DOWN 4     /* down + bias + router-weighted combine into y */

/*
 * moe_ffn_layer_packed_stage -- the stages of moe_ffn_layer_packed on the
 * decode rail (T <= MOE_GEMV_MAX_T), selected by the bit mask `stages`, on the
 * same workspace: a stage reads what the earlier stages of the same workspace
 * left there (the prologue's logits, operand and zeroed counters; the gate/up
 * stage's down operand), so running them one call at a time in order equals
 * one moe_ffn_layer_packed call. The pages gate their fused chain against the
 * per-op composition ("dasLLAMA gpt-oss arc", fused MoE expert chain commit);
 * this is the per-stage view for tests and profiling. The gate/up and down
 * stages are launched as programmatic dependents of the work before them in
 * the stream. y is written by the down stage only; ids_out, weights_out and
 * h_out (each may be NULL) by the gate/up stage.
 */
int moe_ffn_layer_packed_stage(const moe_packed_layer_t* layer, const float* x, int T, void* workspace,
                               size_t workspace_bytes, int stages, float* y, int32_t* ids_out,
                               float* weights_out, float* h_out, cudaStream_t stream);

/*
 * moe_ffn_layer_packed_hostio -- moe_ffn_layer_packed for tokens in host
 * memory: x_host [T][D] in, y_host [T][D] out, one call per step. With pinned
 * (page-locked) buffers on the decode rail nothing is copied by the copy
 * engines: the prologue reads x through the pinned mapping and the down
 * kernel stores y into it; pageable buffers are staged through the workspace
 * with cudaMemcpyAsync. The call only enqueues: synchronise the stream before
 * reading y_host.
 */
int moe_ffn_layer_packed_hostio(const moe_packed_layer_t* layer, int T, int rail, void* workspace,
                                size_t workspace_bytes, const float* x_host, float* y_host, cudaStream_t stream);

/* Size of the library's static decode scratch (moe_ffn_layer_decode_static). */
#define MOE_DECODE_SCRATCH_BYTES (512 * 1024)

/*
 * moe_ffn_layer_decode_static -- moe_ffn_layer on the GEMV rail for callers
 * that cannot allocate device memory where they run the layer: a serving loop
 * that must stay allocation-free after start-up (cudaMalloc/cudaFree can
 * synchronise the device), or a plugin that is handed only a stream and
 * tensors. The pages have no counterpart; it is a deployment convenience.
 * Arguments, results and limits are those of moe_ffn_layer with
 * rail = MOE_RAIL_GEMV (1 <= T <= MOE_GEMV_MAX_T; T = 0 returns MOE_OK and
 * enqueues nothing); there is no workspace argument: the scratch is one
 * file-scope device array of MOE_DECODE_SCRATCH_BYTES bytes that every GPU
 * which loads the library holds until the process exits. Shapes whose
 * moe_ffn_workspace_bytes(T, D, F, E, k, MOE_RAIL_GEMV) exceeds that size are
 * rejected with MOE_ESCRATCH before anything is enqueued (T = 8, k = 4,
 * D = F = 2880 needs about 370 KB; T = 8, k = 8 at that width does not fit).
 * The first call on each device looks up the array's device address (with
 * that device current) and keeps it for the life of the process; do not use
 * the library across cudaDeviceReset. All calls on a device share the array and it keeps the last
 * call's contents; nothing in it needs to start at zero (every byte a call
 * reads it first writes). Calls whose executions overlap on the GPU (different
 * streams, or concurrent host threads) race on the array: serialise them.
 * Calls no cudaMalloc, cudaFree or allocating library routine.
 */
int moe_ffn_layer_decode_static(const float* x, int T, int D, int F, int E, int k,
                                const float* w_router, const float* b_router, const uint8_t* g_qs,
                                const uint8_t* g_sc, const float* bg, const uint8_t* u_qs,
                                const uint8_t* u_sc, const float* bu, const uint8_t* d_qs,
                                const uint8_t* d_sc, const float* bd, float* y, int32_t* ids_out,
                                float* weights_out, cudaStream_t stream);

/*
 * moe_checked_build -- 1 if this library was compiled with MOE_CHECKED
 * (libmoe_mxfp4_checked.so: the kernels check the indices they form from
 * routing, bucket and segment data against their buffers before each global
 * access or bulk copy and set MOE_STATUS_OUT_OF_BOUNDS instead of touching
 * memory outside them; a skipped copy still completes its pipeline stage, so
 * nothing waits on it), 0 for the regular build. Same ABI in both.
 */
int moe_checked_build(void);

/*
 * moe_get_status -- waits for `stream`, then reads and clears the calling
 * device's status word (MOE_STATUS_* bits set by kernels since the last
 * read) into *status. This is the one call that synchronises.
 */
int moe_get_status(cudaStream_t stream, int* status);

/*
 * moe_get_timeout_site -- waits for `stream`, then reads and clears the site of
 * the first pipeline wait that gave up on the calling device since the last
 * read (0: none): kernel << 24 | role << 20 | stage << 12 | sequence index,
 * kernel 1 = decode gate/up, 2 = decode down (GEMV rail), 3 = grouped GEMM
 * (bf16), 4 = grouped GEMM (block-scaled), 5 = decode gate/up, 6 = decode down
 * (block-scaled decode rail), 7 = gate/up, 8 = down (kind::mxf4 grouped rail);
 * role 0 = a producer waiting for a free stage, 1 = a consumer waiting for
 * data, 2 = an epilogue waiting for its accumulator (grouped GEMMs: the warp
 * index of the waiting role, 3 or 4 = the dequantising or expanding warps;
 * kind::mxf4 rail: 0 = a copy issuer waiting for a free stage, 1 = the MMA
 * thread, 2 = an epilogue warp, 3 = a scale loader waiting for data, 4 = a
 * scale loader and 5 = a copy issuer waiting for its next work unit). For
 * diagnosis only.
 */
int moe_get_timeout_site(cudaStream_t stream, int* site);

/*
 * moe_selftest_wait_timeout -- exercises the failure path of the bounded
 * pipeline waits without any fault: one CTA lands a 1 KB bulk copy from `src`
 * (device memory, 16-byte aligned, at least 1024 bytes, only read), holds 32
 * columns of tensor memory, and waits for an mbarrier that nothing arrives at.
 * After the wait limit (about 2 s) the kernel sets MOE_STATUS_WAIT_TIMEOUT in
 * the device status word with the site (15 << 24) | (2 << 20) (see
 * moe_get_timeout_site), waits for its copy, frees tensor memory and returns;
 * the context stays usable. Enqueued on `stream` only. Returns MOE_EINVAL for
 * a NULL or unaligned `src`.
 */
int moe_selftest_wait_timeout(const void* src, cudaStream_t stream);

/* moe_last_cuda_error -- the cudaError_t of the last MOE_ECUDA in this thread. */
int moe_last_cuda_error(void);

/* moe_kernel_launches -- number of kernels this library enqueued from this process (a counter). */
uint64_t moe_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_MXFP4_H */
