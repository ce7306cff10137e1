// Routing table of the decode rails (T <= 8 tokens): top-k + softmax of the
// router logits (or given ids), the active experts in ascending order, and
// each expert's assignments. Built in shared memory by one warp per CTA.
#pragma once

#include "moe_common.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Routing table, built in shared memory by one warp per CTA from the router
// logits (top-k + softmax, the same routine as moe_route_topk) or from given
// ids: the active experts in ascending order and, per expert, its assignments
// a = t*k + j in ascending order. T*k <= 64.
// ---------------------------------------------------------------------------
constexpr int kMaxAssign = 64;

struct DecodeRouting {
  int nact;
  int act_e[kMaxAssign];
  int act_off[kMaxAssign + 1];
  int lst[kMaxAssign];
  int ids[kMaxAssign];
  float w[kMaxAssign];
  int lead[kMaxAssign];  // 1 if the assignment is the first of its expert
};

// One warp, from R.ids[0..TK): lane l holds assignments l and l + 32. An
// assignment's place in the expert-major list is the number of valid ids below
// its own plus the number of equal ids before it; the first assignment of each
// expert (its leader) also fixes the expert's index, the number of leaders
// with a smaller id. Every lane reads the id list with broadcast shared loads.
__device__ __forceinline__ void build_routing(DecodeRouting& R, int TK, int E, int lane, int* status) {
  const int e0 = lane < TK ? R.ids[lane] : -1;
  const int e1 = lane + 32 < TK ? R.ids[lane + 32] : -1;
  const bool v0 = e0 >= 0 && e0 < E, v1 = e1 >= 0 && e1 < E;
  if ((lane < TK && !v0) || (lane + 32 < TK && !v1)) set_status(status, 0x1);
  int less0 = 0, less1 = 0, rank0 = 0, rank1 = 0;
#pragma unroll 4
  for (int bb = 0; bb < TK; ++bb) {
    const int eb = R.ids[bb];
    const bool vb = eb >= 0 && eb < E;
    less0 += vb && eb < e0;
    less1 += vb && eb < e1;
    rank0 += vb && (eb == e0) && (bb < lane);
    rank1 += vb && (eb == e1) && (bb < lane + 32);
  }
  const bool lead0 = v0 && rank0 == 0, lead1 = v1 && rank1 == 0;
  if (lane < TK) R.lead[lane] = lead0;
  if (lane + 32 < TK) R.lead[lane + 32] = lead1;
  __syncwarp();
  int ix0 = 0, ix1 = 0, nact = 0, nvalid = 0;
#pragma unroll 4
  for (int bb = 0; bb < TK; ++bb) {
    const int eb = R.ids[bb];
    const int lb = R.lead[bb];
    ix0 += lb && eb < e0;
    ix1 += lb && eb < e1;
    nact += lb;
    nvalid += eb >= 0 && eb < E;
  }
  if (v0) R.lst[less0 + rank0] = lane;
  if (v1) R.lst[less1 + rank1] = lane + 32;
  if (lead0) {
    R.act_e[ix0] = e0;
    R.act_off[ix0] = less0;
  }
  if (lead1) {
    R.act_e[ix1] = e1;
    R.act_off[ix1] = less1;
  }
  if (lane == 0) {
    R.nact = nact;
    R.act_off[nact] = nvalid;
  }
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

}  // namespace moe
