// Warp-level top-k over one token's router logits, with the selected-only
// softmax ("Qwen creates three distinct workload shapes": the router scores
// every expert and selects k; the weights are a softmax over all experts
// renormalised over the selected ones, which equals a softmax over the
// selected logits).
#pragma once
#include <cfloat>
#include <climits>
#include "moe_common.cuh"

namespace moe {

// Total order used for selection: larger logit first, equal logits -> lower
// expert index first.  `eb == INT_MAX` marks "no candidate".
__device__ __forceinline__ bool topk_better(float va, int ea, float vb, int eb) {
  return (va > vb) || (va == vb && ea < eb);
}

// Lane l holds logits of experts l, l+32, ... (v[r] for expert l + 32r).
// After the call, lane j < k holds the j-th selection (value, expert) and
// its renormalised weight.  Deterministic: the reductions are fixed
// butterflies, every lane computes the same result.
template <int R>
__device__ __forceinline__ void warp_topk(const float (&v)[R], int E, int k, float &sel_v,
                                          int &sel_e, float &sel_w) {
  const int lane = threadIdx.x & 31;
  uint32_t taken = 0;
#pragma unroll
  for (int r = 0; r < R; ++r)
    if (lane + 32 * r >= E) taken |= 1u << r;
  sel_v = -FLT_MAX;
  sel_e = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = INT_MAX;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int e = lane + 32 * r;
      if (!((taken >> r) & 1u) && topk_better(v[r], e, bv, be)) {
        bv = v[r];
        be = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (topk_better(ov, oe, bv, be)) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == j) {
      sel_v = bv;
      sel_e = be;
    }
  }
  const float vmax = __shfl_sync(0xffffffffu, sel_v, 0);
  const float ex = (lane < k) ? expf(sel_v - vmax) : 0.0f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  sel_w = ex / sum;
}

}  // namespace moe
