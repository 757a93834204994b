// Warp-level top-k over one token's router logits, with the selected-only
// softmax ("Qwen creates three distinct workload shapes": the router scores
// every expert and selects k; the weights are a softmax over all experts
// renormalised over the selected ones, which equals a softmax over the
// selected logits).  Used by the prefill routing and by the decode kernel.
#pragma once
#include "moe_common.cuh"

namespace moe {

// Order-preserving 32-bit key of a logit (-0 folded into +0 so that equal
// values compare equal, as floats do).
__device__ __forceinline__ uint32_t logit_key(float v) {
  const uint32_t u = __float_as_uint(v + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Top-k of the E logits (lane l holds experts l + 32 r in v[r]) in the order
// larger logit first, equal logits -> lower expert first; then the weights
// softmax(selected logits), which equal the softmax over all E logits
// renormalised over the selection ("Qwen creates three distinct workload
// shapes").  Lane j < k receives selection j: expert sel_e and weight sel_w.
// Each round takes the warp maximum of the lanes' best keys and the lowest
// expert holding it with two redux.sync reductions; every lane computes the
// same result.
template <int R>
__device__ __forceinline__ void warp_topk_redux(const float (&v)[R], int E, int k, int &sel_e,
                                                float &sel_w) {
  const int lane = threadIdx.x & 31;
  uint32_t key[R];
#pragma unroll
  for (int r = 0; r < R; ++r) key[r] = (lane + 32 * r < E) ? logit_key(v[r]) : 0u;
  uint32_t sel_key = 0;
  sel_e = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = key[0];
    int br = 0;
#pragma unroll
    for (int r = 1; r < R; ++r)
      if (key[r] > bk) {
        bk = key[r];
        br = r;
      }
    const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t e = __reduce_min_sync(0xffffffffu, bk == m ? static_cast<uint32_t>(lane + 32 * br)
                                                              : 0xffffffffu);
#pragma unroll
    for (int r = 0; r < R; ++r)
      key[r] = (e == static_cast<uint32_t>(lane + 32 * r)) ? 0u : key[r];
    if (lane == j) {
      sel_key = m;
      sel_e = static_cast<int>(e);
    }
  }
  const float sv = key_logit(sel_key);
  const float vmax = __shfl_sync(0xffffffffu, sv, 0);
  const float ex = (lane < k) ? expf(sv - vmax) : 0.0f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  sel_w = ex / sum;
}

}  // namespace moe
