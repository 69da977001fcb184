// Warp-level router top-k shared by the routing kernels.
//
// Ranking follows the "handover briefs" page's device-side selection rule: entries ordered by
// (value descending, index ascending), a NaN never wins (it counts as -inf), and -0 ties +0.
#pragma once

#include "internal.cuh"

namespace moe {

constexpr unsigned kFullMask = 0xffffffffu;

// Order-preserving 32-bit key of a logit: larger key = preferred.  NaN counts as -inf and
// -0 equals +0, so equal logits tie and the lower index wins.
__device__ __forceinline__ uint32_t logit_key(float x) {
  if (isnan(x)) x = -INFINITY;
  if (x == 0.0f) x = 0.0f;
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// One warp ranks one row of E logits (lane l holds entries l, l+32, ...).  Lane j < k receives
// the rank-j winner and its routing weight: the renormalised softmax over the k winners,
// w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0), the sum taken in rank order.  A row with no
// finite or +inf logit gets weights 0; +inf winners share the mass equally.
template <int EPL>
__device__ __forceinline__ void warp_topk(const float* __restrict__ row, int E, int k, int lane,
                                          int& my_id, float& my_w) {
  uint32_t key[EPL];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    key[i] = (e < E) ? logit_key(__ldg(row + e)) : 0u;
    if (e >= E) taken |= 1u << i;
  }
  my_id = -1;
  float my_val = -INFINITY;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0u;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      if (!((taken >> i) & 1u) && key[i] > bk) {  // within a lane indices increase with i
        bk = key[i];
        be = lane + 32 * i;
      }
    }
    // the warp's winner: the largest key, and among lanes holding it the smallest index (two
    // warp-wide reductions)
    const uint32_t wk = __reduce_max_sync(kFullMask, bk);
    be = static_cast<int>(__reduce_min_sync(kFullMask, bk == wk ? static_cast<uint32_t>(be) : 0xffffffffu));
    bk = wk;
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == j) {
      my_id = be;
      my_val = key_value(bk);
    }
  }
  const float m = __shfl_sync(kFullMask, my_val, 0);
  const bool live = lane < k;
  float ev;
  if (m == -INFINITY) {
    ev = 0.0f;
  } else if (m == INFINITY) {
    ev = (live && my_val == INFINITY) ? 1.0f : 0.0f;
  } else {
    ev = live ? expf(my_val - m) : 0.0f;
  }
  float sum = 0.0f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(kFullMask, ev, j);
  my_w = (sum > 0.0f) ? ev / sum : 0.0f;
}


}  // namespace moe
