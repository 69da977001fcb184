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

// Lane l's logits of a row of E (entries l, l + 32, ...; 0 past the end).
template <int EPL>
__device__ __forceinline__ void warp_load_logits(const float* __restrict__ row, int E, int lane, float (&v)[EPL]) {
#pragma unroll
  for (int i = 0; i < EPL; ++i) v[i] = (lane + 32 * i < E) ? __ldg(row + lane + 32 * i) : 0.0f;
}

// Threshold selection of the k winners of a warp's row (keys as in warp_topk_vals, padding keys 0
// and marked in `taken`), into lanes j < k (my_id, my_val).  The k-th largest of the 32 lane
// maxima, tau, is at most the row's k-th largest key (the k lanes whose maxima reach tau hold k
// entries of at least tau), so every winner is among the entries with key >= tau -- usually a
// little over k of them.  Those candidates are written to the warp's 32-entry scratch, each
// counts the candidates that precede it in (key descending, index ascending) order, which is its
// rank, and the first k ranks are read back.  Returns false, with nothing selected, when fewer
// than k or more than 32 entries reach tau (many equal keys, or fewer than k entries).
template <int EPL>
__device__ __forceinline__ bool warp_select_threshold(const uint32_t (&key)[EPL], uint32_t taken, int k, int lane,
                                                      uint2* scratch, int& my_id, float& my_val) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i) m = max(m, key[i]);
  uint32_t tau = 0;
  for (int j = 0; j < k; ++j) {   // remove the largest lane maximum k times (lowest lane first)
    tau = __reduce_max_sync(kFullMask, m);
    const uint32_t l = __reduce_min_sync(kFullMask, m == tau ? static_cast<uint32_t>(lane) : 32u);
    if (static_cast<uint32_t>(lane) == l) m = 0;
  }
  uint32_t cm = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if (!((taken >> i) & 1u) && key[i] >= tau) cm |= 1u << i;
  const int c = __popc(cm);
  int incl = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(kFullMask, incl, off);
    if (lane >= off) incl += y;
  }
  const int C = __shfl_sync(kFullMask, incl, 31);
  if (C < k || C > 32) return false;
  int pos = incl - c;
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if ((cm >> i) & 1u) scratch[pos++] = make_uint2(key[i], static_cast<uint32_t>(lane + 32 * i));
  __syncwarp();
  uint2 me = make_uint2(0u, 0u);
  if (lane < C) me = scratch[lane];
  int rank = 0;
  for (int q = 0; q < C; ++q) {
    const uint2 o = scratch[q];
    rank += (o.x > me.x || (o.x == me.x && o.y < me.y)) ? 1 : 0;
  }
  __syncwarp();
  if (lane < C && rank < k) scratch[rank] = me;
  __syncwarp();
  if (lane < k) {
    const uint2 wv = scratch[lane];
    my_id = static_cast<int>(wv.y);
    my_val = key_value(wv.x);
  }
  __syncwarp();   // the scratch is free for the warp's next row
  return true;
}

// One warp ranks one row of E logits (lane l holds entries l, l+32, ...).  Lane j < k receives
// the rank-j winner and its routing weight: the renormalised softmax over the k winners,
// w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0), the sum taken in rank order.  A row with no
// finite or +inf logit gets weights 0; +inf winners share the mass equally.  With a 32-entry
// shared-memory scratch for the warp the winners come from warp_select_threshold; without one,
// or when it declines, from k rounds that each take the largest remaining key (lowest index
// among equal keys) -- the same winners in the same order.
template <int EPL>
__device__ __forceinline__ void warp_topk_vals(const float (&v)[EPL], int E, int k, int lane, int& my_id,
                                               float& my_w, uint2* scratch = nullptr) {
  uint32_t key[EPL];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    key[i] = (e < E) ? logit_key(v[i]) : 0u;
    if (e >= E) taken |= 1u << i;
  }
  my_id = -1;
  float my_val = -INFINITY;
  const bool selected = scratch && warp_select_threshold<EPL>(key, taken, k, lane, scratch, my_id, my_val);
  for (int j = 0; !selected && j < k; ++j) {
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

// The same, loading the row first.
template <int EPL>
__device__ __forceinline__ void warp_topk(const float* __restrict__ row, int E, int k, int lane, int& my_id,
                                          float& my_w, uint2* scratch = nullptr) {
  float v[EPL];
  warp_load_logits<EPL>(row, E, lane, v);
  warp_topk_vals<EPL>(v, E, k, lane, my_id, my_w, scratch);
}


}  // namespace moe
