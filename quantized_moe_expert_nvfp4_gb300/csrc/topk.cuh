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

// 64-bit ranking key of entry e: the logit's key above, then the complemented index, so that a
// larger value means a preferred entry (larger logit, then lower index) and all keys differ.
__device__ __forceinline__ uint64_t rank_key(uint32_t key, int e) {
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(e));
}

__device__ __forceinline__ uint64_t shfl_u64(uint64_t v, int src) {
  const uint32_t lo = __shfl_sync(kFullMask, static_cast<uint32_t>(v), src);
  const uint32_t hi = __shfl_sync(kFullMask, static_cast<uint32_t>(v >> 32), src);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// Sorts one 64-bit value per lane across the warp, descending (lane 0 holds the largest): a
// bitonic network of shuffles.
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t v, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint64_t o = shfl_u64(v, lane ^ stride);
      // the lower lane of a pair keeps the larger value in a descending run, the smaller in an
      // ascending one; runs of `size` alternate so that the next merge sees bitonic sequences
      const bool lower = (lane & stride) == 0;
      const bool desc = (lane & size) == 0 || size == 32;
      const bool keep_max = lower == desc;
      v = keep_max ? (o > v ? o : v) : (o < v ? o : v);
    }
  }
  return v;
}

// One warp ranks one row of E logits (lane l holds entries l, l+32, ...).  Lane j < k receives
// the rank-j winner and its routing weight: the renormalised softmax over the k winners,
// w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0), the sum taken in rank order.  A row with no
// finite or +inf logit gets weights 0; +inf winners share the mass equally.
//
// Selection: with every entry's 64-bit rank key distinct, let tau be the k-th largest of the 32
// lanes' maxima; those k maxima are k entries at or above tau, so every one of the k winners is
// at or above tau too.  The entries at or above tau (usually about k of them) are moved to one
// lane each and sorted across the warp.  Should more than 32 entries reach tau (a few lanes
// holding most of the largest logits), the row is ranked by k rounds of warp-wide maxima instead.
// Both ways give the same order.
template <int EPL>
__device__ __forceinline__ void warp_topk(const float* __restrict__ row, int E, int k, int lane,
                                          int& my_id, float& my_w) {
  // 32-bit logit keys held per lane (0 past E: a real entry's key is at least that of -inf,
  // 0x007fffff); the 64-bit rank key of entry lane + 32 i is formed when needed
  uint32_t kv[EPL];
  uint64_t lmax = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    kv[i] = (e < E) ? logit_key(__ldg(row + e)) : 0u;
  }
  auto key = [&](int i) -> uint64_t { return kv[i] ? rank_key(kv[i], lane + 32 * i) : 0ull; };
#pragma unroll
  for (int i = 0; i < EPL; ++i) lmax = key(i) > lmax ? key(i) : lmax;
  const uint64_t tau = shfl_u64(warp_sort_desc(lmax, lane), k - 1);
  uint32_t cand = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if (key(i) >= tau && kv[i] != 0u) cand |= 1u << i;
  const int c = __popc(cand);
  int incl = c;   // inclusive prefix of the candidate counts over the lanes
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(kFullMask, incl, off);
    if (lane >= off) incl += y;
  }
  const int total = __shfl_sync(kFullMask, incl, 31);
  uint64_t mine = 0;   // the rank-lane entry after the sort
  if (total <= 32) {
    // lane j takes candidate j: the source lane L is the first with incl > j, the entry the
    // (j - (incl_L - c_L))-th set bit of L's candidate mask
    int src = 0;
#pragma unroll
    for (int step = 16; step > 0; step >>= 1) {
      const int probe = __shfl_sync(kFullMask, incl, src + step - 1);
      if (probe <= lane) src += step;
    }
    const int src_incl = __shfl_sync(kFullMask, incl, src);
    const int src_c = __shfl_sync(kFullMask, c, src);
    const uint32_t src_mask = __shfl_sync(kFullMask, cand, src);
    const int r = lane - (src_incl - src_c);
    const int want = (lane < total) ? __fns(src_mask, 0, r + 1) : -1;
    uint64_t got = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const uint64_t v = shfl_u64(key(i), src);
      if (i == want) got = v;
    }
    mine = warp_sort_desc(got, lane);
  } else {
    uint32_t taken = 0;
    for (int j = 0; j < k; ++j) {
      uint64_t best = 0;
      int bi = 0;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        if (!((taken >> i) & 1u) && key(i) > best) {
          best = key(i);
          bi = i;
        }
      }
      const uint32_t hi = __reduce_max_sync(kFullMask, static_cast<uint32_t>(best >> 32));
      const uint32_t lo = __reduce_max_sync(kFullMask, static_cast<uint32_t>(best >> 32) == hi
                                                           ? static_cast<uint32_t>(best) : 0u);
      const uint64_t w = (static_cast<uint64_t>(hi) << 32) | lo;
      if (best == w && best != 0ull) taken |= 1u << bi;
      if (lane == j) mine = w;
    }
  }
  my_id = -1;
  float my_val = -INFINITY;
  if (lane < k) {
    my_id = static_cast<int>(~static_cast<uint32_t>(mine));
    my_val = key_value(static_cast<uint32_t>(mine >> 32));
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
