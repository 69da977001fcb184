// Router top-k and token permutation, built entirely on the device.
//
// Routing follows the layer statement of the "long-context cold prefill to SGLang parity"
// issue (router top-k ids and weights among the op-dump tensors) with the selection rule of
// the "handover briefs" page's device-side indexer selection: rank an entry by (value desc,
// index asc), a NaN never wins.  The permutation is the issue's "token permutation": slots
// grouped by expert, stable in slot order, with counts and exclusive prefix offsets, computed
// here by warp-level match/scan so that nothing returns to the host.
#include <algorithm>

#include "internal.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

template <int EPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T,
                                                         int E, int k, int32_t* __restrict__ ids,
                                                         float* __restrict__ w) {
  __shared__ uint2 s_topk[8][32];   // each warp's top-k scratch
  pdl_wait_then_release();
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  int my_id;
  float my_w;
  warp_topk<EPL>(logits + static_cast<int64_t>(t) * E, E, k, lane, my_id, my_w, s_topk[threadIdx.x >> 5]);
  if (lane < k) {
    ids[static_cast<int64_t>(t) * k + lane] = my_id;
    w[static_cast<int64_t>(t) * k + lane] = my_w;
  }
}

// Exclusive scan over blockDim.x (<= 1024, multiple of 32) values, one per thread.
__device__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(kFull, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = (lane < nw) ? s_warp[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(kFull, s, off);
      if (lane >= off) s += y;
    }
    if (lane < nw) s_warp[lane] = s;  // inclusive warp prefix
  }
  __syncthreads();
  const int base = (warp > 0) ? s_warp[warp - 1] : 0;
  const int tot = s_warp[nw - 1];
  __syncthreads();
  if (total) *total = tot;
  return base + x - v;
}

// Work list: for each group with rows, ceil(rows / tile_rows) items {g, row_begin, rows, 0};
// routed groups first (ascending expert), then the shared group (rows S .. S+T-1).  Called by
// one whole block of >= E threads; cnt(e) / off(e) come from the caller (shared memory), and
// s_base (E entries of shared memory the caller no longer reads) receives each expert's first
// item.  The items are written by all threads in parallel, item j by thread j mod blockDim: its
// expert is the last one whose first item is at most j (an expert without rows shares its first
// item with the next), so one busy expert's many items do not fall to one thread.
__device__ void write_tiles_block(int E, int S, int T, int has_shared, int tile_rows,
                                  const int* cnt_of, const int* off_of, int4* tiles,
                                  int32_t* meta, int* s_warp, int* s_base) {
  const int e = threadIdx.x;
  const int c = (e < E) ? cnt_of[e] : 0;
  const int n = (c + tile_rows - 1) / tile_rows;
  int total = 0;
  const int base = block_exclusive_scan(n, s_warp, &total);
  if (e < E) s_base[e] = base;
  __syncthreads();
  for (int j = threadIdx.x; j < total; j += blockDim.x) {
    int lo = 0, hi = E - 1;   // the last expert whose first item is <= j
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_base[mid] <= j) lo = mid;
      else hi = mid - 1;
    }
    const int r0 = (j - s_base[lo]) * tile_rows;
    tiles[j] = make_int4(lo, off_of[lo] + r0, min(tile_rows, cnt_of[lo] - r0), 0);
  }
  const int n_shared = has_shared ? (T + tile_rows - 1) / tile_rows : 0;
  for (int i = threadIdx.x; i < n_shared; i += blockDim.x) {
    const int r0 = i * tile_rows;
    tiles[total + i] = make_int4(E, S + r0, min(tile_rows, T - r0), 0);
  }
  if (threadIdx.x == 0) meta[0] = total + n_shared;
}

// Stable placement of n consecutive slots [s0, s0 + n) by one warp: every slot gets
// cursor[e] + (number of earlier slots of the same expert in this run); the cursors advance.
__device__ __forceinline__ void warp_stable_scatter(const int32_t* ids, int s0, int n, int E,
                                                    int* cursor, int32_t* sorted_slot,
                                                    int32_t* slot_pos) {
  constexpr int kBatch = 4;   // 32-slot steps whose ids are loaded together, ahead of their use
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  for (int b0 = 0; b0 < n; b0 += 32 * kBatch) {
    int ev[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) ev[j] = (b0 + 32 * j + lane < n) ? ids[s0 + b0 + 32 * j + lane] : -1;
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int b = b0 + 32 * j;
      if (b >= n) break;
      const int s = s0 + b + lane;
      int e = ev[j];
      if (e >= E) e = -2;  // out-of-range ids are ignored (the caller validated them)
      const unsigned grp = __match_any_sync(kFull, e);
      const int rank = __popc(grp & lt);
      if (e >= 0) {
        const int pos = cursor[e] + rank;
        sorted_slot[pos] = s;
        slot_pos[s] = pos;
      }
      __syncwarp();
      if (e >= 0 && rank == 0) cursor[e] += __popc(grp);
      __syncwarp();
    }
  }
}

// Decode arm: routing (or given ids), counts, offsets, stable permutation and the work list of
// a small batch in a single CTA of 1024 threads.
template <int EPL>
__global__ void __launch_bounds__(1024) route_permute_small_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ ids_in, int T, int E, int k,
    int has_shared, int32_t* __restrict__ ids, float* __restrict__ w, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_slot,
    int32_t* __restrict__ slot_pos, int4* __restrict__ tiles, int32_t* __restrict__ meta,
    int tile_rows) {
  __shared__ int s_ids[kDecodeMaxT * kMaxK];
  __shared__ uint2 s_topk[32][32];   // each warp's top-k scratch
  __shared__ int s_cnt[kMaxE];
  __shared__ int s_off[kMaxE];
  __shared__ int s_cur[kMaxE];
  __shared__ int s_warp[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int S = T * k;

  if (logits) {
    for (int t = warp; t < T; t += 32) {
      int my_id;
      float my_w;
      // (the threshold selection's registers do not fit 1024-thread blocks above 512 experts)
      warp_topk<EPL>(logits + static_cast<int64_t>(t) * E, E, k, lane, my_id, my_w, EPL <= 16 ? s_topk[warp] : nullptr);
      if (lane < k) {
        ids[t * k + lane] = my_id;
        w[t * k + lane] = my_w;
        s_ids[t * k + lane] = my_id;
      }
    }
  } else {
    for (int s = threadIdx.x; s < S; s += blockDim.x) s_ids[s] = ids_in[s];
  }
  for (int e = threadIdx.x; e < kMaxE; e += blockDim.x) {
    s_cnt[e] = 0;
    s_cur[e] = 0;
  }
  __syncthreads();
  for (int s = threadIdx.x; s < S; s += blockDim.x) {
    const int e = s_ids[s];
    if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  const int my = (threadIdx.x < E) ? s_cnt[threadIdx.x] : 0;
  const int off = block_exclusive_scan(my, s_warp, nullptr);
  if (threadIdx.x < E) {
    s_off[threadIdx.x] = off;
    s_cur[threadIdx.x] = off;
    counts[threadIdx.x] = my;
    offsets[threadIdx.x] = off;
  }
  if (threadIdx.x == 0) offsets[E] = S;
  __syncthreads();
  if (warp == 0) warp_stable_scatter(s_ids, 0, S, E, s_cur, sorted_slot, slot_pos);
  // (s_cur is free once the work list's scan has passed its barriers: warp 0 has placed every slot)
  write_tiles_block(E, S, T, has_shared, tile_rows, s_cnt, s_off, tiles, meta, s_warp, s_cur);
}

// Batched decode on the tensor-core arm (T <= kDecodeMaxT), after the top-k: permutation, work
// list and the expert-ordered f16 rows of x in one launch with no grid-wide wait.  Every CTA reads
// the batch's S = T k expert ids, builds the counts, offsets and the stable placement in shared
// memory, and then converts its share of the tokens (token b, b + gridDim, ...): each x row is read
// once, scaled by 2^-e (e = floor(log2 max|row|) - 14, at least -126) and written as f16 to the k
// expert-ordered rows that hold the token and to the shared expert's row S + t, with the factor
// 2^e per row -- the rows act_scatter_f16 writes.  CTA 0 also writes the permutation and the work
// list for the later stages.
__global__ void __launch_bounds__(1024) permute_gather_small_kernel(
    const int32_t* __restrict__ ids, const uint16_t* __restrict__ x, int T, int E, int k, int has_shared, int H,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_slot,
    int32_t* __restrict__ slot_pos, int4* __restrict__ tiles, int32_t* __restrict__ meta, int tile_rows,
    uint16_t* __restrict__ xf, float* __restrict__ xe, int32_t* __restrict__ status) {
  constexpr int kPlaceWarps = 4;   // warps placing the batch's slots, a contiguous chunk each
  __shared__ int s_ids[kDecodeMaxT * kMaxK];
  __shared__ int s_pos[kDecodeMaxT * kMaxK];
  __shared__ int s_cnt[kMaxE];
  __shared__ int s_off[kMaxE];
  __shared__ int s_cur[kMaxE];
  __shared__ int s_wc[kPlaceWarps * kMaxE];   // per-warp expert counts, then per-warp cursors
  __shared__ int s_warp[32];
  __shared__ float s_max[32];
  pdl_wait_then_release();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool lead = blockIdx.x == 0;
  const int S = T * k;
  for (int s = threadIdx.x; s < S; s += blockDim.x) {
    int e = __ldg(ids + s);
    if (e < 0 || e >= E) {   // written by the library's top-k; a bad value is reported and clamped
      if (lead) report_device_error(status, kDevBadIndex);
      e = 0;
    }
    s_ids[s] = e;
  }
  for (int e = threadIdx.x; e < kMaxE; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  for (int s = threadIdx.x; s < S; s += blockDim.x) atomicAdd(&s_cnt[s_ids[s]], 1);
  __syncthreads();
  const int my = (threadIdx.x < E) ? s_cnt[threadIdx.x] : 0;
  const int off = block_exclusive_scan(my, s_warp, nullptr);
  if (threadIdx.x < E) {
    s_off[threadIdx.x] = off;
    s_cur[threadIdx.x] = off;
    if (lead) {
      counts[threadIdx.x] = my;
      offsets[threadIdx.x] = off;
    }
  }
  if (lead && threadIdx.x == 0) offsets[E] = S;
  __syncthreads();
  // stable placement by kPlaceWarps warps, each a contiguous chunk of the slots: every warp counts
  // its chunk per expert, each expert's offset is split into per-warp cursors in chunk order, and
  // the warps place their chunks 32 slots a step (a slot goes after the earlier slots of its
  // expert)
  const int chunk = (S + kPlaceWarps - 1) / kPlaceWarps;
  const int c0 = min(S, warp * chunk), c1 = min(S, c0 + chunk);
  for (int i = threadIdx.x; i < kPlaceWarps * E; i += blockDim.x) s_wc[i] = 0;
  __syncthreads();
  if (warp < kPlaceWarps)
    for (int i = c0 + lane; i < c1; i += 32) atomicAdd(&s_wc[warp * E + s_ids[i]], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = s_cur[e];
    for (int w2 = 0; w2 < kPlaceWarps; ++w2) {
      const int cw = s_wc[w2 * E + e];
      s_wc[w2 * E + e] = run;
      run += cw;
    }
  }
  __syncthreads();
  if (warp < kPlaceWarps && c1 > c0) {
    int* cur = s_wc + warp * E;
    const unsigned lt = (1u << lane) - 1u;
    for (int b = c0; b < c1; b += 32) {
      const int s = b + lane;
      const int e = (s < c1) ? s_ids[s] : -1;
      const unsigned same = __match_any_sync(kFull, e);
      const int rank = __popc(same & lt);
      if (e >= 0) {
        const int pos = cur[e] + rank;
        s_pos[s] = pos;
        if (lead) {
          sorted_slot[pos] = s;
          slot_pos[s] = pos;
        }
      }
      __syncwarp();
      if (e >= 0 && rank == 0) cur[e] += __popc(same);
      __syncwarp();
    }
  }
  // (s_cur is free: the placement reads its per-warp cursors)
  if (lead) write_tiles_block(E, S, T, has_shared, tile_rows, s_cnt, s_off, tiles, meta, s_warp, s_cur);
  __syncthreads();
  // this CTA's tokens: f16 rows scaled by the row's power of two, to every row that holds the token
  const int nv = H / 8;   // 16-byte columns of a row
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * H);
    float m = 0.0f;
    for (int c = threadIdx.x; c < nv; c += blockDim.x) {
      const uint4 v = __ldg(src + c);
      const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        m = fmaxf(m, fabsf(__uint_as_float(q[i] << 16)));
        m = fmaxf(m, fabsf(__uint_as_float(q[i] & 0xffff0000u)));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    if (lane == 0) s_max[warp] = m;
    __syncthreads();
    m = (lane < static_cast<int>(blockDim.x >> 5)) ? s_max[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    const int ex = (m > 0.0f && m <= 3.4e38f) ? max(ilogbf(m) - 14, -126) : 0;
    const float inv = __int_as_float((127 - ex) << 23);
    if (threadIdx.x <= k) xe[threadIdx.x < k ? s_pos[t * k + threadIdx.x] : S + t] = __int_as_float((127 + ex) << 23);
    for (int c = threadIdx.x; c < nv; c += blockDim.x) {
      const uint4 v = __ldg(src + c);
      const uint32_t q[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 h = __floats2half2_rn(__uint_as_float(q[i] << 16) * inv, __uint_as_float(q[i] & 0xffff0000u) * inv);
        o[i] = *reinterpret_cast<const uint32_t*>(&h);
      }
      const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
      for (int j = 0; j <= k; ++j) {
        const int64_t p = (j < k) ? s_pos[t * k + j] : S + t;
        reinterpret_cast<uint4*>(xf + p * H)[c] = ov;
      }
    }
    __syncthreads();   // s_max is reused by the next token
  }
}

constexpr int kScatterWarps = 8;   // warps placing a CTA's slots in the cooperative permutation

// Any T, one cooperative launch of up to kPermuteMaxGrid CTAs of 1024 threads: routing (or given
// ids), per-CTA expert histograms of contiguous token ranges, a grid-wide barrier, every CTA's
// stable placement base per expert (the histograms of the CTAs before it plus the expert's
// offset), the stable scatter of its range, and (CTA 0) the work list.  The barrier is a
// monotonic 64-bit arrival counter in the workspace (every launch on a workspace uses the same
// grid), waited for with a bound.
__device__ __forceinline__ uint64_t rp_now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

template <int EPL>
__global__ void __launch_bounds__(1024, 1) route_permute_large_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ ids_in, int T, int E, int k,
    int has_shared, int32_t* __restrict__ ids, float* __restrict__ w, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_slot, int32_t* __restrict__ slot_pos,
    int32_t* __restrict__ hist, int4* __restrict__ tiles, int32_t* __restrict__ meta, int tile_rows,
    unsigned long long* __restrict__ bar, int32_t* __restrict__ status) {
  __shared__ int s_cnt[kMaxE];   // this CTA's histogram, then its placement cursors
  // routing: each warp's top-k scratch; placement: per-warp expert counts, then cursors
  __shared__ __align__(16) unsigned char s_raw[kScatterWarps * kMaxE * sizeof(int)];
  uint2 (*s_topk)[32] = reinterpret_cast<uint2 (*)[32]>(s_raw);
  __shared__ int s_tot[kMaxE];   // expert counts (for the work list)
  __shared__ int s_off[kMaxE];   // expert offsets
  __shared__ int s_warp[32];
  __shared__ int s_ok;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int S = T * k, G = gridDim.x, b = blockIdx.x;
  const int per = (T + G - 1) / G;
  const int t0 = min(T, b * per), t1 = min(T, t0 + per);
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  // routing of this CTA's tokens (warp per token) and its histogram
  if (logits) {
    for (int t = t0 + warp; t < t1; t += 32) {
      int my_id;
      float my_w;
      // (the threshold selection's registers do not fit 1024-thread blocks above 512 experts)
      warp_topk<EPL>(logits + static_cast<int64_t>(t) * E, E, k, lane, my_id, my_w, EPL <= 16 ? s_topk[warp] : nullptr);
      if (lane < k) {
        ids[static_cast<int64_t>(t) * k + lane] = my_id;
        w[static_cast<int64_t>(t) * k + lane] = my_w;
        atomicAdd(&s_cnt[my_id], 1);
      }
    }
  } else {
    for (int64_t s = static_cast<int64_t>(t0) * k + threadIdx.x; s < static_cast<int64_t>(t1) * k; s += blockDim.x) {
      const int e = ids_in[s];
      if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
      else report_device_error(status, kDevBadIndex);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[static_cast<int64_t>(b) * E + e] = s_cnt[e];
  // grid-wide barrier (all histograms written)
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned long long old = atomicAdd(bar, 1ull);
    const unsigned long long target = (old / G + 1) * G;
    const uint64_t ts = rp_now_ns();
    int ok = 1;
    for (uint32_t i = 0;; ++i) {
      unsigned long long v;
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(bar) : "memory");
      if (v >= target) break;
      if ((i & 63u) == 63u && rp_now_ns() - ts > 1000000000ull) {
        report_device_error(status, kDevTimeout);
        ok = 0;
        break;
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  if (!s_ok) return;
  // counts, offsets and this CTA's bases: column e of the histograms (of the CTAs that own
  // tokens: with T < G the others' are zero) summed by thread e, or, when the block has two
  // threads per expert, by threads e and E + e over the two halves of the CTAs
  const int e = threadIdx.x;
  const int g_used = per > 0 ? (T + per - 1) / per : 0;
  const bool split = 2 * E <= static_cast<int>(blockDim.x);
  const int col = (split && e >= E) ? e - E : e;
  const int c_lo = (split && e >= E) ? g_used / 2 : 0;
  const int c_hi = (split && e < E) ? g_used / 2 : g_used;
  int before = 0, total = 0;
  if (col < E) {
#pragma unroll 8
    for (int c = c_lo; c < c_hi; ++c) {
      const int v = __ldcg(hist + static_cast<int64_t>(c) * E + col);
      total += v;
      before += (c < b) ? v : 0;
    }
  }
  if (split) {
    if (e >= E && col < E) {
      s_tot[col] = total;
      s_off[col] = before;
    }
    __syncthreads();
    if (e < E) {
      total += s_tot[e];
      before += s_off[e];
    }
    __syncthreads();
  }
  const int off = block_exclusive_scan(e < E ? total : 0, s_warp, nullptr);
  if (e < E) {
    s_cnt[e] = off + before;
    s_tot[e] = total;
    s_off[e] = off;
    if (b == 0) {
      counts[e] = total;
      offsets[e] = off;
    }
  }
  if (b == 0 && threadIdx.x == 0) offsets[E] = S;
  __syncthreads();
  // stable placement of the CTA's slots (its own ids, written above or given) by kScatterWarps
  // warps, each a contiguous chunk: every warp counts its chunk's slots per expert, each expert's
  // cursor is split into per-warp cursors in chunk order, and the warps place their chunks
  {
    const int32_t* src = logits ? ids : ids_in;
    const int s_begin = t0 * k, n_sl = (t1 - t0) * k;
    const int chunk = (n_sl + kScatterWarps - 1) / kScatterWarps;
    const int c0 = min(n_sl, warp * chunk), c1 = min(n_sl, c0 + chunk);
    int* wc = reinterpret_cast<int*>(s_raw);   // [kScatterWarps][E]
    for (int i = threadIdx.x; i < kScatterWarps * E; i += blockDim.x) wc[i] = 0;
    __syncthreads();
    if (warp < kScatterWarps) {
      for (int i = c0 + lane; i < c1; i += 32) {
        const int ex = src[s_begin + i];
        if (ex >= 0 && ex < E) atomicAdd(&wc[warp * E + ex], 1);
      }
    }
    __syncthreads();
    for (int ex = threadIdx.x; ex < E; ex += blockDim.x) {
      int run = s_cnt[ex];
      for (int w2 = 0; w2 < kScatterWarps; ++w2) {
        const int cw = wc[w2 * E + ex];
        wc[w2 * E + ex] = run;
        run += cw;
      }
    }
    __syncthreads();
    if (warp < kScatterWarps && c1 > c0)
      warp_stable_scatter(src, s_begin + c0, c1 - c0, E, wc + warp * E, sorted_slot, slot_pos);
  }
  // (s_cnt is free: the placement reads its per-warp cursors)
  if (b == 0) write_tiles_block(E, S, T, has_shared, tile_rows, s_tot, s_off, tiles, meta, s_warp, s_cnt);
}

__global__ void __launch_bounds__(1024) build_tiles_kernel(const int32_t* __restrict__ offsets,
                                                           int T, int E, int k, int has_shared,
                                                           int tile_rows, int4* __restrict__ tiles,
                                                           int32_t* __restrict__ meta,
                                                           int32_t* __restrict__ status) {
  __shared__ int s_cnt[kMaxE];
  __shared__ int s_off[kMaxE];
  __shared__ int s_base[kMaxE];
  __shared__ int s_warp[32];
  __shared__ int s_bad;
  const int S = T * k;
  if (threadIdx.x == 0) s_bad = (offsets[0] != 0 || offsets[E] != S);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    s_off[e] = offsets[e];
    s_cnt[e] = offsets[e + 1] - offsets[e];
    if (s_cnt[e] < 0) s_bad = 1;
  }
  __syncthreads();
  if (s_bad) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
    if (threadIdx.x == 0) report_device_error(status, kDevBadIndex);
  }
  __syncthreads();
  write_tiles_block(E, S, T, has_shared, tile_rows, s_cnt, s_off, tiles, meta, s_warp, s_base);
}

}  // namespace

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, bool pdl,
                              cudaStream_t st) {
  const int blocks = (T + 7) / 8;
  auto kern = (E <= 256) ? route_topk_kernel<8> : (E <= 512) ? route_topk_kernel<16> : route_topk_kernel<32>;
  return launch_pdl(pdl, kern, dim3(blocks), dim3(256), 0, st, logits, T, E, k, ids, w);
}

cudaError_t launch_route_permute_small(const float* logits, const int32_t* ids_in, int T, int E,
                                       int k, int has_shared, int32_t* ids, float* w,
                                       int32_t* counts, int32_t* offsets, int32_t* sorted_slot,
                                       int32_t* slot_pos, int4* tiles, int32_t* meta,
                                       int tile_rows, cudaStream_t st) {
  auto kern = (E <= 256) ? route_permute_small_kernel<8>
             : (E <= 512) ? route_permute_small_kernel<16> : route_permute_small_kernel<32>;
  kern<<<1, 1024, 0, st>>>(logits, ids_in, T, E, k, has_shared, ids, w, counts, offsets,
                           sorted_slot, slot_pos, tiles, meta, tile_rows);
  return cudaGetLastError();
}

cudaError_t launch_route_permute_large(const float* logits, const int32_t* ids_in, int T, int E, int k,
                                      int has_shared, int32_t* ids, float* w, int32_t* counts,
                                      int32_t* offsets, int32_t* sorted_slot, int32_t* slot_pos,
                                      int32_t* hist, int4* tiles, int32_t* meta, int tile_rows,
                                      int32_t* status, cudaStream_t st) {
  int n_sm = 0;
  cudaError_t e = current_sm_count(&n_sm);
  if (e != cudaSuccess) return e;
  auto kern = (E <= 256) ? route_permute_large_kernel<8>
             : (E <= 512) ? route_permute_large_kernel<16> : route_permute_large_kernel<32>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(std::min(n_sm, kPermuteMaxGrid));   // fixed per device: the barrier count is monotonic
  cfg.blockDim = dim3(1024);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  unsigned long long* bar = reinterpret_cast<unsigned long long*>(meta + 4);
  return cudaLaunchKernelEx(&cfg, kern, logits, ids_in, T, E, k, has_shared, ids, w, counts, offsets,
                            sorted_slot, slot_pos, hist, tiles, meta, tile_rows, bar, status);
}

cudaError_t launch_permute_gather_small(const int32_t* ids, const uint16_t* x, int T, int E, int k, int has_shared,
                                        int H, int32_t* counts, int32_t* offsets, int32_t* sorted_slot,
                                        int32_t* slot_pos, int4* tiles, int32_t* meta, int tile_rows, uint16_t* xf,
                                        float* xe, int32_t* status, cudaStream_t st) {
  if (T < 1 || T > kDecodeMaxT || H % 8) return cudaErrorInvalidValue;
  int n_sm = 0;
  cudaError_t e = current_sm_count(&n_sm);
  if (e != cudaSuccess) return e;
  return launch_pdl(true, permute_gather_small_kernel, dim3(std::min(T, n_sm)), dim3(1024), 0, st, ids, x, T, E, k,
                    has_shared, H, counts, offsets, sorted_slot, slot_pos, tiles, meta, tile_rows, xf, xe, status);
}

cudaError_t launch_build_tiles(const int32_t* offsets, int T, int E, int k, int has_shared,
                               int tile_rows, int4* tiles, int32_t* meta, int32_t* status,
                               cudaStream_t st) {
  build_tiles_kernel<<<1, 1024, 0, st>>>(offsets, T, E, k, has_shared, tile_rows, tiles, meta,
                                         status);
  return cudaGetLastError();
}

}  // namespace moe
