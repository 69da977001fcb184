// Decode/verify arm (T <= 8 rows): the whole layer in one persistent cooperative kernel.
//
// The "handover briefs" page asks of the decode arm: a vectorised NVFP4 GEMV that streams only
// the selected experts' bytes (bandwidth floor = bytes of the active experts / stream bandwidth,
// done when within 1.3x of it), the routed top-k and the shared expert in one launch per
// projection, gate+up fused and silu+down fused, and no host round trip.  Here one launch does
// all of it:
//   phase A  every CTA routes the T tokens itself (one warp per token, the same selection as the
//            routing kernel; no launch boundary between routing and the weight stream) and
//            builds the permutation in SMEM with block-wide scans;
//   phase B  gate_up units (8 gate + 8 up rows of one active expert): h = SiLU(g) * u in bf16;
//   grid barrier (h complete);
//   phase C  down units (64 output rows of one active expert): y in fp32; the unit that
//            completes a 64-column block (the last of the active experts' units for it, found by
//            an arrival counter) runs the fixed-order fp32 combine of that block,
//            out[t] = sum_j w[t,j] y[slot(t,j)] + y[shared t].
// A producer warp streams each CTA's units (phase B then C, without waiting for the barrier)
// into a ring of SMEM slots with TMA bulk copies; 8 compute warps dequantize (e2m1 x e4m3,
// exact) and accumulate in fp32.  Units are dealt round-robin to the CTAs, one CTA per SM.
// Every wait is bounded: an mbarrier or grid-barrier wait that runs past 1 s records
// MOE_ERR_DEVICE_TIMEOUT in the status word and the kernel winds down.
#include <algorithm>

#include "internal.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kFdGroups = 2;                   // compute warp groups, alternate units
constexpr int kFdGroupWarps = 8;
constexpr int kFdComputeWarps = kFdGroups * kFdGroupWarps;
constexpr int kFdThreads = (kFdComputeWarps + 1) * 32;
constexpr int kFdProducer = kFdComputeWarps;   // warp index of the producer
constexpr int kFdGuPairs = 8;                  // gate_up unit: 8 gate rows + the 8 up rows
constexpr int kFdDnRows = 64;                  // down unit rows (8 per warp of a group)
constexpr int kFdMaxSlots = 16;
constexpr int kFdMaxS = kFdMaxT * kMaxK;
constexpr int kFdSmemLimit = 227 * 1024;
constexpr uint64_t kFdTimeoutNs = 1000000000ull;

struct FdArgs {
  const uint16_t* x;
  const float* logits;
  const uint8_t* gu_packed;
  const uint8_t* gu_scales;
  const float* gu_scale2;
  const uint8_t* dn_packed;
  const uint8_t* dn_scales;
  const float* dn_scale2;
  int T, H, I, E, k, has_shared;
  int32_t* ids;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted_slot;
  int32_t* slot_pos;
  uint16_t* h;          // [S + T, I]
  float* y;             // [S + T, H]
  void* out;
  int out_is_fp32;
  unsigned long long* grid_ctr;   // grid-barrier arrivals, monotonic
  unsigned* ccnt;                 // arrivals per 64-column output block, zeroed each launch
  int32_t* status;
  int x_bytes, smem_off, ring_off, slot_bytes, n_slots;
};

struct FdSmem {
  uint64_t full[kFdMaxSlots];
  uint64_t empty[kFdMaxSlots];
  int32_t ids[kFdMaxS];
  float w[kFdMaxS];
  int32_t sorted[kFdMaxS];
  int32_t slot_pos[kFdMaxS];
  int32_t act[kFdMaxS + 1];
  int32_t act_row[kFdMaxS + 1];
  int32_t act_cnt[kFdMaxS + 1];
  int32_t cnt[kMaxE];
  int wsum[kFdComputeWarps];   // block scan of the expert counts: per-warp totals, then bases
  int wnz[kFdComputeWarps];
  int last[kFdGroups];         // this group's down unit completed its output block
  int n_act;
  int abort_flag;
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ bool fd_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ bool fd_wait(uint64_t* b, uint32_t parity, FdSmem* sm, int32_t* status) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (fd_try(b, parity)) return true;
    if ((i & 255u) == 255u) {
      if (*reinterpret_cast<volatile int*>(&sm->abort_flag)) return false;
      const uint64_t t = now_ns();
      if (t0 == 0) {
        t0 = t;
      } else if (t - t0 > kFdTimeoutNs) {
        report_device_error(status, kDevTimeout);
        *reinterpret_cast<volatile int*>(&sm->abort_flag) = 1;
        return false;
      }
    }
  }
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void compute_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kFdComputeWarps * 32) : "memory");
}
__device__ __forceinline__ void group_sync(int wg) {
  asm volatile("bar.sync %0, %1;" ::"r"(2 + wg), "n"(kFdGroupWarps * 32) : "memory");
}

// Grid-wide barrier of a cooperative launch (one thread per CTA): arrivals on a monotonic 64-bit
// counter; the barrier instance an arrival belongs to is old / gridDim, so each CTA waits for the
// counter to reach the end of its instance.  One atomic per CTA, no reset.
__device__ bool grid_barrier(unsigned long long* ctr, FdSmem* sm, int32_t* status) {
  __threadfence();
  const unsigned long long n = gridDim.x;
  const unsigned long long target = (atomicAdd(ctr, 1ull) / n + 1) * n;
  volatile unsigned long long* v = ctr;
  const uint64_t t0 = now_ns();
  for (uint32_t i = 0;; ++i) {
    if (*v >= target) break;
    if ((i & 1023u) == 1023u && now_ns() - t0 > kFdTimeoutNs) {
      report_device_error(status, kDevTimeout);
      sm->abort_flag = 1;
      return false;
    }
  }
  __threadfence();
  return true;
}

// sum over one 16-element NVFP4 block of e2m1(q_i) * x_i (two interleaved fp32 chains), times
// the block's e4m3 scale.
__device__ __forceinline__ float block_dot(uint2 q, uint32_t scale_byte, const float (&x)[16]) {
  float v[8], w[8];
  e2m1x8_to_f32(q.x, v);
  e2m1x8_to_f32(q.y, w);
  float d0 = v[0] * x[0], d1 = v[1] * x[1], d2 = w[0] * x[8], d3 = w[1] * x[9];
#pragma unroll
  for (int i = 2; i < 8; i += 2) {
    d0 = fmaf(v[i], x[i], d0);
    d1 = fmaf(v[i + 1], x[i + 1], d1);
    d2 = fmaf(w[i], x[8 + i], d2);
    d3 = fmaf(w[i + 1], x[9 + i], d3);
  }
  return ((d0 + d1) + (d2 + d3)) * e4m3_to_f32(scale_byte);
}

__device__ __forceinline__ void bf16x16_to_f32(const uint16_t* p, float (&x)[16], bool coherent) {
  uint4 a, b;
  if (coherent) {   // data written by other CTAs earlier in this kernel: bypass L1
    a = __ldcg(reinterpret_cast<const uint4*>(p));
    b = __ldcg(reinterpret_cast<const uint4*>(p) + 1);
  } else {
    a = *reinterpret_cast<const uint4*>(p);
    b = *(reinterpret_cast<const uint4*>(p) + 1);
  }
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Warp reduction of N values at once by recursive halving: after it, lane l holds the full
// sum of value ((l >> 2) & (N - 1)) for N = 8 (value (l >> 4) & 1 for N = 2).
template <int N>
__device__ __forceinline__ float warp_reduce_multi(float (&v)[N], int lane) {
  int n = N;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    if (n > 1) {
      const bool up = (lane & m) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        if (i < n / 2) {
          const float send = up ? v[i] : v[i + n / 2];
          const float keep = up ? v[i + n / 2] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
      }
      n >>= 1;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], m);
    }
  }
  return v[0];
}

template <int EPL>
__global__ void __launch_bounds__(kFdThreads, 1) decode_fused_kernel(FdArgs a) {
  extern __shared__ __align__(1024) uint8_t fd_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(fd_raw) + 1023) & ~uintptr_t(1023));
  uint16_t* xs = reinterpret_cast<uint16_t*>(base);
  FdSmem* sm = reinterpret_cast<FdSmem*>(base + a.smem_off);
  uint8_t* ring = base + a.ring_off;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = a.T, H = a.H, I = a.I, E = a.E, k = a.k, S = T * k;
  const int NS = a.n_slots;
  const int gu_per_group = I / kFdGuPairs;
  const int dn_per_group = H / kFdDnRows;
  const uint32_t gu_pb = kFdGuPairs * (H / 2), gu_sb = kFdGuPairs * (H / 16);
  const uint32_t dn_pb = kFdDnRows * (I / 2), dn_sb = kFdDnRows * (I / 16);

  // The producer issues one unit: u < nB is a gate_up unit of active group u / gu_per_group,
  // otherwise a down unit.  The shared expert is active group 0, so this CTA's first unit is
  // known before routing when blockIdx.x < gu_per_group.
  auto issue = [&](int u, int nB, uint32_t it) {
    const int slot = it % NS;
    uint8_t* dst = ring + slot * a.slot_bytes;
    uint64_t* bar = &sm->full[slot];
    if (u < nB) {
      const int g = (u < gu_per_group && a.has_shared) ? E : sm->act[u / gu_per_group];
      const int j0 = (u % gu_per_group) * kFdGuPairs;
      const int64_t rg = static_cast<int64_t>(g) * 2 * I + j0;
      const int64_t ru = rg + I;
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                   "r"(2 * gu_pb + 2 * gu_sb)
                   : "memory");
      bulk_g2s(dst, a.gu_packed + rg * (H / 2), gu_pb, bar);
      bulk_g2s(dst + gu_pb, a.gu_packed + ru * (H / 2), gu_pb, bar);
      bulk_g2s(dst + 2 * gu_pb, a.gu_scales + rg * (H / 16), gu_sb, bar);
      bulk_g2s(dst + 2 * gu_pb + gu_sb, a.gu_scales + ru * (H / 16), gu_sb, bar);
    } else {
      const int v = u - nB;
      const int g = sm->act[v / dn_per_group];
      const int64_t r0 = static_cast<int64_t>(g) * H + (v % dn_per_group) * kFdDnRows;
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                   "r"(dn_pb + dn_sb)
                   : "memory");
      bulk_g2s(dst, a.dn_packed + r0 * (I / 2), dn_pb, bar);
      bulk_g2s(dst + dn_pb, a.dn_scales + r0 * (I / 16), dn_sb, bar);
    }
  };

  // ------------------------------------------------------------ phase A: route + permute
  bool early = false;
  if (warp == kFdProducer && lane == 0) {
    for (int s = 0; s < NS; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sm->full[s])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&sm->empty[s])),
                   "r"(kFdGroupWarps));
    }
    sm->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (a.has_shared && blockIdx.x < gu_per_group) {   // first unit: shared expert, gate_up
      issue(blockIdx.x, 1 << 30, 0);
      early = true;
    }
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) sm->cnt[e] = 0;
  if (blockIdx.x == 0)   // the block counters of phase C, which only runs after the grid barrier
    for (int i = threadIdx.x; i < kFdMaxBlocks; i += blockDim.x) a.ccnt[i] = 0u;
  {
    const uint4* src = reinterpret_cast<const uint4*>(a.x);
    uint4* dst = reinterpret_cast<uint4*>(xs);
    for (int i = threadIdx.x; i < T * H / 8; i += blockDim.x) dst[i] = __ldg(src + i);
  }
  // routing: warp t < T ranks token t; lane j < k keeps the rank-j winner and its weight
  int my_id = 0;
  float my_w = 0.0f;
  if (warp < T) warp_topk<EPL>(a.logits + static_cast<int64_t>(warp) * E, E, k, lane, my_id, my_w);
  __syncthreads();
  if (warp < T && lane < k) {
    sm->ids[warp * k + lane] = my_id;
    sm->w[warp * k + lane] = my_w;
    atomicAdd(&sm->cnt[my_id], 1);
    if (blockIdx.x == 0) {
      a.ids[warp * k + lane] = my_id;
      a.topk_w[warp * k + lane] = my_w;
    }
  }
  __syncthreads();
  // exclusive scan of the counts over the block: compute thread u takes experts 2u, 2u + 1
  // (E <= 1024); the active list is the shared expert first, then the routed experts ascending
  const int sh = a.has_shared;
  const int u2 = 2 * threadIdx.x;
  int c0 = 0, c1 = 0;
  if (warp < kFdComputeWarps) {
    c0 = (u2 < E) ? sm->cnt[u2] : 0;
    c1 = (u2 + 1 < E) ? sm->cnt[u2 + 1] : 0;
  }
  int vs = c0 + c1, vn = (c0 > 0) + (c1 > 0);   // inclusive warp scans of rows and of active experts
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int ys = __shfl_up_sync(0xffffffffu, vs, off), yn = __shfl_up_sync(0xffffffffu, vn, off);
    if (lane >= off) {
      vs += ys;
      vn += yn;
    }
  }
  if (warp < kFdComputeWarps && lane == 31) {
    sm->wsum[warp] = vs;
    sm->wnz[warp] = vn;
  }
  __syncthreads();
  if (warp == 0) {
    int ts = lane < kFdComputeWarps ? sm->wsum[lane] : 0, tn = lane < kFdComputeWarps ? sm->wnz[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int ys = __shfl_up_sync(0xffffffffu, ts, off), yn = __shfl_up_sync(0xffffffffu, tn, off);
      if (lane >= off) {
        ts += ys;
        tn += yn;
      }
    }
    __syncwarp();
    if (lane < kFdComputeWarps) {   // exclusive bases of each warp
      sm->wsum[lane] = ts - sm->wsum[lane];
      sm->wnz[lane] = tn - sm->wnz[lane];
    }
    if (lane == kFdComputeWarps - 1) {
      if (sh) {
        sm->act[0] = E;
        sm->act_row[0] = S;
        sm->act_cnt[0] = T;
      }
      sm->n_act = tn + sh;
      if (blockIdx.x == 0) a.offsets[E] = S;
    }
  }
  __syncthreads();
  if (warp < kFdComputeWarps) {
    int run = sm->wsum[warp] + vs - (c0 + c1), pos = sm->wnz[warp] + vn - ((c0 > 0) + (c1 > 0)) + sh;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int e = u2 + q, c = q ? c1 : c0;
      if (e < E) {
        if (blockIdx.x == 0) {
          a.counts[e] = c;
          a.offsets[e] = run;
        }
        if (c > 0) {
          sm->act[pos] = e;
          sm->act_row[pos] = run;
          sm->act_cnt[pos] = c;
          ++pos;
        }
        sm->cnt[e] = run;   // the expert's first sorted position
        run += c;
      }
    }
  }
  __syncthreads();
  // stable scatter: slot s goes after the earlier slots of its expert
  for (int s = threadIdx.x; s < S; s += blockDim.x) {
    const int e = sm->ids[s];
    int rank = 0;
    for (int s2 = 0; s2 < s; ++s2) rank += sm->ids[s2] == e;
    const int p = sm->cnt[e] + rank;
    sm->sorted[p] = s;
    sm->slot_pos[s] = p;
    if (blockIdx.x == 0) {
      a.sorted_slot[p] = s;
      a.slot_pos[s] = p;
    }
  }
  __syncthreads();

  const int n_act = sm->n_act;
  const int nB = n_act * gu_per_group;
  const int nC = n_act * dn_per_group;

  if (warp == kFdProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = early ? 1 : 0;
      bool ok = true;
      for (int u = blockIdx.x + static_cast<int>(it) * gridDim.x; u < nB + nC; u += gridDim.x, ++it) {
        const int slot = it % NS;
        if (!(ok = fd_wait(&sm->empty[slot], ((it / NS) & 1) ^ 1, sm, a.status))) break;
        issue(u, nB, it);
      }
      if (!ok) {  // let copies already issued land before the CTA exits (bounded)
        for (uint32_t j = 0; j < static_cast<uint32_t>(NS) && j < it; ++j) {
          const uint32_t q = it - 1 - j;
          for (uint32_t i = 0; i < (1u << 20) && !fd_try(&sm->full[q % NS], (q / NS) & 1); ++i) {
          }
        }
      }
    }
    return;
  }

  // ------------------------------------------------------------ compute warps
  // This CTA's units are u = blockIdx.x + i * gridDim.x, i = 0, 1, ... over [0, nB + nC), in
  // the producer's order; warp group wg takes i = wg, wg + 2, ...  (slot i % NS).
  const int wg = warp / kFdGroupWarps, gw = warp % kFdGroupWarps;
  bool ok = true;
  const int hb = H / 16;   // 16-element blocks per gate_up row
  const int nB_cta = (blockIdx.x < nB) ? (nB - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const int n_cta = (blockIdx.x < nB + nC) ? (nB + nC - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  // phase B: gate_up units; warp gw owns gate row j0 + gw and up row j0 + gw of the unit
  for (int i = wg; i < nB_cta; i += kFdGroups) {
    const int u = blockIdx.x + i * gridDim.x;
    const int slot = i % NS;
    if (ok) ok = __all_sync(0xffffffffu, fd_wait(&sm->full[slot], (i / NS) & 1, sm, a.status));
    if (ok) {
      const int gi = u / gu_per_group;
      const int g = sm->act[gi];
      const int j = (u % gu_per_group) * kFdGuPairs + gw;
      const int row0 = sm->act_row[gi], nt = sm->act_cnt[gi];
      const uint8_t* sl = ring + slot * a.slot_bytes;
      const uint8_t* pg = sl + gw * (H / 2);
      const uint8_t* pu = sl + (kFdGuPairs + gw) * (H / 2);
      const uint8_t* sg = sl + 2 * kFdGuPairs * (H / 2) + gw * (H / 16);
      const uint8_t* su = sg + kFdGuPairs * (H / 16);
      const float s2 = __ldg(a.gu_scale2 + g);
      for (int te = 0; te < nt; ++te) {
        const int p = row0 + te;
        const int t = (g == E) ? te : sm->sorted[p] / k;
        const uint16_t* xt = xs + t * H;
        float acc[2] = {0.0f, 0.0f};
#pragma unroll 4
        for (int b = lane; b < hb; b += 32) {
          float xv[16];
          bf16x16_to_f32(xt + b * 16, xv, false);
          acc[0] += block_dot(*reinterpret_cast<const uint2*>(pg + b * 8), sg[b], xv);
          acc[1] += block_dot(*reinterpret_cast<const uint2*>(pu + b * 8), su[b], xv);
        }
        const float r = warp_reduce_multi<2>(acc, lane);   // lanes 0-15: gate, 16-31: up
        const float uval = __shfl_sync(0xffffffffu, r, 16);
        if (lane == 0) a.h[static_cast<int64_t>(p) * I + j] = f32_to_bf16_bits(silu_f32(r * s2) * (uval * s2));
      }
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&sm->empty[slot])) : "memory");
  }
  compute_sync();
  if (threadIdx.x == 0 && ok && !sm->abort_flag) grid_barrier(a.grid_ctr, sm, a.status);
  compute_sync();
  ok = ok && !*reinterpret_cast<volatile int*>(&sm->abort_flag);

  // phase C: down units; warp gw owns output rows n0 + 8 gw .. n0 + 8 gw + 7
  const int ib = I / 16;
  const int i0 = nB_cta + ((wg - nB_cta) % kFdGroups + kFdGroups) % kFdGroups;   // first i >= nB_cta with i % 2 == wg
  for (int i = i0; i < n_cta; i += kFdGroups) {
    const int u = blockIdx.x + i * gridDim.x;
    const int slot = i % NS;
    if (ok) ok = __all_sync(0xffffffffu, fd_wait(&sm->full[slot], (i / NS) & 1, sm, a.status));
    if (ok) {
      const int v = u - nB;
      const int gi = v / dn_per_group;
      const int g = sm->act[gi];
      const int n0 = (v % dn_per_group) * kFdDnRows + gw * 8;
      const int row0 = sm->act_row[gi], nt = sm->act_cnt[gi];
      const uint8_t* sl = ring + slot * a.slot_bytes;
      const uint8_t* pr = sl + gw * 8 * (I / 2);
      const uint8_t* sr = sl + kFdDnRows * (I / 2) + gw * 8 * (I / 16);
      const float s2 = __ldg(a.dn_scale2 + g);
      for (int te = 0; te < nt; ++te) {
        const int p = row0 + te;
        const uint16_t* hp = a.h + static_cast<int64_t>(p) * I;
        float acc[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
        for (int b = lane; b < ib; b += 32) {
          float hv[16];
          bf16x16_to_f32(hp + b * 16, hv, true);
#pragma unroll
          for (int r = 0; r < 8; ++r)
            acc[r] += block_dot(*reinterpret_cast<const uint2*>(pr + r * (I / 2) + b * 8), sr[r * (I / 16) + b], hv);
        }
        const float r = warp_reduce_multi<8>(acc, lane);   // lane l: row (l >> 2) & 7
        if ((lane & 3) == 0) a.y[static_cast<int64_t>(p) * H + n0 + (lane >> 2)] = r * s2;
      }
      __threadfence();   // this warp's y visible device-wide before the unit's arrival is counted
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&sm->empty[slot])) : "memory");
    // the unit's arrival on its 64-column block; the last arrival of a block runs its combine
    group_sync(wg);
    const int blk = (u - nB) % dn_per_group;
    if (gw == 0 && lane == 0)
      sm->last[wg] = ok && (atomicAdd(a.ccnt + blk, 1u) == static_cast<unsigned>(n_act) - 1u);
    group_sync(wg);
    if (sm->last[wg]) {
      // every active expert's y of columns [64 blk, 64 blk + 64) is final: the fixed-order combine
      // out[t, n] = sum_j w[t, j] * y[slot_pos[t*k + j], n] + y[S + t, n]
      __threadfence();
      for (int idx = gw * 32 + lane; idx < T * kFdDnRows; idx += kFdGroupWarps * 32) {
        const int t = idx / kFdDnRows, n = blk * kFdDnRows + idx % kFdDnRows;
        float acc = 0.0f;
        for (int j = 0; j < k; ++j)
          acc = fmaf(sm->w[t * k + j], __ldcg(a.y + static_cast<int64_t>(sm->slot_pos[t * k + j]) * H + n), acc);
        if (a.has_shared) acc += __ldcg(a.y + static_cast<int64_t>(S + t) * H + n);
        if (a.out_is_fp32)
          static_cast<float*>(a.out)[t * H + n] = acc;
        else
          static_cast<uint16_t*>(a.out)[t * H + n] = f32_to_bf16_bits(acc);
      }
    }
  }
}

struct FdPlan {
  int x_bytes, smem_off, ring_off, slot_bytes, n_slots;
  size_t smem_total;
};

bool fd_plan(const moe_shape_t& s, FdPlan* p) {
  if (s.T < 1 || s.T > kFdMaxT || s.H % 512 || s.H > 4096 || s.I > 1024 || s.I % kFdGuPairs) return false;
  p->x_bytes = ((s.T * s.H * 2 + 127) / 128) * 128;
  p->smem_off = p->x_bytes;
  p->ring_off = ((p->smem_off + static_cast<int>(sizeof(FdSmem)) + 1023) / 1024) * 1024;
  const int gu_unit = 2 * kFdGuPairs * (s.H / 2 + s.H / 16);
  const int dn_unit = kFdDnRows * (s.I / 2 + s.I / 16);
  p->slot_bytes = ((std::max(gu_unit, dn_unit) + 127) / 128) * 128;
  const int avail = kFdSmemLimit - 1024 - p->ring_off;
  p->n_slots = std::min(kFdMaxSlots, avail / p->slot_bytes);
  p->smem_total = 1024 + static_cast<size_t>(p->ring_off) + static_cast<size_t>(p->n_slots) * p->slot_bytes;
  return p->n_slots >= 3;
}

template <int EPL>
cudaError_t launch_fd(const FdArgs& args, const FdPlan& plan, cudaStream_t st) {
  static int configured_smem = 0;
  const auto kern = decode_fused_kernel<EPL>;
  if (configured_smem < static_cast<int>(plan.smem_total)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(plan.smem_total));
    if (e != cudaSuccess) return e;
    configured_smem = static_cast<int>(plan.smem_total);
  }
  int dev = 0, n_sm = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFdThreads, plan.smem_total);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_sm);
  cfg.blockDim = dim3(kFdThreads);
  cfg.dynamicSmemBytes = plan.smem_total;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args);
}

}  // namespace

bool decode_fused_supported(const moe_shape_t& s) {
  FdPlan p;
  return fd_plan(s, &p);
}

cudaError_t launch_decode_fused(const DecodeFusedArgs& d, cudaStream_t st) {
  const moe_shape_t& s = d.shape;
  FdPlan plan;
  if (!fd_plan(s, &plan)) return cudaErrorInvalidValue;
  FdArgs a;
  a.x = d.x;
  a.logits = d.logits;
  a.gu_packed = d.gate_up.packed;
  a.gu_scales = d.gate_up.scales;
  a.gu_scale2 = d.gate_up.scale2;
  a.dn_packed = d.down.packed;
  a.dn_scales = d.down.scales;
  a.dn_scale2 = d.down.scale2;
  a.T = s.T;
  a.H = s.H;
  a.I = s.I;
  a.E = s.E;
  a.k = s.k;
  a.has_shared = s.has_shared;
  a.ids = d.ids;
  a.topk_w = d.topk_w;
  a.counts = d.counts;
  a.offsets = d.offsets;
  a.sorted_slot = d.sorted_slot;
  a.slot_pos = d.slot_pos;
  a.h = d.h;
  a.y = d.y;
  a.out = d.out;
  a.out_is_fp32 = d.out_is_fp32;
  a.grid_ctr = reinterpret_cast<unsigned long long*>(d.grid_bar);
  a.ccnt = d.sync;
  a.status = d.status;
  a.x_bytes = plan.x_bytes;
  a.smem_off = plan.smem_off;
  a.ring_off = plan.ring_off;
  a.slot_bytes = plan.slot_bytes;
  a.n_slots = plan.n_slots;
  if (s.E <= 256) return launch_fd<8>(a, plan, st);
  if (s.E <= 512) return launch_fd<16>(a, plan, st);
  return launch_fd<32>(a, plan, st);
}

}  // namespace moe
