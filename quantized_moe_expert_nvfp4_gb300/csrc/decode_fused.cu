// Decode/verify arm (T <= 8 rows): the whole layer in one persistent cooperative kernel.
//
// The "handover briefs" page asks of the decode arm: a vectorised NVFP4 GEMV that streams only
// the selected experts' bytes (bandwidth floor = bytes of the active experts / stream bandwidth,
// done when within 1.3x of it), the routed top-k and the shared expert in one launch per
// projection, gate+up fused and silu+down fused, and no host round trip.  Here one launch does
// all of it:
//   phase A  every CTA routes the T tokens itself (one warp per token), builds the permutation
//            in shared memory with block-wide scans, and stages x as f16 rows scaled by a power
//            of two per row (exact for every element of at least 2^-31 of the row maximum);
//   phase B  work units of two kinds, all gate_up units of the launch before all down units:
//            a gate_up unit is one active expert (the shared expert first) and one 64-wide slice
//            of its intermediate dimension -- it streams the slice's 64 gate rows and their 64 up
//            rows, computes h = SiLU(g) * u for its 64 columns (rounded to bf16), writes them to
//            the expert's rows of h in global memory and counts itself done for the expert; a
//            down unit is one active expert and 256 output rows -- it streams those rows' whole
//            down weights (contiguous 128-byte lines), waits until every slice of its expert's h
//            is written, stages that h as f16 and writes the 256 outputs of every token row
//            of the expert (y, fp32);
//   phase C  once every unit of the launch is done (one counter), each CTA combines a block of
//            output columns in the fixed order out[t] = sum_j w[t,j] y[t,j] + y_shared[t], fp32.
// A down unit's weights do not depend on h, so its CTA streams them while the gate_up units it
// waits for finish elsewhere; a CTA reaches its first down unit only after its own gate_up
// units, so no wait can close a cycle (all CTAs are co-resident: cooperative launch).
// A producer warp streams each CTA's units into a ring of shared-memory slots with large copies
// (a GB300 SM keeps only a few bulk copies in flight, so its stream rate grows with the copy
// size): a gate_up chunk is one 32 KB TMA tensor copy (128 rows x 512 K, 128-byte swizzle) and
// one copy of its 4 KB of scales; a down chunk one 32 KB copy (256 rows x 256 K) and one of its
// 4 KB of scales.  All 16 compute warps consume every chunk (each takes its share of the rows or
// of K), so the ring is consumed in order and its depth does not depend on the warp count.
// Products run on the tensor cores (mma.sync m16n8k16, f16 operands, fp32 accumulation): the
// weights are dequantized exactly into f16 (e2m1 x e4m3 has at most 6 significant bits and lies
// in [2^-10, 2688]) and the MMA columns are the expert's tokens (up to 8).
// The launch's counter set is the parity of the launch count (one atomic per CTA at entry); each
// launch zeroes the other set for the next one.  Every wait is bounded: an mbarrier or counter
// wait that runs past 1 s records MOE_ERR_DEVICE_TIMEOUT in the status word and the kernel winds
// down.
#include <algorithm>

#include "internal.cuh"
#include "mma_frag.cuh"
#include "tensor_map.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kDkCompute = 16;                 // compute warps
constexpr int kDkWarps = kDkCompute + 1;       // + the producer
constexpr int kDkThreads = kDkWarps * 32;
constexpr int kDkCThreads = kDkCompute * 32;
constexpr int kDkProducer = kDkCompute;        // warp index of the producer
constexpr int kDkXWarp0 = 8;                   // warps 8 .. 8 + T - 1 stage the activations
constexpr int kIs = kFdSlice;                  // intermediate columns of one unit
constexpr int kGuK = 512;                      // K of one gate_up chunk (two 128-byte lines per row)
constexpr int kGuPacked = 2 * kIs * kGuK / 2;  // 32 KB: [line 2][gate|up][64 rows][128 B]
constexpr int kGuScales = 2 * kIs * kGuK / 16; // 4 KB:  [gate|up][64 rows][32 B]
constexpr int kDnRows = 256;                   // output rows of a down unit
constexpr int kDnK = 256;                      // K of one down chunk (one 128-byte line per row)
constexpr int kDnScaleOff = 32 * 1024;         // down chunk: packed [256 rows][128 B], then [256 rows][16 B] scales
constexpr int kSlotBytes = 36 * 1024;
constexpr int kDkMaxSlots = 8;
constexpr int kFdMaxS = kFdMaxT * kMaxK;
constexpr int kFdSmemLimit = 227 * 1024;
constexpr int kFdMaxI = 1024;                 // intermediate size of the one-launch arm, at most
constexpr uint64_t kFdTimeoutNs = 1000000000ull;
constexpr int kRedCols = 16;                   // output columns per reduction block

static_assert(kIs == 64, "a gate_up unit's h slice is 8 MMA tiles of 8 gate + 8 up rows");
static_assert(kDnRows == 16 * kDkCompute, "a down chunk gives each compute warp one MMA tile of rows");
static_assert(2 * kFdMaxAct + 2 <= kFdSyncWords, "sync words: units-done counters and per-expert h counters");

// TMA descriptors:
//   gu   packed gate_up {128 B, row of [G * 2I - I], gate/up half (stride I rows), 128-byte line
//        (stride 128 B)}: a box of 64 rows x 2 halves x 2 lines is one gate_up chunk
//   gus  gate_up scales {H/16 B, row of [G * 2I - I], gate/up half}: a box of 32 B x 64 x 2
//   dn   packed down {I/2 B, row of [G * H]}: a box of 128 B x 256 rows is one down chunk
//   dns  down scales {I/16 B, row of [G * H]}: a box of 16 B x 256 rows
// (the row dimension of the gate_up maps stops I rows early, so that the up half of every box
// stays inside the tensor and the out-of-range fill would cover a bad coordinate)
struct FdMaps {
  CUtensorMap gu;
  CUtensorMap gus;
  CUtensorMap dn;
  CUtensorMap dns;
};

struct FdArgs {
  const uint16_t* x;
  const float* logits;
  const float* gu_scale2;
  const float* dn_scale2;
  int T, H, I, E, k, has_shared;
  int32_t* ids;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted_slot;
  int32_t* slot_pos;
  uint16_t* h;                    // [S + T][I] bf16, expert-ordered rows (gate_up units -> down units)
  float* y;                       // [S + T][H] fp32 expert outputs (down units -> combine)
  void* out;
  int out_is_fp32;
  unsigned long long* grid_ctr;   // launch count: one arrival per CTA and launch, monotonic
  unsigned* done;                 // [2] units-done counters (CTAs), one per launch parity
  unsigned* hdone;                // [2][kFdMaxAct] gate_up units done per active expert, per parity
  int32_t* status;
  int x_pitch, hb_pitch, ctl_off, ring_off, n_slots;
};

struct FdSmem {
  uint64_t full[kDkMaxSlots];
  uint64_t empty[kDkMaxSlots];
  int32_t ids[kFdMaxS];
  float w[kFdMaxS];
  int32_t sorted[kFdMaxS];
  int32_t slot_pos[kFdMaxS];
  int32_t act[kFdMaxS + 1];
  int32_t act_row[kFdMaxS + 1];
  int32_t act_cnt[kFdMaxS + 1];
  int32_t cnt[kMaxE];
  int wsum[kDkCompute];        // block scan of the expert counts: per-warp totals, then bases
  int wnz[kDkCompute];
  float xfac[kFdMaxT];         // 2^e of each staged f16 activation row
  alignas(16) float red[8][32 * 4];            // gate_up: the second K half's sums, per MMA tile
  float hfac[kFdMaxT];         // 2^e of each staged f16 row of h (down units)
  int n_act;
  int abort_flag;
  int ep;                      // this launch's counter set (parity of the launch count)
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
// Bounded wait on an mbarrier phase; false when the CTA is aborting or this wait ran out.
__device__ bool fd_wait(uint64_t* b, uint32_t parity, int* abort_flag, int32_t* status,
                        uint64_t limit_ns = kFdTimeoutNs) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (fd_try(b, parity)) return true;
    if ((i & 255u) == 255u) {
      if (*reinterpret_cast<volatile int*>(abort_flag)) return false;
      const uint64_t t = now_ns();
      if (t0 == 0) {
        t0 = t;
      } else if (t - t0 > limit_ns) {
        report_device_error(status, kDevTimeout);
        *reinterpret_cast<volatile int*>(abort_flag) = 1;
        return false;
      }
    }
  }
}

// One warp waits, with the kernel's bounded wait, on an mbarrier that nothing arrives at: the
// wait runs out after limit_ns and records the timeout in the status word (the test of the
// timeout path; nothing faults or hangs).
__global__ void __launch_bounds__(32) fd_timeout_probe_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&bar)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  fd_wait(&bar, 0, &abort_flag, status, limit_ns);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(tm), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* tm, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(tm), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* tm, int x, int y, int z, int w,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_addr(dst)),
      "l"(tm), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_addr(bar))
      : "memory");
}

// Two fp32 -> f16x2 (round to nearest; exact for the power-of-two-scaled bf16 values used here).
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
// Row exponent of the f16 staging: floor(log2(max)) - 14 puts the row maximum in [2^14, 2^15)
// (kept >= -126 so that 2^-e is a normal float; such a row is then scaled less than it could be).
__device__ __forceinline__ int row_exponent(float m) {
  return (m > 0.0f && m <= 3.4e38f) ? max(ilogbf(m) - 14, -126) : 0;
}
__device__ __forceinline__ float pow2i(int n) { return __int_as_float((127 + n) << 23); }   // n in [-126, 127]
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float absmax_bf16x8(float m, const uint4& v) {
  const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int c = 0; c < 4; ++c) m = fmaxf(m, fmaxf(fabsf(bf16_lo(q[c])), fabsf(bf16_hi(q[c]))));
  return m;
}
__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

template <int EPL>
__global__ void __launch_bounds__(kDkThreads, 1) decode_fused_kernel(const __grid_constant__ FdMaps maps, FdArgs a) {
  extern __shared__ __align__(1024) uint8_t fd_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(fd_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* xs = base;   // f16 activation rows, x_pitch bytes apart (gate_up units)
  uint8_t* hb = base;   // the same area for a down unit's f16 rows of h, hb_pitch bytes apart
  FdSmem* sm = reinterpret_cast<FdSmem*>(base + a.ctl_off);
  uint8_t* ring = base + a.ring_off;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = a.T, H = a.H, I = a.I, E = a.E, k = a.k, S = T * k;
  const int NS = a.n_slots;
  const int nslice = I / kIs;                // gate_up units per active expert
  const int nrb = H / kDnRows;               // down units per active expert
  const int n_gu = H / kGuK;                 // chunks of a gate_up unit
  const int n_dnc = I / kDnK;                // chunks of a down unit

  // Lane 0 of the producer warp issues chunk c of a gate_up unit (group g, slice m), or of a down
  // unit (group g, 256-row block rb), into ring position it.
  auto issue_gu = [&](int g, int m, int c, uint32_t it) {
    const int slot = it % NS;
    uint8_t* dst = ring + slot * kSlotBytes;
    uint64_t* bar = &sm->full[slot];
    const int r0 = g * 2 * I + m * kIs;   // first gate row of the slice; its up row is + I
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(kGuPacked + kGuScales)
                 : "memory");
    tma_load_4d(dst, &maps.gu, 0, r0, 0, 2 * c, bar);
    tma_load_3d(dst + kGuPacked, &maps.gus, 32 * c, r0, 0, bar);
  };
  auto issue_dn = [&](int g, int rb, int c, uint32_t it) {
    const int slot = it % NS;
    uint8_t* dst = ring + slot * kSlotBytes;
    uint64_t* bar = &sm->full[slot];
    const int r0 = g * H + rb * kDnRows;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(kDnRows * (kDnK / 2 + kDnK / 16))
                 : "memory");
    tma_load_2d(dst, &maps.dn, c * (kDnK / 2), r0, bar);
    tma_load_2d(dst + kDnScaleOff, &maps.dns, c * (kDnK / 16), r0, bar);
  };

  // ------------------------------------------------------------ phase A: route + permute
  uint32_t early = 0;   // chunks the producer issued before routing
  if (warp == kDkProducer) {
    if (lane == 0) {
      for (int s = 0; s < kDkMaxSlots; ++s) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sm->full[s])));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&sm->empty[s])), "r"(kDkCompute));
      }
      sm->abort_flag = 0;
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    // the shared expert is active group 0: this CTA's first unit is known before routing
    if (a.has_shared && static_cast<int>(blockIdx.x) < nslice) {
      early = static_cast<uint32_t>(min(n_gu, NS));
      if (lane == 0)
        for (uint32_t c = 0; c < early; ++c) issue_gu(E, blockIdx.x, c, c);
    }
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) sm->cnt[e] = 0;
  // this launch's counter set: the launch count's parity (the atomic's result is used after
  // routing, so its round trip overlaps the logits loads)
  unsigned long long launch_n = 0;
  if (threadIdx.x == 32) launch_n = atomicAdd(a.grid_ctr, 1ull);
  // activations: warp 8 + t stages token t as f16(x * 2^-e), e = floor(log2 max|x|) - 14 (at
  // least -126), the row maximum in [2^14, 2^15); the factor 2^e is applied to the dot products
  if (warp >= kDkXWarp0 && warp < kDkXWarp0 + T) {
    constexpr int kMaxV = 4096 / 256;   // uint4 per lane for H <= 4096
    const int t = warp - kDkXWarp0, nv = H / 256;
    const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<int64_t>(t) * H);
    uint4 v[kMaxV];
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < kMaxV; ++i) {
      if (i < nv) {
        v[i] = __ldg(src + i * 32 + lane);
        m = absmax_bf16x8(m, v[i]);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const int e = row_exponent(m);
    const float inv = pow2i(-e);
    if (lane == 0) sm->xfac[t] = pow2i(e);
    uint4* dst = reinterpret_cast<uint4*>(xs + t * a.x_pitch);
#pragma unroll
    for (int i = 0; i < kMaxV; ++i) {
      if (i < nv) {
        dst[i * 32 + lane] = make_uint4(f32x2_to_f16x2(bf16_lo(v[i].x) * inv, bf16_hi(v[i].x) * inv),
                                        f32x2_to_f16x2(bf16_lo(v[i].y) * inv, bf16_hi(v[i].y) * inv),
                                        f32x2_to_f16x2(bf16_lo(v[i].z) * inv, bf16_hi(v[i].z) * inv),
                                        f32x2_to_f16x2(bf16_lo(v[i].w) * inv, bf16_hi(v[i].w) * inv));
      }
    }
  }
  // routing: warp t < T ranks token t; lane j < k keeps the rank-j winner and its weight
  int my_id = 0;
  float my_w = 0.0f;
  if (warp < T) warp_topk<EPL>(a.logits + static_cast<int64_t>(warp) * E, E, k, lane, my_id, my_w);
  if (threadIdx.x == 32) sm->ep = static_cast<int>((launch_n / gridDim.x) & 1ull);
  __syncthreads();
  const int ep = sm->ep;
  if (blockIdx.x == 0) {   // the next launch's counters
    if (threadIdx.x == 0) a.done[ep ^ 1] = 0u;
    for (int i = threadIdx.x; i < kFdMaxAct; i += blockDim.x) a.hdone[(ep ^ 1) * kFdMaxAct + i] = 0u;
  }
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
  // exclusive scan of the counts over the compute warps: thread u takes experts 2u, 2u + 1
  // (E <= 1024); the active list is the shared expert first, then the routed experts ascending
  const int sh = a.has_shared;
  const int u2 = 2 * threadIdx.x;
  const int c0 = (warp < kDkCompute && u2 < E) ? sm->cnt[u2] : 0;
  const int c1 = (warp < kDkCompute && u2 + 1 < E) ? sm->cnt[u2 + 1] : 0;
  int vs = c0 + c1, vn = (c0 > 0) + (c1 > 0);   // inclusive warp scans of rows and of active experts
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int ys = __shfl_up_sync(0xffffffffu, vs, off), yn = __shfl_up_sync(0xffffffffu, vn, off);
    if (lane >= off) {
      vs += ys;
      vn += yn;
    }
  }
  if (lane == 31 && warp < kDkCompute) {
    sm->wsum[warp] = vs;
    sm->wnz[warp] = vn;
  }
  __syncthreads();
  if (warp == 0) {
    int ts = lane < kDkCompute ? sm->wsum[lane] : 0, tn = lane < kDkCompute ? sm->wnz[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int ys = __shfl_up_sync(0xffffffffu, ts, off), yn = __shfl_up_sync(0xffffffffu, tn, off);
      if (lane >= off) {
        ts += ys;
        tn += yn;
      }
    }
    __syncwarp();
    if (lane < kDkCompute) {   // exclusive bases of each warp
      sm->wsum[lane] = ts - sm->wsum[lane];
      sm->wnz[lane] = tn - sm->wnz[lane];
    }
    if (lane == kDkCompute - 1) {
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
  if (warp < kDkCompute) {
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
  // stable scatter by warp 0, 32 slots a step: slot s goes after the earlier slots of its expert
  // (its rank among the step's slots of the same expert, then the expert's cursor advances)
  if (warp == 0) {
    for (int s0 = 0; s0 < S; s0 += 32) {
      const int s = s0 + lane;
      const int e = (s < S) ? sm->ids[s] : -1;
      const unsigned same = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(same & ((1u << lane) - 1u));
      if (s < S) {
        const int p = sm->cnt[e] + rank;
        sm->sorted[p] = s;
        sm->slot_pos[s] = p;
        if (blockIdx.x == 0) {
          a.sorted_slot[p] = s;
          a.slot_pos[s] = p;
        }
      }
      __syncwarp();
      if (s < S && rank == 0) sm->cnt[e] += __popc(same);
      __syncwarp();
    }
  }
  __syncthreads();

  const int n_gu_units = sm->n_act * nslice;
  const int n_units = n_gu_units + sm->n_act * nrb;
  unsigned* const done = a.done + ep;
  unsigned* const hdone = a.hdone + ep * kFdMaxAct;

  if (warp == kDkProducer) {
    // ------------------------------------------------------------ producer
    uint32_t it = early;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
      const bool gu = u < n_gu_units;
      const int v = gu ? u : u - n_gu_units, per = gu ? nslice : nrb;
      const int g = sm->act[v / per], sub = v % per;
      const int nch = gu ? n_gu : n_dnc;
      for (int c = (u == static_cast<int>(blockIdx.x)) ? static_cast<int>(early) : 0; c < nch; ++c, ++it) {
        const int slot = it % NS;
        if (it >= static_cast<uint32_t>(NS)) {   // the slot's previous chunk must be consumed
          bool got = true;
          if (lane == 0) got = fd_wait(&sm->empty[slot], ((it / NS) - 1) & 1, &sm->abort_flag, a.status);
          ok = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
          if (!ok) break;
        }
        if (lane == 0) {
          if (gu)
            issue_gu(g, sub, c, it);
          else
            issue_dn(g, sub, c, it);
        }
      }
    }
    if (!ok && lane == 0) {   // let copies already issued land before the CTA winds down (bounded)
      for (uint32_t j = 0; j < static_cast<uint32_t>(NS) && j < it; ++j) {
        const uint32_t q = it - 1 - j;
        for (uint32_t i = 0; i < (1u << 20) && !fd_try(&sm->full[q % NS], (q / NS) & 1); ++i) {
        }
      }
    }
    return;
  }

  // ------------------------------------------------------------ compute warps
  bool ok = true;
  const int grp = lane >> 2, tig = lane & 3;
  // this lane's scale bytes of the piece pair 2 p, 2 p + 1 (piece q's lane block is 2 q + tig / 2):
  // bytes tig / 2 and 2 + tig / 2 of the pair's scale word, into the low and the high half
  const uint32_t psel = scale_pair_sel(tig);
  const int mt = warp & 7, kh = warp >> 3;                 // gate_up: MMA tile and 128-byte line
  uint32_t it = 0;
  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    if (u < n_gu_units) {
      // ======== gate_up unit: active group gi, intermediate columns 64 m .. 64 m + 63
      const int gi = u / nslice, m = u % nslice;
      const int g = sm->act[gi], row0 = sm->act_row[gi], nt = sm->act_cnt[gi];
      // B column grp is the expert's token grp (columns past its count repeat token 0, ignored)
      const int cb = (grp < nt) ? grp : 0;
      const int tb = (g == E) ? cb : sm->sorted[row0 + cb] / k;
      const uint8_t* xr = xs + tb * a.x_pitch + 16 * tig;
      // rows 8 mt + grp of the slice's gate half and of its up half; this warp takes line kh
      // (K 256 kh .. 256 kh + 255) of every chunk
      float d[4][4];
#pragma unroll
      for (int q = 0; q < 4; ++q) d[q][0] = d[q][1] = d[q][2] = d[q][3] = 0.0f;
      for (int c = 0; c < n_gu; ++c, ++it) {
        const int slot = it % NS;
        if (ok) ok = __all_sync(0xffffffffu, fd_wait(&sm->full[slot], (it / NS) & 1, &sm->abort_flag, a.status));
        if (ok) {
          const uint8_t* sl = ring + slot * kSlotBytes;
          const uint8_t* lg = sl + kh * (2 * kIs * 128) + (8 * mt + grp) * 128 + 4 * tig;   // gate row; up 64 rows on
          const uint4 sgv = *reinterpret_cast<const uint4*>(sl + kGuPacked + (8 * mt + grp) * 32 + 16 * kh);
          const uint4 suv = *reinterpret_cast<const uint4*>(sl + kGuPacked + (kIs + 8 * mt + grp) * 32 + 16 * kh);
          const uint8_t* xc = xr + 2 * (kGuK * c + 256 * kh);
#pragma unroll
          for (int q = 0; q < 8; ++q) {   // piece q of the line (stored at q ^ grp): blocks 2 q, 2 q + 1
            const uint32_t wg = *reinterpret_cast<const uint32_t*>(lg + ((q ^ grp) << 4));
            const uint32_t wu = *reinterpret_cast<const uint32_t*>(lg + kIs * 128 + ((q ^ grp) << 4));
            const uint4 xb = *reinterpret_cast<const uint4*>(xc + 64 * q);
            const __half2 sgp = e4m3_pair_f16x2_2m8((&sgv.x)[q >> 1], psel);
            const __half2 sup = e4m3_pair_f16x2_2m8((&suv.x)[q >> 1], psel);
            uint32_t gr[4], ur[4];
            piece_frag(wg, (q & 1) ? __high2half2(sgp) : __low2half2(sgp), gr);
            piece_frag(wu, (q & 1) ? __high2half2(sup) : __low2half2(sup), ur);
            mma16816(d[(q & 1) * 2], gr[0], ur[0], gr[1], ur[1], xb.x, xb.y);
            mma16816(d[(q & 1) * 2 + 1], gr[2], ur[2], gr[3], ur[3], xb.z, xb.w);
          }
        }
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&sm->empty[slot])) : "memory");
      }
      float p[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) p[r] = (d[0][r] + d[1][r]) + (d[2][r] + d[3][r]);
      // the two K halves meet (fixed order), then h[row0 + n][64 m + 8 mt + grp] =
      // bf16(SiLU(g) * u) for the lane's tokens n = 2 tig, 2 tig + 1, written to global memory
      if (kh == 1) *reinterpret_cast<float4*>(&sm->red[mt][4 * lane]) = make_float4(p[0], p[1], p[2], p[3]);
      named_sync(1, kDkCThreads);
      if (kh == 0) {
        const float4 o = *reinterpret_cast<const float4*>(&sm->red[mt][4 * lane]);
        p[0] += o.x;
        p[1] += o.y;
        p[2] += o.z;
        p[3] += o.w;
        const float s2 = __ldg(a.gu_scale2 + g);
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int n = 2 * tig + c2;
          if (n < nt) {
            const int t = (g == E) ? n : sm->sorted[row0 + n] / k;
            const float f = s2 * sm->xfac[t] * kScaleUnbias;
            a.h[static_cast<int64_t>(row0 + n) * I + m * kIs + 8 * mt + grp] =
                f32_to_bf16_bits(silu_f32(p[c2] * f) * (p[2 + c2] * f));
          }
        }
      }
      // every slice of h written by this unit is published before the unit counts as done
      named_sync(1, kDkCThreads);
      if (threadIdx.x == 0 && ok) {
        __threadfence();
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(hdone + gi) : "memory");
      }
    } else {
      // ======== down unit: active group gi, output rows 256 rb .. 256 rb + 255
      const int v = u - n_gu_units;
      const int gi = v / nrb, rb = v % nrb;
      const int g = sm->act[gi], row0 = sm->act_row[gi], nt = sm->act_cnt[gi];
      // wait until every gate_up unit of the group has written its slice of h
      if (threadIdx.x == 0 && ok) {
        const uint64_t t0 = now_ns();
        for (uint32_t i = 0;; ++i) {
          unsigned c;
          asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(c) : "l"(hdone + gi) : "memory");
          if (c >= static_cast<unsigned>(nslice)) break;
          if ((i & 63u) == 63u && (*reinterpret_cast<volatile int*>(&sm->abort_flag) || now_ns() - t0 > kFdTimeoutNs)) {
            if (!*reinterpret_cast<volatile int*>(&sm->abort_flag)) report_device_error(a.status, kDevTimeout);
            sm->abort_flag = 1;
            break;
          }
        }
      }
      named_sync(1, kDkCThreads);
      if (*reinterpret_cast<volatile int*>(&sm->abort_flag)) ok = false;
      // the group's rows of h as f16 scaled by 2^-e per row (e from the row's maximum over all I
      // columns, as for x): warp n stages token row n
      if (ok && warp < nt) {
        // the row stays in registers between its maximum and its conversion (I <= kFdMaxI: at
        // most kFdMaxI / 256 16-byte pieces per lane), one read of h from L2
        constexpr int kMaxHv = kFdMaxI / 256;
        const int nhv = I / 256;
        const uint4* src = reinterpret_cast<const uint4*>(a.h + static_cast<int64_t>(row0 + warp) * I);
        uint4 hv[kMaxHv];
        float mx = 0.0f;
#pragma unroll
        for (int i = 0; i < kMaxHv; ++i) {
          if (i < nhv) {
            hv[i] = __ldcg(src + i * 32 + lane);
            mx = absmax_bf16x8(mx, hv[i]);
          }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const int e = row_exponent(mx);
        const float inv = pow2i(-e);
        if (lane == 0) sm->hfac[warp] = pow2i(e);
        uint4* dst = reinterpret_cast<uint4*>(hb + warp * a.hb_pitch);
#pragma unroll
        for (int i = 0; i < kMaxHv; ++i) {
          if (i < nhv) {
            dst[i * 32 + lane] = make_uint4(f32x2_to_f16x2(bf16_lo(hv[i].x) * inv, bf16_hi(hv[i].x) * inv),
                                            f32x2_to_f16x2(bf16_lo(hv[i].y) * inv, bf16_hi(hv[i].y) * inv),
                                            f32x2_to_f16x2(bf16_lo(hv[i].z) * inv, bf16_hi(hv[i].z) * inv),
                                            f32x2_to_f16x2(bf16_lo(hv[i].w) * inv, bf16_hi(hv[i].w) * inv));
          }
        }
      }
      named_sync(1, kDkCThreads);
      // this warp's MMA tile: rows ra = 16 warp + grp and ra + 8 of the block, all of K; B column
      // grp is the group's token grp (columns past its count repeat token 0, never written)
      const int ra = 16 * warp + grp, rc = ra + 8;
      const uint8_t* hrow = hb + ((grp < nt) ? grp : 0) * a.hb_pitch + 16 * tig;
      float acc[2][4];
#pragma unroll
      for (int q = 0; q < 2; ++q) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.0f;
      for (int c = 0; c < n_dnc; ++c, ++it) {
        const int slot = it % NS;
        if (ok) ok = __all_sync(0xffffffffu, fd_wait(&sm->full[slot], (it / NS) & 1, &sm->abort_flag, a.status));
        if (ok) {
          const uint8_t* sl = ring + slot * kSlotBytes;
          const uint8_t* rowa = sl + ra * (kDnK / 2);
          const uint8_t* rowc = sl + rc * (kDnK / 2);
          const uint4 sca = *reinterpret_cast<const uint4*>(sl + kDnScaleOff + ra * (kDnK / 16));
          const uint4 scc = *reinterpret_cast<const uint4*>(sl + kDnScaleOff + rc * (kDnK / 16));
          const uint8_t* hc = hrow + 2 * kDnK * c;
#pragma unroll
          for (int q = 0; q < kDnK / 32; ++q) {   // piece q: K 32 q .. 32 q + 31 (128-byte swizzle)
            const uint32_t wa = *reinterpret_cast<const uint32_t*>(rowa + ((q ^ (ra & 7)) << 4) + 4 * tig);
            const uint32_t wc = *reinterpret_cast<const uint32_t*>(rowc + ((q ^ (rc & 7)) << 4) + 4 * tig);
            const uint4 xb = *reinterpret_cast<const uint4*>(hc + 64 * q);
            const __half2 sap = e4m3_pair_f16x2_2m8((&sca.x)[q >> 1], psel);
            const __half2 scp = e4m3_pair_f16x2_2m8((&scc.x)[q >> 1], psel);
            uint32_t ar[4], cr[4];
            piece_frag(wa, (q & 1) ? __high2half2(sap) : __low2half2(sap), ar);
            piece_frag(wc, (q & 1) ? __high2half2(scp) : __low2half2(scp), cr);
            mma16816(acc[q & 1], ar[0], cr[0], ar[1], cr[1], xb.x, xb.y);
            mma16816(acc[q & 1], ar[2], cr[2], ar[3], cr[3], xb.z, xb.w);
          }
        }
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&sm->empty[slot])) : "memory");
      }
      // y[row0 + n][256 rb + ra] (and ra + 8) for the lane's tokens n = 2 tig, 2 tig + 1
      if (ok) {
        const float s2d = __ldg(a.dn_scale2 + g) * kScaleUnbias;
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int n = 2 * tig + c2;
          if (n < nt) {
            const float f = s2d * sm->hfac[n];
            float* yr = a.y + static_cast<int64_t>(row0 + n) * H + rb * kDnRows + ra;
            yr[0] = (acc[0][c2] + acc[1][c2]) * f;
            yr[8] = (acc[0][2 + c2] + acc[1][2 + c2]) * f;
          }
        }
      }
    }
  }

  // ------------------------------------------------------------ phase C: combine
  // every CTA's outputs are published by its arrival on the launch's counter (release), and
  // the combine starts once all CTAs have arrived (acquire)
  named_sync(1, kDkCThreads);
  if (threadIdx.x == 0) {
    if (ok) {
      __threadfence();
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(done) : "memory");
      const uint64_t t0 = now_ns();
      for (uint32_t i = 0;; ++i) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(done) : "memory");
        if (v >= gridDim.x) break;
        if ((i & 63u) == 63u && now_ns() - t0 > kFdTimeoutNs) {
          report_device_error(a.status, kDevTimeout);
          sm->abort_flag = 1;
          break;
        }
      }
    } else {
      sm->abort_flag = 1;
    }
  }
  named_sync(1, kDkCThreads);
  if (*reinterpret_cast<volatile int*>(&sm->abort_flag)) return;
  // columns in blocks of 16: warp w takes the tasks (token t, 4 columns c4) w, w + 16, ...; lane
  // j < k loads rank j's 4 values of token t and lane k the shared expert's, all at once, and lane
  // 0 sums them in rank order, then adds the shared expert's (the values reach it by shuffles)
  const int cw = threadIdx.x >> 5;   // compute warp
  for (int b = blockIdx.x; b < H / kRedCols; b += gridDim.x) {
    const int col0 = b * kRedCols;
    for (int task = cw; task < T * 4; task += kDkCompute) {
      const int t = task >> 2, c4 = task & 3;
      float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      float wv = 0.0f;
      if (lane < k) {
        wv = sm->w[t * k + lane];
        v = __ldcg(reinterpret_cast<const float4*>(a.y + static_cast<int64_t>(sm->slot_pos[t * k + lane]) * H +
                                                   col0 + 4 * c4));
      } else if (lane == k && a.has_shared) {
        v = __ldcg(reinterpret_cast<const float4*>(a.y + static_cast<int64_t>(S + t) * H + col0 + 4 * c4));
      }
      float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 1
      for (int j = 0; j < k; ++j) {
        const float wj = __shfl_sync(0xffffffffu, wv, j);
        acc.x = fmaf(wj, __shfl_sync(0xffffffffu, v.x, j), acc.x);
        acc.y = fmaf(wj, __shfl_sync(0xffffffffu, v.y, j), acc.y);
        acc.z = fmaf(wj, __shfl_sync(0xffffffffu, v.z, j), acc.z);
        acc.w = fmaf(wj, __shfl_sync(0xffffffffu, v.w, j), acc.w);
      }
      if (a.has_shared) {
        acc.x += __shfl_sync(0xffffffffu, v.x, k);
        acc.y += __shfl_sync(0xffffffffu, v.y, k);
        acc.z += __shfl_sync(0xffffffffu, v.z, k);
        acc.w += __shfl_sync(0xffffffffu, v.w, k);
      }
      if (lane == 0) {
        const int64_t o = static_cast<int64_t>(t) * H + col0 + 4 * c4;
        if (a.out_is_fp32) {
          *reinterpret_cast<float4*>(static_cast<float*>(a.out) + o) = acc;
        } else {
          *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + o) =
              make_uint2(static_cast<uint32_t>(f32_to_bf16_bits(acc.x)) | (static_cast<uint32_t>(f32_to_bf16_bits(acc.y)) << 16),
                         static_cast<uint32_t>(f32_to_bf16_bits(acc.z)) | (static_cast<uint32_t>(f32_to_bf16_bits(acc.w)) << 16));
        }
      }
    }
  }
}

struct FdPlan {
  int x_pitch, hb_pitch, x_bytes, ctl_off, ring_off, n_slots;
  size_t smem_total;
};

bool fd_plan(const moe_shape_t& s, FdPlan* p) {
  if (s.T < 1 || s.T > kFdMaxT || s.H % 512 || s.H > 4096 || s.I % 256 || s.I > kFdMaxI) return false;
  // the 64 extra bytes per row put the 8 rows of an MMA's B loads in distinct banks
  p->x_pitch = 2 * s.H + 64;   // f16 rows of x (gate_up units)
  p->hb_pitch = 2 * s.I + 64;  // f16 rows of h (down units), in the same area
  p->x_bytes = ((s.T * std::max(p->x_pitch, p->hb_pitch) + 127) / 128) * 128;
  p->ctl_off = p->x_bytes;
  p->ring_off = ((p->ctl_off + static_cast<int>(sizeof(FdSmem)) + 1023) / 1024) * 1024;
  p->n_slots = std::min(kDkMaxSlots, (kFdSmemLimit - 1024 - p->ring_off) / kSlotBytes);
  p->smem_total = 1024 + static_cast<size_t>(p->ring_off) + static_cast<size_t>(p->n_slots) * kSlotBytes;
  return p->n_slots >= 3;
}

template <int EPL>
cudaError_t launch_fd(const FdMaps& maps, const FdArgs& args, const FdPlan& plan, cudaStream_t st) {
  const auto kern = decode_fused_kernel<EPL>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), static_cast<int>(plan.smem_total));
  if (e != cudaSuccess) return e;
  int n_sm = 0, per_sm = 0;
  if ((e = current_sm_count(&n_sm)) != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDkThreads, plan.smem_total);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_sm);
  cfg.blockDim = dim3(kDkThreads);
  cfg.dynamicSmemBytes = plan.smem_total;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, maps, args);
}

}  // namespace

cudaError_t launch_fd_timeout_probe(int32_t* status, uint64_t limit_ns, cudaStream_t st) {
  fd_timeout_probe_kernel<<<1, 32, 0, st>>>(status, limit_ns);
  return cudaGetLastError();
}

bool decode_fused_supported(const moe_shape_t& s) {
  FdPlan p;
  return fd_plan(s, &p);
}

// h [S + T][I] bf16, then (at a 256-byte boundary) y [S + T][H] fp32.
size_t fd_h_bytes(const moe_shape_t& s) {
  const size_t R = static_cast<size_t>(s.T) * s.k + s.T;
  return (R * s.I * sizeof(uint16_t) + 255) & ~static_cast<size_t>(255);
}

size_t fd_scratch_bytes(const moe_shape_t& s) {
  if (!decode_fused_supported(s)) return 0;
  const size_t R = static_cast<size_t>(s.T) * s.k + s.T;
  return fd_h_bytes(s) + R * s.H * sizeof(float);
}

cudaError_t launch_decode_fused(const DecodeFusedArgs& d, cudaStream_t st) {
  const moe_shape_t& s = d.shape;
  FdPlan plan;
  if (!fd_plan(s, &plan)) return cudaErrorInvalidValue;
  FdArgs a;
  a.x = d.x;
  a.logits = d.logits;
  a.gu_scale2 = d.gate_up.scale2;
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
  a.h = static_cast<uint16_t*>(d.scratch);
  a.y = reinterpret_cast<float*>(static_cast<char*>(d.scratch) + fd_h_bytes(s));
  a.out = d.out;
  a.out_is_fp32 = d.out_is_fp32;
  a.grid_ctr = d.grid_ctr;
  a.done = d.sync;
  a.hdone = d.sync + 2;
  a.status = d.status;
  a.x_pitch = plan.x_pitch;
  a.hb_pitch = plan.hb_pitch;
  a.ctl_off = plan.ctl_off;
  a.ring_off = plan.ring_off;
  a.n_slots = plan.n_slots;
  FdMaps maps;
  const uint64_t G = static_cast<uint64_t>(d.gate_up.G);
  const uint64_t H = static_cast<uint64_t>(s.H), I = static_cast<uint64_t>(s.I);
  // gate_up packed {128 B, rows, half, line}; rows stop I early so an up box stays inside
  const uint64_t gu_dims[4] = {128, G * 2 * I - I, 2, H / 256};
  const uint64_t gu_strides[3] = {H / 2, I * (H / 2), 128};
  const uint32_t gu_box[4] = {128, static_cast<uint32_t>(kIs), 2, 2};
  const uint64_t gus_dims[3] = {H / 16, G * 2 * I - I, 2};
  const uint64_t gus_strides[2] = {H / 16, I * (H / 16)};
  const uint32_t gus_box[3] = {32, static_cast<uint32_t>(kIs), 2};
  // down packed {I/2 B, row} with boxes of 128 B x 256 rows; scales {I/16 B, row}, 16 B x 256 rows
  const uint64_t dn_rows = static_cast<uint64_t>(d.down.G) * H;
  const uint64_t dn_dims[2] = {I / 2, dn_rows};
  const uint64_t dn_strides[1] = {I / 2};
  const uint32_t dn_box[2] = {kDnK / 2, kDnRows};
  const uint64_t dns_dims[2] = {I / 16, dn_rows};
  const uint64_t dns_strides[1] = {I / 16};
  const uint32_t dns_box[2] = {kDnK / 16, kDnRows};
  if (!make_tensor_map(&maps.gu, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, d.gate_up.packed, gu_dims, gu_strides, gu_box,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map(&maps.gus, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, d.gate_up.scales, gus_dims, gus_strides,
                       gus_box, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_tensor_map(&maps.dn, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, d.down.packed, dn_dims, dn_strides, dn_box,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map(&maps.dns, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, d.down.scales, dns_dims, dns_strides, dns_box,
                       CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  if (s.E <= 256) return launch_fd<8>(maps, a, plan, st);
  if (s.E <= 512) return launch_fd<16>(maps, a, plan, st);
  return launch_fd<32>(maps, a, plan, st);
}

}  // namespace moe
