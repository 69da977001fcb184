// Decode/verify arm (T <= 8 rows): the whole layer in one persistent cooperative kernel.
//
// The "handover briefs" page asks of the decode arm: a vectorised NVFP4 GEMV that streams only
// the selected experts' bytes (bandwidth floor = bytes of the active experts / stream bandwidth,
// done when within 1.3x of it), the routed top-k and the shared expert in one launch per
// projection, gate+up fused and silu+down fused, and no host round trip.  Here one launch does
// all of it:
//   phase A  every CTA routes the T tokens itself (one warp per token, the same selection as the
//            routing kernel; no launch boundary between routing and the weight stream), builds
//            the permutation in SMEM with block-wide scans, and stages x as f16 rows scaled by a
//            power of two per row (the tensor-core arm's convention: exact for every element of
//            at least 2^-31 of the row maximum);
//   phase B  gate_up units (8 gate rows + the 8 matching up rows of one active expert):
//            h = SiLU(g) * u in bf16; each unit counts itself on its expert's readiness counter;
//   phase C  down units (64 output rows of one active expert), each once its expert's h is
//            complete (no grid-wide barrier): y in fp32; the unit that completes a 64-column
//            block (the last of the active experts' units for it, found by an arrival counter)
//            runs the fixed-order fp32 combine of that block,
//            out[t] = sum_j w[t,j] y[slot(t,j)] + y[shared t].
// A producer warp streams each CTA's units (phase B then C) into a ring of SMEM slots: one TMA
// tensor copy of the unit's packed weights in the 128-byte swizzled layout, one copy of its
// scales (few, large copies keep the SM's copy engine streaming at full rate) and, for a down
// unit, its h rows, copied once the expert's readiness counter shows all its gate_up units done.
// The counters (and the combine's arrival counters) come in two sets used by alternate
// launches: a launch's set is the parity of the launch count, which every CTA takes with one
// atomic at entry, and each launch zeroes the other set for the next one.
// The products run on the tensor cores (mma.sync m16n8k16, f16 operands, fp32 accumulation):
// the weights are dequantized exactly into f16 (e2m1 x e4m3 has at most 6 significant bits and
// lies in [2^-10, 2688]), the MMA columns are the expert's tokens (up to 8), and the activations
// are f16 rows scaled by a power of two (x in phase A; each h row in its slot, from its maximum).
// Units are dealt round-robin to the CTAs, one CTA per SM; ring slot s belongs to the warp pair
// (s, s + NS).  Every wait is bounded: an mbarrier or counter wait that runs past 1 s records
// MOE_ERR_DEVICE_TIMEOUT in the status word and the kernel winds down.
#include <algorithm>

#include "internal.cuh"
#include "tensor_map.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kFdWarps = 16;                   // 4 per SM sub-partition: up to 128 registers a thread
constexpr int kFdThreads = kFdWarps * 32;
constexpr int kFdComputeWarps = kFdWarps - 1;
constexpr int kFdProducer = kFdComputeWarps;   // warp index of the producer
constexpr int kFdXWarp0 = 8;                   // warps 8 .. 8 + T - 1 stage the activations
constexpr int kFdGuPairs = 8;                  // gate_up unit: 8 gate rows + the 8 up rows (one m16 tile)
constexpr int kFdDnRows = 64;                  // down unit: 64 output rows (four m16 tiles)
constexpr int kFdMaxSlots = kFdComputeWarps / 2;   // ring slots; slot s is consumed by warps s and s + NS
static_assert(2 + 2 * kFdMaxSlots <= 16, "two named barriers per slot after barriers 0 and 1");
constexpr int kFdMaxS = kFdMaxT * kMaxK;
constexpr int kFdSmemLimit = 227 * 1024;
constexpr uint64_t kFdTimeoutNs = 1000000000ull;

// TMA descriptors of the packed weights, rows cut into 128-byte lines (swizzled 128B):
//   gu  {128 B, row of [G * 2I], gate/up half (stride I rows), line of the row (H / 256)}
//   dn  {128 B, row of [G * H], line of the row (I / 256)}
// and of the gate_up scales, {H/16 B, row of [G * 2I], gate/up half} (8 gate rows and their 8
// up rows in one copy).
struct FdMaps {
  CUtensorMap gu;
  CUtensorMap dn;
  CUtensorMap gus;
};

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
  unsigned long long* grid_ctr;   // launch count: one arrival per CTA and launch, monotonic
  unsigned* ccnt;                 // [2][kFdMaxBlocks] block arrivals, then [2][kFdMaxActive] readiness
  int32_t* status;
  int x_pitch, smem_off, sh_off, ring_off, ring_bytes;
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
  int wsum[kFdWarps];          // block scan of the expert counts: per-warp totals, then bases
  int wnz[kFdWarps];
  int wmax[kFdWarps];          // and per-warp maxima of the routed counts
  int ns;                      // this launch's ring: slots and slot size (from the routing)
  int slot_b;
  float xfac[kFdMaxT];         // 2^e of each staged f16 activation row
  alignas(16) float red[kFdMaxSlots][32 * 4];   // gate_up: the second warp's partial sums, per slot
  float hfac[kFdMaxSlots][kFdMaxT];              // down: 2^e of each staged h row, per slot
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
__device__ bool fd_wait(uint64_t* b, uint32_t parity, FdSmem* sm, int32_t* status,
                        uint64_t limit_ns = kFdTimeoutNs) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (fd_try(b, parity)) return true;
    if ((i & 255u) == 255u) {
      if (*reinterpret_cast<volatile int*>(&sm->abort_flag)) return false;
      const uint64_t t = now_ns();
      if (t0 == 0) {
        t0 = t;
      } else if (t - t0 > limit_ns) {
        report_device_error(status, kDevTimeout);
        *reinterpret_cast<volatile int*>(&sm->abort_flag) = 1;
        return false;
      }
    }
  }
}

// One warp waits, with the kernel's bounded wait, on an mbarrier that nothing arrives at: the
// wait runs out after limit_ns and records the timeout in the status word (the test of the
// timeout path; nothing faults or hangs).
__global__ void __launch_bounds__(32) fd_timeout_probe_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ FdSmem sm;
  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sm.full[0])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  fd_wait(&sm.full[0], 0, &sm, status, limit_ns);
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
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

// One m16n8k16 tensor-core step, D += A * B with f16 operands and fp32 accumulators.  Fragment
// layout (lane = 4 * grp + tig): A registers {row grp, K 2tig..+1}, {row grp + 8, same K},
// {row grp, K 2tig + 8..+9}, {row grp + 8, same K}; B registers {K 2tig..+1, column grp},
// {K 2tig + 8..+9, column grp}; D {row grp, columns 2tig, 2tig + 1}, {row grp + 8, same}.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  const __half2 p = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&p);
}
// Two e4m3 codes (the low 16 bits, the lower byte first) -> f16x2, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(r) : "r"(v));
  return r;
}
// Two fp32 -> f16x2 (round to nearest; exact for the power-of-two-scaled bf16 values used here).
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
// K order of the MMAs.  A 16-byte piece of a weight row holds 32 elements (two NVFP4 blocks);
// lane tig of a quad takes the piece's word tig, i.e. elements 8 tig .. 8 tig + 7, of which the
// first MMA of the piece uses 8 tig .. + 3 as its K positions (2 tig, 2 tig + 1 | 2 tig + 8,
// 2 tig + 9) and the second MMA 8 tig + 4 .. + 7.  The B operand (activation rows) is read in the
// same order, so each dot product is the pieces' own; the lane's elements all lie in block
// 2 q + tig / 2 of the piece and share one scale.  w: the lane's word of the row, s: the scale as
// an f16x2 splat; r[0], r[1] feed the first MMA, r[2], r[3] the second (e2m1 x e4m3 is exact in
// f16).
__device__ __forceinline__ void piece_frag(uint32_t w, uint32_t s, uint32_t (&r)[4]) {
  e2m1x8_to_f16x2(w, r);
#pragma unroll
  for (int i = 0; i < 4; ++i) r[i] = hmul2(r[i], s);
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


template <int EPL>
__global__ void __launch_bounds__(kFdThreads, 1) decode_fused_kernel(const __grid_constant__ FdMaps maps, FdArgs a) {
  extern __shared__ __align__(1024) uint8_t fd_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(fd_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* xs = base;   // f16 activation rows, x_pitch bytes apart
  FdSmem* sm = reinterpret_cast<FdSmem*>(base + a.smem_off);
  uint8_t* ring = base + a.ring_off;
  uint8_t* sh_h = base + a.sh_off;   // the shared expert's h rows [T][I] for its down unit in this CTA
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = a.T, H = a.H, I = a.I, E = a.E, k = a.k, S = T * k;
  // The ring's layout is set after routing: a slot holds a down unit's h rows for at most the
  // largest routed count (the shared expert's T rows have their own buffer), so routings that
  // spread the tokens get more slots.  Slot 0 starts at the ring in every layout, so the unit
  // issued before routing stays valid.
  int NS = kFdMaxSlots;
  uint32_t slot_bytes = 0;
  const int gu_per_group = I / kFdGuPairs;
  const int dn_per_group = H / kFdDnRows;
  // slot: the unit's packed weights (gate_up: 16 rows x H/2 bytes; down: 64 rows x I/2 bytes; in
  // swizzled 128-byte lines), then its scales (gate_up: [gate 8 | up 8][H/16]; down: [64][I/16]),
  // then a routed expert's down unit's h rows [nt][I]
  const uint32_t gu_wb = 2 * kFdGuPairs * (H / 2), gu_sb = kFdGuPairs * (H / 16);
  const uint32_t dn_wb = kFdDnRows * (I / 2), dn_sb = kFdDnRows * (I / 16);
  const uint32_t w_b = max(gu_wb, dn_wb), sc_b = max(2 * gu_sb, dn_sb), h_off = w_b + sc_b;

  // The producer issues one unit: u < nB is a gate_up unit of active group u / gu_per_group,
  // otherwise a down unit.  The shared expert is active group 0, so this CTA's first unit is
  // known before routing when blockIdx.x < gu_per_group.
  auto issue = [&](int u, int nB, uint32_t it) {
    const int slot = it % NS;
    uint8_t* dst = ring + slot * slot_bytes;
    uint64_t* bar = &sm->full[slot];
    if (u < nB) {
      const int g = (u < gu_per_group && a.has_shared) ? E : sm->act[u / gu_per_group];
      const int rg = g * 2 * I + (u % gu_per_group) * kFdGuPairs;   // first gate row; its up row is + I
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                   "r"(gu_wb + 2 * gu_sb)
                   : "memory");
      tma_load_4d(dst, &maps.gu, 0, rg, 0, 0, bar);
      tma_load_3d(dst + w_b, &maps.gus, 0, rg, 0, bar);
    } else {
      const int v = u - nB, gi = v / dn_per_group;
      const int r0 = sm->act[gi] * H + (v % dn_per_group) * kFdDnRows;
      const uint32_t h_bytes = static_cast<uint32_t>(sm->act_cnt[gi]) * I * 2;
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                   "r"(dn_wb + dn_sb + h_bytes)
                   : "memory");
      tma_load_3d(dst, &maps.dn, 0, r0, 0, bar);
      bulk_g2s(dst + w_b, a.dn_scales + static_cast<int64_t>(r0) * (I / 16), dn_sb, bar);
    }
  };
  // The h rows of down unit u (issued as ring position it) into the end of its slot (the shared
  // expert's into its own buffer: a CTA holds at most one of its H/64 <= 64 down units); only
  // once the expert's readiness counter shows every gate_up unit of it done (other CTAs write them).
  auto issue_h = [&](int u, int nB, uint32_t it) {
    const int gi = (u - nB) / dn_per_group;
    const int slot = it % NS;
    uint8_t* dst = (sm->act[gi] == E) ? sh_h : ring + slot * slot_bytes + h_off;
    bulk_g2s(dst, a.h + static_cast<int64_t>(sm->act_row[gi]) * I,
             static_cast<uint32_t>(sm->act_cnt[gi]) * I * 2, &sm->full[slot]);
  };

  // ------------------------------------------------------------ phase A: route + permute
  bool early = false;
  if (warp == kFdProducer && lane == 0) {
    for (int s = 0; s < kFdMaxSlots; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sm->full[s])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 2;" ::"r"(smem_addr(&sm->empty[s])));   // the slot's 2 warps
    }
    sm->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (a.has_shared && blockIdx.x < gu_per_group) {   // first unit: shared expert, gate_up
      issue(blockIdx.x, 1 << 30, 0);
      early = true;
    }
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) sm->cnt[e] = 0;
  // this launch's counter set: the launch count's parity (the atomic's result is used after
  // routing, so its round trip overlaps the logits loads)
  unsigned long long launch_n = 0;
  if (threadIdx.x == 32) launch_n = atomicAdd(a.grid_ctr, 1ull);
  // activations: warp 8 + t stages token t as f16(x * 2^-e), e = floor(log2 max|x|) - 14 (at
  // least -126), the row maximum in [2^14, 2^15); the factor 2^e is applied to the dot products
  if (warp >= kFdXWarp0 && warp < kFdXWarp0 + T) {
    constexpr int kMaxV = 4096 / 256;   // uint4 per lane for H <= 4096
    const int t = warp - kFdXWarp0, nv = H / 256;
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
  unsigned* const ccnt = a.ccnt + ep * kFdMaxBlocks;                       // this launch's arrivals
  unsigned* const ready = a.ccnt + 2 * kFdMaxBlocks + ep * kFdMaxActive;   // and readiness counters
  if (blockIdx.x == 0) {   // the next launch's set (no CTA of this launch touches it)
    for (int i = threadIdx.x; i < kFdMaxBlocks; i += blockDim.x) a.ccnt[(ep ^ 1) * kFdMaxBlocks + i] = 0u;
    for (int i = threadIdx.x; i < kFdMaxActive; i += blockDim.x)
      a.ccnt[2 * kFdMaxBlocks + (ep ^ 1) * kFdMaxActive + i] = 0u;
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
  // exclusive scan of the counts over the block: thread u takes experts 2u, 2u + 1 (E <= 1024);
  // the active list is the shared expert first, then the routed experts ascending
  const int sh = a.has_shared;
  const int u2 = 2 * threadIdx.x;
  const int c0 = (u2 < E) ? sm->cnt[u2] : 0;
  const int c1 = (u2 + 1 < E) ? sm->cnt[u2 + 1] : 0;
  int vs = c0 + c1, vn = (c0 > 0) + (c1 > 0);   // inclusive warp scans of rows and of active experts
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int ys = __shfl_up_sync(0xffffffffu, vs, off), yn = __shfl_up_sync(0xffffffffu, vn, off);
    if (lane >= off) {
      vs += ys;
      vn += yn;
    }
  }
  const int vmax = __reduce_max_sync(0xffffffffu, max(c0, c1));
  if (lane == 31) {
    sm->wsum[warp] = vs;
    sm->wnz[warp] = vn;
    sm->wmax[warp] = vmax;
  }
  __syncthreads();
  if (warp == 0) {
    int ts = lane < kFdWarps ? sm->wsum[lane] : 0, tn = lane < kFdWarps ? sm->wnz[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int ys = __shfl_up_sync(0xffffffffu, ts, off), yn = __shfl_up_sync(0xffffffffu, tn, off);
      if (lane >= off) {
        ts += ys;
        tn += yn;
      }
    }
    __syncwarp();
    if (lane < kFdWarps) {   // exclusive bases of each warp
      sm->wsum[lane] = ts - sm->wsum[lane];
      sm->wnz[lane] = tn - sm->wnz[lane];
    }
    if (lane == kFdWarps - 1) {
      if (sh) {
        sm->act[0] = E;
        sm->act_row[0] = S;
        sm->act_cnt[0] = T;
      }
      sm->n_act = tn + sh;
      if (blockIdx.x == 0) a.offsets[E] = S;
    }
    if (lane == 0) {   // the ring: h room for the largest routed count
      int mr = 0;
      for (int w2 = 0; w2 < kFdWarps; ++w2) mr = max(mr, sm->wmax[w2]);
      const uint32_t sb = ((w_b + sc_b + static_cast<uint32_t>(mr) * I * 2 + 1023u) / 1024u) * 1024u;
      sm->slot_b = static_cast<int>(sb);
      sm->ns = min(kFdMaxSlots, static_cast<int>(static_cast<uint32_t>(a.ring_bytes) / sb));
    }
  }
  __syncthreads();
  {
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
  NS = sm->ns;
  slot_bytes = static_cast<uint32_t>(sm->slot_b);
  const int nB = n_act * gu_per_group;
  const int nC = n_act * dn_per_group;

  if (warp == kFdProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = early ? 1 : 0;
      bool ok = true;
      // down units whose expert's h is not complete yet wait here for their h copy, in order (at
      // most the ring's slots)
      int pend_u[kFdMaxSlots];
      uint32_t pend_it[kFdMaxSlots];
      int ph = 0, pt = 0;   // head and tail counts
      auto expert_ready = [&](int u) {
        const int gi = (u - nB) / dn_per_group;
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ready + gi) : "memory");
        return v >= static_cast<unsigned>(gu_per_group);
      };
      // issue the waiting h copies whose expert is ready (all of them when force is set)
      auto drain = [&](bool force) {
        while (ph < pt && (force || expert_ready(pend_u[ph % kFdMaxSlots]))) {
          asm volatile("fence.proxy.async.global;" ::: "memory");   // h was written by generic stores
          issue_h(pend_u[ph % kFdMaxSlots], nB, pend_it[ph % kFdMaxSlots]);
          ++ph;
        }
      };
      for (int u = blockIdx.x + static_cast<int>(it) * gridDim.x; u < nB + nC; u += gridDim.x, ++it) {
        const int slot = it % NS;
        const uint32_t parity = ((it / NS) & 1) ^ 1;
        uint64_t t0 = 0;
        for (uint32_t i = 0;; ++i) {   // bounded wait for the slot; start h copies meanwhile
          if ((i & 7u) == 0u) drain(false);
          if (fd_try(&sm->empty[slot], parity)) break;
          if ((i & 255u) == 255u) {
            if (*reinterpret_cast<volatile int*>(&sm->abort_flag)) {
              ok = false;
              break;
            }
            const uint64_t t = now_ns();
            if (t0 == 0) {
              t0 = t;
            } else if (t - t0 > kFdTimeoutNs) {
              report_device_error(a.status, kDevTimeout);
              *reinterpret_cast<volatile int*>(&sm->abort_flag) = 1;
              ok = false;
              break;
            }
          }
        }
        if (!ok) break;
        issue(u, nB, it);
        if (u >= nB) {
          pend_u[pt % kFdMaxSlots] = u;
          pend_it[pt % kFdMaxSlots] = it;
          ++pt;
          drain(false);
        }
      }
      {   // the last down units wait for their experts (bounded)
        const uint64_t t0 = now_ns();
        for (uint32_t i = 0; ok && ph < pt; ++i) {
          drain(false);
          if ((i & 255u) == 255u) {
            if (*reinterpret_cast<volatile int*>(&sm->abort_flag)) ok = false;
            else if (now_ns() - t0 > kFdTimeoutNs) {
              report_device_error(a.status, kDevTimeout);
              *reinterpret_cast<volatile int*>(&sm->abort_flag) = 1;
              ok = false;
            }
          }
        }
        drain(true);   // on abort too: every issued slot then completes, and the drain below is short
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
  // the producer's order, unit i in slot i % NS.  Slot s belongs to warps s and s + NS (half 0
  // and 1), which take its units i = s, s + NS, ... in order, so a slot's successive phases are
  // awaited one after the other (a parity wait cannot tell phase n from phase n + 2).  A gate_up
  // unit is split by K between the two warps (half 1's partial sums meet half 0's in SMEM), a
  // down unit by rows.  Lane = 4 grp + tig.
  bool ok = true;
  const int grp = lane >> 2, tig = lane & 3;
  const uint32_t ssel = (tig >> 1) ? 0x3232u : 0x1010u;   // this lane's block of a piece: 2 q + tig / 2
  const int nB_cta = (blockIdx.x < nB) ? (nB - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const int n_cta = (blockIdx.x < nB + nC) ? (nB + nC - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const bool consumer = warp < 2 * NS;
  const int my_slot = warp % NS, half = warp / NS;

  // phase B: gate_up units.  MMA rows 0-7 are the gate rows j0 .. j0 + 7, rows 8-15 the matching
  // up rows; column n is the expert's n-th row of tokens (n < nt).
  for (int i = consumer ? my_slot : nB_cta; i < nB_cta; i += NS) {
    const int u = blockIdx.x + i * gridDim.x;
    const int slot = my_slot;
    if (ok) ok = __all_sync(0xffffffffu, fd_wait(&sm->full[slot], (i / NS) & 1, sm, a.status));
    const int gi = u / gu_per_group;
    const int g = sm->act[gi];
    const int j0 = (u % gu_per_group) * kFdGuPairs;
    const int row0 = sm->act_row[gi], nt = sm->act_cnt[gi];
    const float s2 = (half == 0) ? __ldg(a.gu_scale2 + g) : 0.0f;   // used by the epilogue
    float p[4] = {0.0f, 0.0f, 0.0f, 0.0f};   // rows grp / grp + 8, columns 2 tig, 2 tig + 1
    if (ok) {
      const uint8_t* sl = ring + slot * slot_bytes;
      const uint8_t* scg = sl + w_b + grp * (H / 16);      // scales of gate row grp
      const uint8_t* scu = scg + gu_sb;                    // and of its up row
      const int cb = (grp < nt) ? grp : 0;                 // B column grp (row 0 past nt: ignored)
      const int tb = (g == E) ? cb : sm->sorted[row0 + cb] / k;
      const uint8_t* xr = xs + tb * a.x_pitch + 16 * tig;  // x[32 p + 8 tig .. + 7] of piece p at + 64 p
      float d[4][4];   // four independent accumulation chains
#pragma unroll
      for (int q = 0; q < 4; ++q) d[q][0] = d[q][1] = d[q][2] = d[q][3] = 0.0f;
      const int nch = H / 256, c0 = half * (nch / 2);
      for (int c = c0; c < c0 + nch / 2; ++c) {   // line c of every row: pieces 8 c .. 8 c + 7
        const uint4 sgv = *reinterpret_cast<const uint4*>(scg + 16 * c);
        const uint4 suv = *reinterpret_cast<const uint4*>(scu + 16 * c);
        const uint8_t* lg = sl + (16 * c + grp) * 128 + 4 * tig;   // gate row grp; the up rows 8 lines on
        const uint8_t* xc = xr + 512 * c;
#pragma unroll
        for (int q = 0; q < 8; ++q) {   // piece q of the line (stored at q ^ grp): blocks 16 c + 2 q, + 1
          const uint32_t wg = *reinterpret_cast<const uint32_t*>(lg + ((q ^ grp) << 4));
          const uint32_t wu = *reinterpret_cast<const uint32_t*>(lg + 8 * 128 + ((q ^ grp) << 4));
          const uint4 xb = *reinterpret_cast<const uint4*>(xc + 64 * q);
          const uint32_t sg = __byte_perm(e4m3x2_to_f16x2((&sgv.x)[q >> 1] >> (16 * (q & 1))), 0u, ssel);
          const uint32_t su = __byte_perm(e4m3x2_to_f16x2((&suv.x)[q >> 1] >> (16 * (q & 1))), 0u, ssel);
          uint32_t gr[4], ur[4];
          piece_frag(wg, sg, gr);
          piece_frag(wu, su, ur);
          mma16816(d[(q & 1) * 2], gr[0], ur[0], gr[1], ur[1], xb.x, xb.y);
          mma16816(d[(q & 1) * 2 + 1], gr[2], ur[2], gr[3], ur[3], xb.z, xb.w);
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) p[r] = (d[0][r] + d[1][r]) + (d[2][r] + d[3][r]);
    }
    // the two halves meet: half 1 leaves its sums in SMEM, half 0 adds them (fixed order)
    if (half == 1) *reinterpret_cast<float4*>(&sm->red[slot][4 * lane]) = make_float4(p[0], p[1], p[2], p[3]);
    asm volatile("bar.sync %0, 64;" ::"r"(2 + slot) : "memory");
    if (half == 0 && ok) {
      const float4 o = *reinterpret_cast<const float4*>(&sm->red[slot][4 * lane]);
      p[0] += o.x;
      p[1] += o.y;
      p[2] += o.z;
      p[3] += o.w;
      // h[row0 + n, j0 + grp] = SiLU(g) * u for the lane's columns n = 2 tig, 2 tig + 1
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int col = 2 * tig + c2;
        if (col < nt) {
          const int t = (g == E) ? col : sm->sorted[row0 + col] / k;
          const float f = s2 * sm->xfac[t];
          a.h[static_cast<int64_t>(row0 + col) * I + j0 + grp] =
              f32_to_bf16_bits(silu_f32(p[c2] * f) * (p[2 + c2] * f));
        }
      }
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&sm->empty[slot])) : "memory");
    // the unit counts on its expert's readiness: half 0 signals its h stores with a non-blocking
    // arrive and goes on; half 1 (otherwise idle until its next unit's data) waits for that and
    // publishes them with its release, which the barrier makes cover half 0's stores
    if (half == 0) {
      asm volatile("bar.arrive %0, 64;" ::"r"(2 + kFdMaxSlots + slot) : "memory");
    } else {
      asm volatile("bar.sync %0, 64;" ::"r"(2 + kFdMaxSlots + slot) : "memory");
      if (lane == 0 && ok) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ready + gi) : "memory");
    }
  }

  // phase C: down units.  The unit's 64 rows are four MMA tiles (rows 16 r + grp, + 8); half h
  // takes tiles 2 h and 2 h + 1.  Column n is h row row0 + n, staged as f16 scaled by 2^-e_n with
  // e_n from that row's maximum.
  const int i0 = consumer ? nB_cta + ((my_slot - nB_cta) % NS + NS) % NS : n_cta;   // first i >= nB_cta in my slot
  for (int i = i0; i < n_cta; i += NS) {
    const int u = blockIdx.x + i * gridDim.x;
    const int slot = my_slot;
    const int blk = (u - nB) % dn_per_group;
    if (ok) ok = __all_sync(0xffffffffu, fd_wait(&sm->full[slot], (i / NS) & 1, sm, a.status));
    const int gi = (u - nB) / dn_per_group;
    const int g = sm->act[gi];
    const int row0 = sm->act_row[gi], nt = sm->act_cnt[gi];
    uint8_t* sl = ring + slot * slot_bytes;
    uint16_t* hs = reinterpret_cast<uint16_t*>(g == E ? sh_h : sl + h_off);   // h rows [nt][I]
    if (ok) {
      // each h row, in place, as f16(h * 2^-e) with e from the row's maximum (half h takes the
      // rows te with te % 2 == h); 2^e goes to hfac for the epilogue
      for (int te = half; te < nt; te += 2) {
        uint4* hr = reinterpret_cast<uint4*>(hs + te * I);
        constexpr int kMaxV = 1024 / 256;   // uint4 per lane for I <= 1024
        uint4 v[kMaxV];
        float m = 0.0f;
#pragma unroll
        for (int q = 0; q < kMaxV; ++q)
          if (q < I / 256) {
            v[q] = hr[q * 32 + lane];
            m = absmax_bf16x8(m, v[q]);
          }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        const int e = row_exponent(m);
        const float inv = pow2i(-e);
#pragma unroll
        for (int q = 0; q < kMaxV; ++q)
          if (q < I / 256)
            hr[q * 32 + lane] = make_uint4(f32x2_to_f16x2(bf16_lo(v[q].x) * inv, bf16_hi(v[q].x) * inv),
                                           f32x2_to_f16x2(bf16_lo(v[q].y) * inv, bf16_hi(v[q].y) * inv),
                                           f32x2_to_f16x2(bf16_lo(v[q].z) * inv, bf16_hi(v[q].z) * inv),
                                           f32x2_to_f16x2(bf16_lo(v[q].w) * inv, bf16_hi(v[q].w) * inv));
        if (lane == 0) sm->hfac[slot][te] = pow2i(e);
      }
    }
    // both halves' rows converted (executed by both warps whatever their status, so that neither
    // waits for a partner that skipped it)
    asm volatile("bar.sync %0, 64;" ::"r"(2 + slot) : "memory");
    if (ok) {
      const float s2 = __ldg(a.dn_scale2 + g);
      const uint8_t* sc = sl + w_b;   // scales [64][I/16]
      const float fac0 = (2 * tig < nt) ? sm->hfac[slot][2 * tig] : 0.0f;
      const float fac1 = (2 * tig + 1 < nt) ? sm->hfac[slot][2 * tig + 1] : 0.0f;
      const uint8_t* hb = reinterpret_cast<const uint8_t*>(hs + ((grp < nt) ? grp : 0) * I) + 16 * tig;
      float acc[2][2][4];   // [tile 2 half + r][piece parity]
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) acc[r][e2][0] = acc[r][e2][1] = acc[r][e2][2] = acc[r][e2][3] = 0.0f;
      for (int c = 0; c < I / 256; ++c) {
#pragma unroll 2
        for (int q = 0; q < 8; ++q) {   // piece q of line c: blocks 16 c + 2 q, + 1
          const uint4 xb = *reinterpret_cast<const uint4*>(hb + 512 * c + 64 * q);
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int ra = 16 * (2 * half + r) + grp;   // rows ra and ra + 8 (both stored with swizzle grp)
            const uint8_t* la = sl + (c * kFdDnRows + ra) * 128 + ((q ^ grp) << 4) + 4 * tig;
            const uint32_t wa = *reinterpret_cast<const uint32_t*>(la);
            const uint32_t wb = *reinterpret_cast<const uint32_t*>(la + 8 * 128);
            const uint32_t sa = __byte_perm(
                e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sc + ra * (I / 16) + 16 * c + 2 * q)), 0u, ssel);
            const uint32_t sb = __byte_perm(
                e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sc + (ra + 8) * (I / 16) + 16 * c + 2 * q)), 0u, ssel);
            uint32_t ar[4], br[4];
            piece_frag(wa, sa, ar);
            piece_frag(wb, sb, br);
            mma16816(acc[r][q & 1], ar[0], br[0], ar[1], br[1], xb.x, xb.y);
            mma16816(acc[r][q & 1], ar[2], br[2], ar[3], br[3], xb.z, xb.w);
          }
        }
      }
      // y[row0 + n, 64 blk + row] for the lane's columns n = 2 tig, 2 tig + 1
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int col = 2 * tig + c2;
        if (col < nt) {
          const float f = s2 * (c2 ? fac1 : fac0);
          float* yr = a.y + static_cast<int64_t>(row0 + col) * H + blk * kFdDnRows + 32 * half + grp;
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            yr[16 * r] = (acc[r][0][c2] + acc[r][1][c2]) * f;
            yr[16 * r + 8] = (acc[r][0][2 + c2] + acc[r][1][2 + c2]) * f;
          }
        }
      }
    }
    // the in-place h conversion (generic stores) is ordered before the next unit's copy into the
    // slot; the warp's y stores before lane 0's release below
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&sm->empty[slot])) : "memory");
    // the unit's arrival on its 64-column block (n_act in all), by half 1 once half 0's y stores
    // are ordered before it (half 0 goes on); the last arrival runs the combine
    unsigned last = 0;
    if (half == 0) {
      asm volatile("bar.arrive %0, 64;" ::"r"(2 + kFdMaxSlots + slot) : "memory");
    } else {
      asm volatile("bar.sync %0, 64;" ::"r"(2 + kFdMaxSlots + slot) : "memory");
      if (lane == 0 && ok) {
        unsigned old;
        asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(old) : "l"(ccnt + blk) : "memory");
        last = old == static_cast<unsigned>(n_act) - 1u;
      }
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
      // every active expert's y of columns [64 blk, 64 blk + 64) is final: the fixed-order combine
      // out[t, n] = sum_j w[t, j] * y[slot_pos[t*k + j], n] + y[S + t, n], lane l: n = 64 blk + 2 l, + 1
      __threadfence();
      const int n = blk * kFdDnRows + 2 * lane;
#pragma unroll 4
      for (int t = 0; t < T; ++t) {
        float ax = 0.0f, ay = 0.0f;
        for (int j = 0; j < k; ++j) {
          const float wj = sm->w[t * k + j];
          const float2 yv = __ldcg(reinterpret_cast<const float2*>(a.y + static_cast<int64_t>(sm->slot_pos[t * k + j]) * H + n));
          ax = fmaf(wj, yv.x, ax);
          ay = fmaf(wj, yv.y, ay);
        }
        if (a.has_shared) {
          const float2 yv = __ldcg(reinterpret_cast<const float2*>(a.y + static_cast<int64_t>(S + t) * H + n));
          ax += yv.x;
          ay += yv.y;
        }
        if (a.out_is_fp32) {
          *reinterpret_cast<float2*>(static_cast<float*>(a.out) + t * H + n) = make_float2(ax, ay);
        } else {
          *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.out) + t * H + n) =
              static_cast<uint32_t>(f32_to_bf16_bits(ax)) | (static_cast<uint32_t>(f32_to_bf16_bits(ay)) << 16);
        }
      }
    }
  }
}

struct FdPlan {
  int x_pitch, x_bytes, smem_off, sh_off, ring_off, ring_bytes, n_slots_worst;
  size_t smem_total;
};

bool fd_plan(const moe_shape_t& s, FdPlan* p) {
  if (s.T < 1 || s.T > kFdMaxT || s.H % 512 || s.H > 4096 || s.I % 256 || s.I > 1024) return false;
  p->x_pitch = 2 * s.H + 64;   // the 64 extra bytes put the 8 rows of an MMA's B loads in distinct banks
  p->x_bytes = ((s.T * p->x_pitch + 127) / 128) * 128;
  p->smem_off = p->x_bytes;
  p->sh_off = ((p->smem_off + static_cast<int>(sizeof(FdSmem)) + 127) / 128) * 128;
  const int sh_bytes = s.has_shared ? s.T * s.I * 2 : 0;   // the shared expert's h rows
  p->ring_off = ((p->sh_off + sh_bytes + 1023) / 1024) * 1024;
  p->ring_bytes = kFdSmemLimit - 1024 - p->ring_off;
  const int w_b = std::max(2 * kFdGuPairs * (s.H / 2), kFdDnRows * (s.I / 2));
  const int sc_b = std::max(2 * kFdGuPairs * (s.H / 16), kFdDnRows * (s.I / 16));
  // the kernel sizes its slots after routing; at worst a routed expert holds all T rows
  const int worst = ((w_b + sc_b + s.T * s.I * 2 + 1023) / 1024) * 1024;
  p->n_slots_worst = std::min(kFdMaxSlots, p->ring_bytes / worst);
  p->smem_total = 1024 + static_cast<size_t>(p->ring_off) + static_cast<size_t>(p->ring_bytes);
  return p->n_slots_worst >= 3;
}

template <int EPL>
cudaError_t launch_fd(const FdMaps& maps, const FdArgs& args, const FdPlan& plan, cudaStream_t st) {
  const auto kern = decode_fused_kernel<EPL>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), static_cast<int>(plan.smem_total));
  if (e != cudaSuccess) return e;
  int n_sm = 0, per_sm = 0;
  if ((e = current_sm_count(&n_sm)) != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFdThreads, plan.smem_total);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  if (n_sm < args.H / kFdDnRows) return cudaErrorInvalidValue;   // one shared-expert down unit per CTA at most
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
  a.x_pitch = plan.x_pitch;
  a.smem_off = plan.smem_off;
  a.ring_off = plan.ring_off;
  a.sh_off = plan.sh_off;
  a.ring_bytes = plan.ring_bytes;
  FdMaps maps;
  const uint64_t gu_dims[4] = {128, static_cast<uint64_t>(d.gate_up.G) * 2 * s.I, 2, static_cast<uint64_t>(s.H) / 256};
  const uint64_t gu_strides[3] = {static_cast<uint64_t>(s.H) / 2, static_cast<uint64_t>(s.I) * (s.H / 2), 128};
  const uint32_t gu_box[4] = {128, kFdGuPairs, 2, static_cast<uint32_t>(s.H) / 256};
  const uint64_t dn_dims[3] = {128, static_cast<uint64_t>(d.down.G) * s.H, static_cast<uint64_t>(s.I) / 256};
  const uint64_t dn_strides[2] = {static_cast<uint64_t>(s.I) / 2, 128};
  const uint32_t dn_box[3] = {128, kFdDnRows, static_cast<uint32_t>(s.I) / 256};
  const uint64_t gus_dims[3] = {static_cast<uint64_t>(s.H) / 16, static_cast<uint64_t>(d.gate_up.G) * 2 * s.I, 2};
  const uint64_t gus_strides[2] = {static_cast<uint64_t>(s.H) / 16, static_cast<uint64_t>(s.I) * (s.H / 16)};
  const uint32_t gus_box[3] = {static_cast<uint32_t>(s.H) / 16, kFdGuPairs, 2};
  if (!make_tensor_map(&maps.gu, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, d.gate_up.packed, gu_dims, gu_strides, gu_box,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map(&maps.gus, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, d.gate_up.scales, gus_dims, gus_strides,
                       gus_box, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_tensor_map(&maps.dn, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, d.down.packed, dn_dims, dn_strides, dn_box,
                       CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (s.E <= 256) return launch_fd<8>(maps, a, plan, st);
  if (s.E <= 512) return launch_fd<16>(maps, a, plan, st);
  return launch_fd<32>(maps, a, plan, st);
}

}  // namespace moe
