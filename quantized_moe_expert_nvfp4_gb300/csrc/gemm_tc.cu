// Grouped NVFP4 x bf16 GEMM on the fifth-generation tensor cores (tcgen05) -- the prefill arm.
//
// W4A16 as in the untransposed column of the "long-context cold prefill to SGLang parity"
// issue's kernel table (16-bit MMA, f32 accumulation, scale2 and SiLU(gate)*up in an fp32
// epilogue), computed over the resident [N, K/2] weight layout that the same issue prices as the
// option without a separate dequantization pass or transpose.
//
// Swap-AB: the MMA's M dimension is 128 weight rows of one expert, N is up to 128 of that
// expert's tokens, so a small expert group still fills M.  Per CTA (one per SM, persistent):
//   warp 0       TMA producer of the packed e2m1 tiles (K = 256 per stage)
//   warp 1       MMA issuer: the whole warp waits, one elected lane issues tcgen05.mma kind::f16
//                with A from TMEM and B from SMEM
//   warps 2-9    dequant: one weight row per thread (two warps per TMEM lane quarter, taking
//                alternate 64-wide K chunks), e2m1 x e4m3 -> f16 exactly (every product has at
//                most 6 significant bits and lies in [2^-10, 2688]), written to TMEM with
//                tcgen05.st as the A operand
//   warp 10      TMA producer of the activation tiles (K = 256 per stage)
//   warps 11-14  epilogue: tcgen05.ld of the fp32 accumulator, x scale2 x 2^e (the activation
//                row's exponent), SiLU(gate)*up (gate_up)
//   warp 15      TMA producer of the e4m3 scale tiles (a second issuing thread: each thread
//                keeps only a few bulk copies in flight, so the packed tiles get their own)
// The MMA is kind::f16 with f16 operands: the activations arrive as f16 rows in expert order,
// scaled by a power of two per row (exact for every element above 2^-31 of the row maximum), so
// the dequantization is one conversion and one packed multiply per pair of weights, and the
// products and the fp32 accumulation are those of the bf16 activations.
// The pipeline advances in groups of K = 256 (16 MMAs): one packed-weight stage, and one group
// stage made of a TMEM stage of dequantized A and an SMEM stage of activations, behind a single
// barrier.  Each readiness check of the MMA warp idles the tensor pipe for about 200 cycles at
// N <= 128 (measured on GB300), so the MMA warp checks once per group.  The accumulator is
// double-buffered in TMEM so the epilogue of one tile overlaps the next tile's main loop.  Every
// mbarrier wait is bounded; on timeout the kernel records MOE_ERR_DEVICE_TIMEOUT in the
// workspace status word and winds down.
#include "internal.cuh"
#include "mma_frag.cuh"
#include "tc_common.cuh"
#include "tensor_map.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kBM = 128;                      // weight rows per tile (MMA M)
constexpr int kBK = 64;                       // K per 128-byte swizzled operand row
constexpr int kGK = 256;                      // K per pipeline group
constexpr int kAStages = 4;                   // packed-weight ring (SMEM), one group per stage
constexpr int kAPackedBytes = kBM * kGK / 2;  // 16 KB: 128 rows x 128 B, 128B swizzle
constexpr int kAScaleBytes = kBM * kGK / 16;  // 2 KB: 128 rows x 16 B
constexpr int kAStageBytes = kAPackedBytes + kAScaleBytes;
constexpr int kTmemCols = 512;
constexpr int kGStagesMax = 3, kBStagesMax = 4;
static_assert(kGK / kBK == 4, "a group is four 64-wide chunks");

// Per-tile-size layout.  kBN = the tile's token rows at most (MMA N, rounded up to 16): 128 for
// prefill; 64 for small batches, where the smaller accumulators leave TMEM room for a third
// dequantized A stage and the smaller activation stages for four of them in the same SMEM (the
// activation stage's load is otherwise exposed once per group at a few tokens per expert).
template <int kBNt>
struct TcCfg {
  static constexpr int kBN = kBNt;
  static constexpr int kGStages = kBNt == 64 ? 3 : 2;          // dequantized A stages (TMEM)
  static constexpr int kBStages = kBNt == 64 ? 4 : 2;          // activation stages (SMEM)
  static constexpr int kBSubBytes = kBN * kBK * 2;             // kBN rows x 128 B, 128B swizzle
  static constexpr int kBStageBytes = (kGK / kBK) * kBSubBytes;  // four 64-wide sub-tiles
  static constexpr int kDCol = 0;                              // accumulators: 2 x kBN columns
  static constexpr int kACol = 2 * kBN;                        // A stages: kGStages x kGK / 2 columns
  static_assert(kBN == 64 || kBN == 128, "tile rows");
  static_assert(kACol + kGStages * (kGK / 2) <= kTmemCols, "TMEM budget");
  static_assert(kGStages <= kGStagesMax && kBStages <= kBStagesMax, "barrier arrays");
};

constexpr int kWarpTma = 0, kWarpMma = 1, kWarpDeq = 2, kWarpTmaB = 10, kWarpEpi = 11, kWarpTmaS = 15;
constexpr int kDeqWarps = 8;
constexpr int kEpiWarps = 4;
constexpr int kThreads = 16 * 32;
constexpr uint32_t kSpinLimit = 1u << 24;      // drain loops only
constexpr uint64_t kWaitTimeoutNs = 1000000000ull;  // 1 s: no legitimate wait comes close

// Tensor maps of one launch.  Weights: gate_up reads a tile's 64 gate rows and the matching 64 up
// rows (I rows further down the group) as one 3D box {K bytes, 64 rows, 2 halves}; down reads
// 128 consecutive rows.  Activations: one 3D box {64 columns, rows, 2 sub-tiles} per 128-wide K
// stage lands as two [rows][128 B] swizzled sub-tiles; b[i] has a box of 16 (i + 1) rows, so a
// tile loads its own rows rounded up to 16.
struct TcMaps {
  CUtensorMap a;                // packed e2m1
  CUtensorMap s;                // e4m3 scales
  CUtensorMap b[kTcTileRows / 16];   // f16 activations (the 64-row tiles use the first four)
};

struct TcArgs {
  const float* scale2;
  int Nw, K;                    // weight rows per group, reduction length
  const int4* tiles;
  const int32_t* meta;
  void* out;                    // h [S + T, I] bf16 or y [S + T, H] fp32
  int out_ld;
  const float* act_factor;      // 2^e of each f16 activation row (expert order)
  int32_t* status;
  uint16_t* y16;                // down: compact y, f16(accumulator * y16_scale), when set,
  float y16_scale;              // and per row the factor that restores it
  float* y16_rowf;
  int narrow_rows;              // items of at most this many rows take the register arm (0: none)
};

struct Smem {
  uint64_t a_full[kAStages];     // packed tile + scales landed (TMA transaction)
  uint64_t a_free[kAStages];     // every dequant warp is done reading the stage
  uint64_t g_full[kGStagesMax];  // a group's A is in TMEM (one arrival per dequant warp)
  uint64_t g_free[kGStagesMax];  // the MMAs reading that TMEM stage completed
  uint64_t b_full[kBStagesMax];  // a group's activations landed (the producer's transaction)
  uint64_t b_free[kBStagesMax];  // the MMAs reading that activation stage completed
  uint64_t acc_full[2];
  uint64_t acc_empty[2];         // one arrival per epilogue warp
  uint64_t drain;
  uint32_t nb_done[kBStagesMax];   // register arm: dequant warps done with an activation stage
  uint32_t tmem_base;
  int abort_flag;
};

// Bounded waits on this kernel's barriers (the CTA's abort flag lives in Smem).
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, Smem* sm, int32_t* status) {
  return tc::mbar_wait_flag(b, parity, &sm->abort_flag, status, kWaitTimeoutNs);
}

__device__ __forceinline__ bool warp_wait(uint64_t* b, uint32_t parity, Smem* sm, int32_t* status) {
  const bool ok = mbar_wait(b, parity, sm, status);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor: D f32, A f16, B f16, both K-major, M = 128, N.
__device__ __forceinline__ uint32_t make_idesc(int n) { return tc::idesc_f32acc(kBM, n); }

#define TC_ST32(taddr, r)                                                                          \
  asm volatile(                                                                                    \
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15," \
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),           \
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),      \
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), \
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]),          \
      "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]),          \
      "r"(r[30]), "r"(r[31])                                                                       \
      : "memory")

// Eight e2m1 codes (one 32-bit word, element i in bits 4i..4i+3) times the block scale ->
// four f16x2 words.  e2m1 -> f16 is the hardware conversion and the product with the e4m3
// scale is exact in f16 (at most 6 significant bits, |v| in [2^-10, 2688]).
__device__ __forceinline__ void dequant8(uint32_t w, uint32_t scale_f16x2, uint32_t* o) {
  uint32_t h[4];
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
  const __half2 s = *reinterpret_cast<const __half2*>(&scale_f16x2);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 p = __hmul2(*reinterpret_cast<const __half2*>(&h[i]), s);
    o[i] = *reinterpret_cast<const uint32_t*>(&p);
  }
}

__device__ __forceinline__ uint32_t e4m3_to_f16x2_splat(uint32_t byte) {
  const __half_raw hr = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(byte), __NV_E4M3);
  const uint32_t h = hr.x;
  return h | (h << 16);
}

__device__ __forceinline__ void tc_mma_acc(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc) {
  asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 1;" ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc),
               "r"(idesc)
               : "memory");
}

// Tile descriptor of a work item (zeros past the end).  Every role loads the next item's
// descriptor one item ahead, so its latency hides behind the current item.
__device__ __forceinline__ int4 load_tile(const TcArgs& a, int item, int n_items, int MB) {
  return item < n_items ? __ldg(a.tiles + item / MB) : make_int4(0, 0, 0, 0);
}

// The register arm of one work item whose tile has at most 8 rows (a tiny expert group): the eight
// dequant warps multiply the packed stages straight from shared memory with mma.sync, 16 weight
// rows per warp (gate_up: 8 gate rows and the matching 8 up rows, so a lane holds both halves of
// its h columns; down: 16 consecutive output rows) against the tile's tokens as the 8 MMA columns,
// and write the item's outputs themselves; the TMEM stages, the MMA warp and the epilogue warps
// skip the item.  The packed and activation stages are consumed in the rings' order like the
// tensor-core items'; the last dequant warp done with an activation stage releases it.  The
// dequant warps wait on every group's activation stage, tensor-core groups included, so that their
// parity waits never run two phases ahead of the loads (the MMA warp, which waits only on its own
// groups' stages, first waits for their dequantized A, i.e. after the dequant warps' waits).  ia
// advances by the item's groups.  Returns false when a wait ran out or the CTA is aborting.
template <bool kGateUp, int kBNt>
__device__ __forceinline__ bool narrow_item(const TcArgs& a, Smem* sm, const uint8_t* sA, const uint8_t* sB, const int4 td,
                                         int mb, int KG, uint32_t& ia) {
  using C = TcCfg<kBNt>;
  constexpr int kBStages = C::kBStages, kBStageBytes = C::kBStageBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w = warp - kWarpDeq, grp = lane >> 2, tig = lane & 3;
  const int ra = kGateUp ? 8 * w + grp : 16 * w + grp;                  // stage rows of MMA rows grp
  const int rb = kGateUp ? kBM / 2 + 8 * w + grp : 16 * w + grp + 8;    // and grp + 8
  const uint32_t psel = scale_pair_sel(tig);
  const int nb = (td.z + 15) & ~15;             // rows of each 64-wide activation sub-tile
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
  for (int g = 0; g < KG; ++g, ++ia) {
    const int st = ia % kAStages, sb = ia % kBStages;
    if (!warp_wait(&sm->a_full[st], (ia / kAStages) & 1, sm, a.status)) return false;
    if (!warp_wait(&sm->b_full[sb], (ia / kBStages) & 1, sm, a.status)) return false;
    const uint8_t* stage = sA + st * kAStageBytes;
    const uint4 sca = *reinterpret_cast<const uint4*>(stage + kAPackedBytes + ra * (kGK / 16));
    const uint4 scb = *reinterpret_cast<const uint4*>(stage + kAPackedBytes + rb * (kGK / 16));
    const uint8_t* rowa = stage + ra * (kGK / 2);
    const uint8_t* rowb = stage + rb * (kGK / 2);
    const uint8_t* brow = sB + sb * kBStageBytes + grp * (kBK * 2);   // token column grp
#pragma unroll
    for (int p = 0; p < kGK / 32; ++p) {   // piece p: K 32 p .. 32 p + 31, 16 bytes of a packed row
      // 128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r & 7)
      const uint32_t wa = *reinterpret_cast<const uint32_t*>(rowa + ((p ^ (ra & 7)) << 4) + 4 * tig);
      const uint32_t wb = *reinterpret_cast<const uint32_t*>(rowb + ((p ^ (rb & 7)) << 4) + 4 * tig);
      // the lane's 8 activations at K 32 p + 8 tig: sub-tile p / 2, chunk 4 (p & 1) + tig
      const uint4 xb = *reinterpret_cast<const uint4*>(brow + (p >> 1) * nb * (kBK * 2) +
                                                       (((4 * (p & 1) + tig) ^ (grp & 7)) << 4));
      const __half2 spa = e4m3_pair_f16x2_2m8((&sca.x)[p >> 1], psel);
      const __half2 spb = e4m3_pair_f16x2_2m8((&scb.x)[p >> 1], psel);
      uint32_t ar[4], br[4];
      piece_frag(wa, (p & 1) ? __high2half2(spa) : __low2half2(spa), ar);
      piece_frag(wb, (p & 1) ? __high2half2(spb) : __low2half2(spb), br);
      mma16816(acc[(p & 1) * 2], ar[0], br[0], ar[1], br[1], xb.x, xb.y);
      mma16816(acc[(p & 1) * 2 + 1], ar[2], br[2], ar[3], br[3], xb.z, xb.w);
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&sm->a_free[st]);
      __threadfence_block();
      if (atomicAdd(&sm->nb_done[sb], 1u) == static_cast<uint32_t>(kDeqWarps - 1)) {
        sm->nb_done[sb] = 0;
        __threadfence_block();
        mbar_arrive(&sm->b_free[sb]);
      }
    }
  }
  float d[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) d[r] = (acc[0][r] + acc[1][r]) + (acc[2][r] + acc[3][r]);
  // D: d[c2] is MMA row grp and token 2 tig + c2, d[2 + c2] MMA row grp + 8 and the same token
  const float s2 = __ldg(a.scale2 + td.x);
#pragma unroll
  for (int c2 = 0; c2 < 2; ++c2) {
    const int n = 2 * tig + c2;
    if (n >= td.z) continue;
    const float cf = __ldg(a.act_factor + td.y + n);
    const int64_t orow = static_cast<int64_t>(td.y + n) * a.out_ld;
    if (kGateUp) {
      const float f = s2 * cf * kScaleUnbias;
      static_cast<uint16_t*>(a.out)[orow + mb * (kBM / 2) + 8 * w + grp] =
          f32_to_bf16_bits(silu_f32(d[c2] * f) * (d[2 + c2] * f));
    } else if (a.y16) {
      const float ys = a.y16_scale * kScaleUnbias;
      uint16_t* yr = a.y16 + orow + mb * kBM + 16 * w + grp;
      yr[0] = __half_as_ushort(__float2half_rn(d[c2] * ys));
      yr[8] = __half_as_ushort(__float2half_rn(d[2 + c2] * ys));
      if (mb == 0 && w == 0 && grp == 0) a.y16_rowf[td.y + n] = s2 * cf / a.y16_scale;
    } else {
      const float f = s2 * cf * kScaleUnbias;
      float* yr = static_cast<float*>(a.out) + orow + mb * kBM + 16 * w + grp;
      yr[0] = d[c2] * f;
      yr[8] = d[2 + c2] * f;
    }
  }
  return true;
}

// kNarrow: whether the launch has the register arm (a separate instantiation, so that the
// tensor-core-only kernel keeps its own register allocation).
template <bool kGateUp, int kBNt, bool kNarrow>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_tc_kernel(const __grid_constant__ TcMaps maps, TcArgs a) {
  using C = TcCfg<kBNt>;
  constexpr int kBN = C::kBN, kGStages = C::kGStages, kBStages = C::kBStages;
  constexpr int kBStageBytes = C::kBStageBytes, kDCol = C::kDCol, kACol = C::kACol;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sB = base;                                   // kBStages activation stages (1024-aligned)
  uint8_t* sA = base + kBStages * kBStageBytes;         // kAStages x 18 KB (1024-aligned)
  Smem* sm = reinterpret_cast<Smem*>(sA + kAStages * kAStageBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int MB = a.Nw / kBM;                           // m-blocks per group
  const int KG = a.K / kGK;                            // pipeline groups per item

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(&sm->a_full[s], 2);   // the packed tile's producer and the scales' producer
      mbar_init(&sm->a_free[s], kDeqWarps);
    }
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(&sm->g_full[s], kDeqWarps);
      mbar_init(&sm->g_free[s], 1);
    }
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(&sm->b_full[s], 1);
      mbar_init(&sm->b_free[s], 1);
    }
    for (int d = 0; d < 2; ++d) {
      mbar_init(&sm->acc_full[d], 1);
      mbar_init(&sm->acc_empty[d], kEpiWarps);
    }
    mbar_init(&sm->drain, 1);
    for (int s = 0; s < kBStagesMax; ++s) sm->nb_done[s] = 0;
    sm->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kWarpTma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sm->tmem_base)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  pdl_wait_then_release();   // the work list and the activations come from earlier launches
  const int n_items = __ldg(a.meta) * MB;

  if (warp == kWarpTma) {
    if (lane == 0) {
      // packed weights and scales, one group per stage; gate_up takes the gate rows and the
      // matching up rows (I rows further down the group) as two 64-row boxes
      const int box_rows = kGateUp ? kBM / 2 : kBM;
      uint32_t ia = 0;
      bool ok = true;
      int4 td_next = load_tile(a, blockIdx.x, n_items, MB);
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const int4 td = td_next;
        td_next = load_tile(a, item + gridDim.x, n_items, MB);
        const int mb = item % MB;
        const int r0 = td.x * a.Nw + mb * box_rows;
        for (int g = 0; g < KG; ++g, ++ia) {
          const int st = ia % kAStages;
          if (!(ok = mbar_wait(&sm->a_free[st], ((ia / kAStages) & 1) ^ 1, sm, a.status))) break;
          uint8_t* dA = sA + st * kAStageBytes;
          mbar_expect_tx(&sm->a_full[st], kAPackedBytes);
          if (kGateUp) {
            tma_load_3d(dA, &maps.a, g * (kGK / 2), r0, 0, &sm->a_full[st]);
          } else {
            tma_load_2d(dA, &maps.a, g * (kGK / 2), r0, &sm->a_full[st]);
          }
        }
      }
      if (!ok) {  // let copies already issued land before the CTA winds down (bounded)
        for (int j = 0; j < kAStages && ia > 0; ++j, --ia) {
          const uint32_t q = ia - 1;
          for (uint32_t i = 0; i < (1u << 16) && !mbar_try(&sm->a_full[q % kAStages], (q / kAStages) & 1); ++i) {
          }
        }
      }
    }
  } else if (warp == kWarpTmaS) {
    if (lane == 0) {
      // the stages' e4m3 scales: a second issuing thread, so that the packed tiles' copies and
      // these small ones are not queued behind each other (a thread keeps only a few bulk copies
      // in flight); it arrives on the stage's barrier with its own byte count
      const int box_rows = kGateUp ? kBM / 2 : kBM;
      uint32_t ia = 0;
      bool ok = true;
      int4 td_next = load_tile(a, blockIdx.x, n_items, MB);
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const int4 td = td_next;
        td_next = load_tile(a, item + gridDim.x, n_items, MB);
        const int mb = item % MB;
        const int r0 = td.x * a.Nw + mb * box_rows;
        for (int g = 0; g < KG; ++g, ++ia) {
          const int st = ia % kAStages;
          if (!(ok = mbar_wait(&sm->a_free[st], ((ia / kAStages) & 1) ^ 1, sm, a.status))) break;
          uint8_t* dS = sA + st * kAStageBytes + kAPackedBytes;
          mbar_expect_tx(&sm->a_full[st], kAScaleBytes);
          if (kGateUp) {
            tma_load_3d(dS, &maps.s, g * (kGK / 16), r0, 0, &sm->a_full[st]);
          } else {
            tma_load_2d(dS, &maps.s, g * (kGK / 16), r0, &sm->a_full[st]);
          }
        }
      }
      if (!ok) {  // let copies already issued land before the CTA winds down (bounded)
        for (int j = 0; j < kAStages && ia > 0; ++j, --ia) {
          const uint32_t q = ia - 1;
          for (uint32_t i = 0; i < (1u << 16) && !mbar_try(&sm->a_full[q % kAStages], (q / kAStages) & 1); ++i) {
          }
        }
      }
    }
  } else if (warp == kWarpTmaB) {
    if (lane == 0) {
      // activation rows [td.y, td.y + n16) of the expert-ordered f16 operand (n16 = the tile's
      // rows rounded up to 16), the four 64-wide sub-tiles of a group in one box; rows past the
      // tile's own belong to the next tiles (or lie beyond the tensor and read as zero) and only
      // feed accumulator columns the epilogue skips
      uint32_t ib = 0;
      bool ok = true;
      int4 td_next = load_tile(a, blockIdx.x, n_items, MB);
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const int4 td = td_next;
        td_next = load_tile(a, item + gridDim.x, n_items, MB);
        const int n16 = (td.z + 15) >> 4;                 // 16-row blocks of the tile
        const CUtensorMap* mb_map = &maps.b[n16 - 1];
        for (int g = 0; g < KG; ++g, ++ib) {
          const int sb = ib % kBStages;
          if (!(ok = mbar_wait(&sm->b_free[sb], ((ib / kBStages) & 1) ^ 1, sm, a.status))) break;
          mbar_expect_tx(&sm->b_full[sb], (kGK / kBK) * n16 * 16 * kBK * 2);
          tma_load_3d(sB + sb * kBStageBytes, mb_map, 0, td.y, g * (kGK / kBK), &sm->b_full[sb]);
        }
      }
      if (!ok) {  // let the copies in flight land: the last stages' transactions (bounded)
        for (int j = 0; j < kBStages && ib > 0; ++j, --ib) {
          const uint32_t q = ib - 1;
          for (uint32_t i = 0; i < (1u << 16) && !mbar_try(&sm->b_full[q % kBStages], (q / kBStages) & 1); ++i) {
          }
        }
      }
    }
  } else if (warp == kWarpMma) {
    // The whole warp waits (converged) once per group; one elected lane issues the group's 16
    // MMAs and the commit that releases its TMEM and activation stages.
    // ig counts the groups of tensor-core items (TMEM stages), ib every group (activation ring)
    uint32_t ig = 0, ib = 0, ic = 0;
    bool ok = true;
    int4 td_next = load_tile(a, blockIdx.x, n_items, MB);
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      const int4 td = td_next;
      td_next = load_tile(a, item + gridDim.x, n_items, MB);
      if (kNarrow && td.z <= a.narrow_rows) {   // the dequant warps' register arm takes this item
        ib += KG;
        continue;
      }
      const int n = (td.z + 15) & ~15;
      const uint32_t idesc = make_idesc(n);
      const int d = ic & 1;
      if (!(ok = warp_wait(&sm->acc_empty[d], ((ic >> 1) & 1) ^ 1, sm, a.status))) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem + kDCol + d * kBN;
      for (int g = 0; g < KG; ++g, ++ig, ++ib) {
        const int gs = ig % kGStages, bs = ib % kBStages;
        if (!(ok = warp_wait(&sm->g_full[gs], (ig / kGStages) & 1, sm, a.status))) break;
        if (!(ok = warp_wait(&sm->b_full[bs], (ib / kBStages) & 1, sm, a.status))) break;
        tc_fence_after();
        if (elect_one()) {
          const uint32_t a_tmem = tmem + kACol + gs * (kGK / 2);
#pragma unroll
          for (int c = 0; c < kGK / kBK; ++c) {       // 64-wide chunk c of the group
            // sub-tile c of the stage starts c * n rows (n * 128 B, a multiple of 2 KB) in
            const uint32_t b_addr = smem_u32(sB + bs * kBStageBytes + c * n * (kBK * 2));
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
              const uint32_t at = a_tmem + c * (kBK / 2) + kk * 8;
              const uint64_t bd = smem_desc_sw128(b_addr + kk * 32);
              if (c == 0 && kk == 0)
                tc_mma(d_tmem, at, bd, idesc, g != 0);
              else
                tc_mma_acc(d_tmem, at, bd, idesc);
            }
          }
          tc_commit(&sm->g_free[gs]);
          tc_commit(&sm->b_free[bs]);
        }
        __syncwarp();
      }
      if (ok) {
        if (elect_one()) tc_commit(&sm->acc_full[d]);
        __syncwarp();
      }
      ++ic;
    }
    // every MMA issued must have completed before TMEM is released (bounded)
    if (elect_one()) {
      tc_commit(&sm->drain);
      for (uint32_t i = 0; i < kSpinLimit && !mbar_try(&sm->drain, 0); ++i) {
      }
    }
    __syncwarp();
  } else if (warp >= kWarpDeq && warp < kWarpDeq + kDeqWarps) {
    const int q = warp & 3;                    // TMEM lane quarter of this warp
    const int hsel = (warp - kWarpDeq) >> 2;   // chunks hsel and hsel + 2 of each group
    int srow;                                  // SMEM row of the packed tile (== weight row offset)
    if (kGateUp) {
      const int half = lane >> 4, j = q * 16 + (lane & 15);
      srow = half * (kBM / 2) + j;             // lanes 0-15 gate rows, 16-31 the matching up rows
    } else {
      srow = q * 32 + lane;
    }
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t ia = 0, iw = 0;   // every group (packed-weight and activation rings); tensor-core groups
    bool ok = true;
    int4 td_next = load_tile(a, blockIdx.x, n_items, MB);
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      const int4 td = td_next;
      td_next = load_tile(a, item + gridDim.x, n_items, MB);
      if (kNarrow && td.z <= a.narrow_rows) {
        ok = narrow_item<kGateUp, kBNt>(a, sm, sA, sB, td, item % MB, KG, ia);
        continue;
      }
      for (int g = 0; g < KG; ++g, ++ia, ++iw) {
        const int st = ia % kAStages, ts = iw % kGStages;
        if (!(ok = warp_wait(&sm->a_full[st], (ia / kAStages) & 1, sm, a.status))) break;
        // with the register arm the dequant warps observe every activation stage's phase in order
        // (a parity wait only tells two consecutive phases apart, and the register arm's waits on
        // these barriers must not run two phases ahead of the loads)
        if (kNarrow && !(ok = warp_wait(&sm->b_full[ia % kBStages], (ia / kBStages) & 1, sm, a.status))) break;
        const uint8_t* stage = sA + st * kAStageBytes;
        const uint8_t* rowp = stage + srow * (kGK / 2);
        const uint4 sc = *reinterpret_cast<const uint4*>(stage + kAPackedBytes + srow * (kGK / 16));
        uint4 pk[2][2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int ss = hsel + 2 * h2;        // 64-wide chunk of this group
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            const int c = 2 * ss + c2;         // 16-byte chunk, 128B swizzle: chunk ^= row & 7
            pk[h2][c2] = *reinterpret_cast<const uint4*>(rowp + ((c ^ (srow & 7)) << 4));
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->a_free[st]);
        if (!(ok = warp_wait(&sm->g_free[ts], ((iw / kGStages) & 1) ^ 1, sm, a.status))) break;
        tc_fence_after();
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int ss = hsel + 2 * h2;
          const uint32_t scw = h2 ? (hsel ? sc.w : sc.z) : (hsel ? sc.y : sc.x);   // scales of chunk ss
          uint32_t o[32];
          const uint32_t pw[8] = {pk[h2][0].x, pk[h2][0].y, pk[h2][0].z, pk[h2][0].w,
                                  pk[h2][1].x, pk[h2][1].y, pk[h2][1].z, pk[h2][1].w};
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const uint32_t s2 = e4m3_to_f16x2_splat((scw >> (8 * b)) & 0xffu);
            dequant8(pw[2 * b], s2, o + 8 * b);
            dequant8(pw[2 * b + 1], s2, o + 8 * b + 4);
          }
          __syncwarp();
          TC_ST32(t_lane + kACol + ts * (kGK / 2) + ss * (kBK / 2), o);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->g_full[ts]);
      }
    }
  } else if (warp >= kWarpEpi && warp < kWarpEpi + kEpiWarps) {
    const int q = warp & 3;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t ic = 0;
    bool ok = true;
    // column scales of an item: scale2 of its group and 2^e of each activation row (lane l holds
    // columns l, l + 32, l + 64, l + 96); those of the next item are fetched while this one's
    // accumulator is awaited and stored
    float s2_next = 0.0f, cf_next[kBN / 32];
    auto fetch_scales = [&](const int4& t) {
      s2_next = __ldg(a.scale2 + t.x);
#pragma unroll
      for (int i = 0; i < kBN / 32; ++i)
        cf_next[i] = (32 * i + lane < t.z) ? __ldg(a.act_factor + t.y + 32 * i + lane) : 0.0f;
    };
    int4 td_next = load_tile(a, blockIdx.x, n_items, MB);
    if (blockIdx.x < n_items) fetch_scales(td_next);
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      const int4 td = td_next;
      td_next = load_tile(a, item + gridDim.x, n_items, MB);
      const float s2 = s2_next;
      float cf[kBN / 32];
#pragma unroll
      for (int i = 0; i < kBN / 32; ++i) cf[i] = cf_next[i];
      if (kNarrow && td.z <= a.narrow_rows) {   // written by the dequant warps' register arm
        if (item + static_cast<int>(gridDim.x) < n_items) fetch_scales(td_next);
        continue;
      }
      const int mb = item % MB;
      const int d = ic & 1;
      if (!kGateUp && a.y16 && mb == 0 && q == 0) {   // the tile's row factors for the combine
#pragma unroll
        for (int i = 0; i < kBN / 32; ++i)
          if (32 * i + lane < td.z) a.y16_rowf[td.y + 32 * i + lane] = s2 * cf[i] / a.y16_scale;
      }
      if (!(ok = warp_wait(&sm->acc_full[d], (ic >> 1) & 1, sm, a.status))) break;
      tc_fence_after();
      const int n = (td.z + 15) & ~15;
      for (int c0 = 0; c0 < n; c0 += 16) {
        uint32_t v[16];
        __syncwarp();
        TC_LD16(t_lane + kDCol + d * kBN + c0, v);
        // scale of column c0 + i: lane (c0 & 31) + i of register c0 / 32
        const int cr = c0 >> 5;
        float colf = cf[0];
#pragma unroll
        for (int i = 1; i < kBN / 32; ++i)
          if (cr == i) colf = cf[i];
        colf *= s2;
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (kGateUp) {
          // lanes 0-15 hold gate rows j, lanes 16-31 the up rows j (j = mb*64 + 16q + lane%16);
          // a gate lane finishes columns c0..c0+7 and its up partner (lane ^ 16) c0+8..c0+15,
          // each receiving the other half of its pair by one exchange
          const bool is_gate = lane < 16;
          const int j = mb * 64 + q * 16 + (lane & 15);
          const int cb = is_gate ? 0 : 8;
          float gv[8], uv[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t other = __shfl_xor_sync(0xffffffffu, is_gate ? v[8 + i] : v[i], 16);
            const float sc = __shfl_sync(0xffffffffu, colf, (c0 & 31) + cb + i);
            gv[i] = __uint_as_float(is_gate ? v[i] : other) * sc;
            uv[i] = __uint_as_float(is_gate ? other : v[8 + i]) * sc;
          }
          // unguarded stores for a full 16-column chunk
          uint16_t* hcol = static_cast<uint16_t*>(a.out) + static_cast<int64_t>(td.y + c0 + cb) * a.out_ld + j;
          if (c0 + 16 <= td.z) {
#pragma unroll
            for (int i = 0; i < 8; ++i) hcol[static_cast<int64_t>(i) * a.out_ld] = f32_to_bf16_bits(silu_f32(gv[i]) * uv[i]);
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (c0 + cb + i < td.z) hcol[static_cast<int64_t>(i) * a.out_ld] = f32_to_bf16_bits(silu_f32(gv[i]) * uv[i]);
          }
        } else if (a.y16) {
          // compact y: the raw accumulator times a fixed power of two, as f16 (the combine applies
          // scale2 and the row factor); two operations per element, half the bytes of fp32
          uint16_t* yh = a.y16 + static_cast<int64_t>(td.y + c0) * a.out_ld + mb * kBM + q * 32 + lane;
          if (c0 + 16 <= td.z) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              yh[static_cast<int64_t>(i) * a.out_ld] = __half_as_ushort(__float2half_rn(__uint_as_float(v[i]) * a.y16_scale));
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (c0 + i < td.z)
                yh[static_cast<int64_t>(i) * a.out_ld] = __half_as_ushort(__float2half_rn(__uint_as_float(v[i]) * a.y16_scale));
          }
        } else {
          float* yrow = static_cast<float*>(a.out) + static_cast<int64_t>(td.y + c0) * a.out_ld + mb * kBM +
                        q * 32 + lane;
          float sc[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) sc[i] = __shfl_sync(0xffffffffu, colf, (c0 & 31) + i);
          if (c0 + 16 <= td.z) {   // a full chunk: no per-column checks
#pragma unroll
            for (int i = 0; i < 16; ++i) yrow[static_cast<int64_t>(i) * a.out_ld] = __uint_as_float(v[i]) * sc[i];
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (c0 + i < td.z) yrow[static_cast<int64_t>(i) * a.out_ld] = __uint_as_float(v[i]) * sc[i];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->acc_empty[d]);
      if (item + static_cast<int>(gridDim.x) < n_items) fetch_scales(td_next);
      ++ic;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpTma) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

// ------------------------------------------------------------------ host side
bool make_map_3d(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* ptr, uint64_t d0, uint64_t d1,
                 uint64_t d2, uint64_t stride1, uint64_t stride2, uint32_t b0, uint32_t b1, uint32_t b2,
                 CUtensorMapSwizzle sw) {
  (void)elem_bytes;
  const uint64_t dims[3] = {d0, d1, d2}, strides[2] = {stride1, stride2};
  const uint32_t box[3] = {b0, b1, b2};
  return make_tensor_map(m, dt, 3, ptr, dims, strides, box, sw);
}

bool make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* ptr, uint64_t inner,
                 uint64_t outer, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  const uint64_t dims[2] = {inner, outer}, strides[1] = {inner * elem_bytes};
  const uint32_t box[2] = {box_inner, box_outer};
  return make_tensor_map(m, dt, 2, ptr, dims, strides, box, sw);
}

template <int kBNt>
constexpr size_t smem_bytes() {
  return 1024 + TcCfg<kBNt>::kBStages * TcCfg<kBNt>::kBStageBytes + kAStages * kAStageBytes + sizeof(Smem);
}
static_assert(smem_bytes<128>() <= 232448 && smem_bytes<64>() <= 232448, "shared memory per CTA");

template <bool kGateUp>
cudaError_t launch_tc(const GroupedArgs& g, cudaStream_t st) {
  const bool small = g.tile_rows == 64;
  const bool narrow = g.narrow_rows > 0;
  const void* kern = small ? (narrow ? reinterpret_cast<const void*>(grouped_gemm_tc_kernel<kGateUp, 64, true>)
                                     : reinterpret_cast<const void*>(grouped_gemm_tc_kernel<kGateUp, 64, false>))
                           : (narrow ? reinterpret_cast<const void*>(grouped_gemm_tc_kernel<kGateUp, 128, true>)
                                     : reinterpret_cast<const void*>(grouped_gemm_tc_kernel<kGateUp, 128, false>));
  const size_t smem = small ? smem_bytes<64>() : smem_bytes<128>();
  if (g.tile_rows != 64 && g.tile_rows != kTcTileRows) return cudaErrorInvalidValue;
  cudaError_t e = ensure_dynamic_smem(kern, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int n_sm = 0;
  if ((e = current_sm_count(&n_sm)) != cudaSuccess) return e;
  const int G = g.E + 1;
  const uint64_t rows = static_cast<uint64_t>(G) * g.N;
  const uint64_t act_rows = static_cast<uint64_t>(g.S) + g.T;
  TcMaps maps;
  bool ok = true;
  if (kGateUp) {
    // rows y of the gate half and y + N/2 of the up half; y < rows - N/2 keeps every box of a
    // valid gate row inside the tensor
    const uint64_t half = static_cast<uint64_t>(g.N / 2);
    ok = ok && make_map_3d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.packed, g.K / 2, rows - half, 2, g.K / 2,
                           half * (g.K / 2), kGK / 2, kBM / 2, 2, CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && make_map_3d(&maps.s, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.scales, g.K / 16, rows - half, 2, g.K / 16,
                           half * (g.K / 16), kGK / 16, kBM / 2, 2, CU_TENSOR_MAP_SWIZZLE_NONE);
  } else {
    ok = ok && make_map_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.packed, g.K / 2, rows, kGK / 2, kBM,
                           CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && make_map_2d(&maps.s, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.scales, g.K / 16, rows, kGK / 16, kBM,
                           CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  // activations viewed as {64 columns, rows, K / 64 chunks}: chunk z of row y at y * 2K + 128 z bytes
  for (int i = 0; ok && i < g.tile_rows / 16; ++i)
    ok = make_map_3d(&maps.b[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, g.act, kBK, act_rows, g.K / kBK,
                     static_cast<uint64_t>(g.K) * 2, kBK * 2, kBK, 16 * (i + 1), kGK / kBK,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;
  TcArgs a;
  a.scale2 = g.scale2;
  a.Nw = g.N;
  a.K = g.K;
  a.tiles = g.tiles;
  a.meta = g.meta;
  a.out = g.out;
  a.out_ld = kGateUp ? g.N / 2 : g.N;
  a.act_factor = g.act_factor;
  a.status = g.status;
  a.y16 = kGateUp ? nullptr : g.y16;
  a.y16_scale = g.y16_scale;
  a.y16_rowf = g.y16_rowf;
  a.narrow_rows = g.narrow_rows;
  const int64_t items_max = g.max_tiles * (g.N / kBM);
  const int grid = static_cast<int>(std::min<int64_t>(items_max, n_sm));
  if (g.narrow_rows < 0 || g.narrow_rows > 8) return cudaErrorInvalidValue;   // one MMA column block
  if (small)
    return narrow ? launch_pdl(g.pdl, grouped_gemm_tc_kernel<kGateUp, 64, true>, dim3(grid), dim3(kThreads), smem, st, maps, a)
                  : launch_pdl(g.pdl, grouped_gemm_tc_kernel<kGateUp, 64, false>, dim3(grid), dim3(kThreads), smem, st, maps, a);
  return narrow ? launch_pdl(g.pdl, grouped_gemm_tc_kernel<kGateUp, 128, true>, dim3(grid), dim3(kThreads), smem, st, maps, a)
                : launch_pdl(g.pdl, grouped_gemm_tc_kernel<kGateUp, 128, false>, dim3(grid), dim3(kThreads), smem, st, maps, a);
}

}  // namespace

bool tc_supported(const moe_shape_t& s) { return s.H % 256 == 0 && s.I % 256 == 0 && s.H <= 16384; }

cudaError_t launch_gate_up_tc(const GroupedArgs& a, cudaStream_t st) { return launch_tc<true>(a, st); }
cudaError_t launch_down_tc(const GroupedArgs& a, cudaStream_t st) { return launch_tc<false>(a, st); }

}  // namespace moe
