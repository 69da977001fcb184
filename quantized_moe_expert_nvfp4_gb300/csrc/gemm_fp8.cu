// Grouped e4m3 x e4m3 GEMM on the fifth-generation tensor cores (tcgen05 kind::f8f6f4) -- the
// FP8-activation prefill arm.
//
// The "long-context cold prefill to SGLang parity" issue's transposed kernels multiply weights
// re-quantized to e4m3 by e4m3 activations; its option (a) scales each activation row into the
// e4m3 range and applies the scale in the f32 epilogue.  Here both operands are e4m3 rows with
// one fp32 scale per row (fp8_quant.cu): the weights' rows (re-quantized once, at load time) and
// the activation rows (quantized in the gather), so there is no dequantization in the loop: TMA
// copies both operands into shared memory and the MMA reads them there.
//
// Swap-AB as in the f16 arm: the MMA's M is 128 weight rows of one expert, N up to 128 of that
// expert's tokens.  Per CTA (one per SM, persistent):
//   warp 0      TMA producer of the weight tiles (K = 256 bytes per stage, two 128-byte chunks; a
//               ring of four stages, two items of lookahead for down)
//   warp 1      MMA issuer: one elected lane issues 8 tcgen05.mma kind::f8f6f4 (K = 32) per stage
//   warp 2      TMA producer of the activation tiles
//   warp 3      TMEM allocation
//   warps 4-7   epilogue: tcgen05.ld of the fp32 accumulator x scale2 x weight-row scale x
//               activation-row scale, SiLU(gate)*up (gate_up)
// gate_up takes 16 gate rows and the matching 16 up rows into each 32-row quarter of the tile
// (a 5-D box), so that every epilogue warp holds gate and up of the same intermediate columns.
// Every mbarrier wait is bounded; on timeout the kernel records MOE_ERR_DEVICE_TIMEOUT and winds
// down.
#include "internal.cuh"
#include "tc_common.cuh"
#include "tensor_map.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kBM = 128;                       // weight rows per tile (MMA M)
constexpr int kBN = kTcTileRows;               // tokens per tile at most (MMA N, rounded up to 16)
constexpr int kChunk = 128;                    // K bytes (= elements) per 128-byte swizzled row
constexpr int kSK = 256;                       // K per stage
constexpr int kAStages = 4;                    // weight ring: two items of lookahead at K = 512
constexpr int kBStages = 3;                    // activation ring (mostly L2 hits)
constexpr int kAStage = kBM * kSK;             // 32 KB: [2 chunks][128 rows][128 B]
constexpr int kBStage = kBN * kSK;             // 32 KB: [2 chunks][<= 128 rows][128 B]
constexpr int kTmemCols = 256;                 // two 128-column accumulators
constexpr int kWarpTmaA = 0, kWarpMma = 1, kWarpTmaB = 2, kWarpAlloc = 3, kWarpEpi = 4;
constexpr int kEpiWarps = 4;
constexpr int kThreads = 8 * 32;
constexpr uint32_t kSpinLimit = 1u << 24;      // drain loops only
constexpr uint64_t kWaitTimeoutNs = 1000000000ull;
static_assert(kBN == 128, "the epilogue holds four 32-column groups of row factors");

struct F8Maps {
  CUtensorMap a;                 // weight codes (gate_up: 5-D interleaved gate/up box; down: 3-D)
  CUtensorMap b[kBN / 16];       // activation codes, a box of 16 (i + 1) rows
};

struct F8Args {
  const float* scale2;           // [G]
  const float* row_scale;        // [G, Nw] weight-row scales
  int Nw, K;
  const int4* tiles;
  const int32_t* meta;
  void* out;                     // h [S + T, I] bf16 or y [S + T, H] fp32
  int out_ld;
  const float* act_scale;        // [S + T] activation-row scales (expert order)
  int32_t* status;
  uint16_t* y16;                 // down: compact y, f16(accumulator * row scale * y16_scale), when set,
  float y16_scale;               // and per row the factor that restores it
  float* y16_rowf;
};

struct F8Smem {
  uint64_t a_full[kAStages];     // the weight stage landed
  uint64_t a_empty[kAStages];    // the MMAs reading it completed
  uint64_t b_full[kBStages];     // the activation stage landed
  uint64_t b_empty[kBStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];         // one arrival per epilogue warp
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ bool wait(uint64_t* b, uint32_t parity, F8Smem* sm, int32_t* status) {
  return mbar_wait_flag(b, parity, &sm->abort_flag, status, kWaitTimeoutNs);
}
__device__ __forceinline__ bool warp_wait(uint64_t* b, uint32_t parity, F8Smem* sm, int32_t* status) {
  const bool ok = wait(b, parity, sm, status);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ int4 load_tile(const F8Args& a, int item, int n_items, int MB) {
  return item < n_items ? __ldg(a.tiles + item / MB) : make_int4(0, 0, 0, 0);
}

template <bool kGateUp>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_fp8_kernel(const __grid_constant__ F8Maps maps, F8Args a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;                                  // kAStages x 32 KB
  uint8_t* sB = base + kAStages * kAStage;             // kBStages x 32 KB
  F8Smem* sm = reinterpret_cast<F8Smem*>(sB + kBStages * kBStage);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int MB = a.Nw / kBM;
  const int KS = a.K / kSK;                            // stages per item
  const int n_items = __ldg(a.meta) * MB;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(&sm->a_full[s], 1);
      mbar_init(&sm->a_empty[s], 1);
    }
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(&sm->b_full[s], 1);
      mbar_init(&sm->b_empty[s], 1);
    }
    for (int d = 0; d < 2; ++d) {
      mbar_init(&sm->acc_full[d], 1);
      mbar_init(&sm->acc_empty[d], kEpiWarps);
    }
    mbar_init(&sm->drain, 1);
    sm->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kWarpAlloc) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sm->tmem_base)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;

  if (warp == kWarpTmaA) {
    if (lane == 0) {
      uint32_t is = 0;
      bool ok = true;
      int4 td_next = load_tile(a, blockIdx.x, n_items, MB);
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const int4 td = td_next;
        td_next = load_tile(a, item + gridDim.x, n_items, MB);
        const int mb = item % MB;
        for (int s = 0; s < KS; ++s, ++is) {
          const int st = is % kAStages;
          if (!(ok = wait(&sm->a_empty[st], ((is / kAStages) & 1) ^ 1, sm, a.status))) break;
          mbar_expect_tx(&sm->a_full[st], kAStage);
          if (kGateUp) {
            // {128 B, 16 rows, gate/up half, 16-row block, 128-byte chunk}: gate rows
            // g 2I + 64 mb + 16 rb + r and the up rows I further, for rb < 4
            const int rb0 = (td.x * a.Nw + mb * (kBM / 2)) / 16;
            tma_load_5d(sA + st * kAStage, &maps.a, 0, 0, 0, rb0, s * (kSK / kChunk), &sm->a_full[st]);
          } else {
            tma_load_3d(sA + st * kAStage, &maps.a, 0, td.x * a.Nw + mb * kBM, s * (kSK / kChunk), &sm->a_full[st]);
          }
        }
      }
      if (!ok) {   // let copies already issued land before the CTA winds down (bounded)
        for (int j = 0; j < kAStages && is > 0; ++j, --is) {
          const uint32_t q = is - 1;
          for (uint32_t i = 0; i < (1u << 16) && !mbar_try(&sm->a_full[q % kAStages], (q / kAStages) & 1); ++i) {
          }
        }
      }
    }
  } else if (warp == kWarpTmaB) {
    if (lane == 0) {
      // rows [td.y, td.y + n16) of the expert-ordered activation codes (n16 = the tile's rows
      // rounded up to 16; rows past the tile's own feed accumulator columns the epilogue skips)
      uint32_t is = 0;
      bool ok = true;
      int4 td_next = load_tile(a, blockIdx.x, n_items, MB);
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const int4 td = td_next;
        td_next = load_tile(a, item + gridDim.x, n_items, MB);
        const int n16 = (td.z + 15) >> 4;
        const CUtensorMap* bm = &maps.b[n16 - 1];
        for (int s = 0; s < KS; ++s, ++is) {
          const int st = is % kBStages;
          if (!(ok = wait(&sm->b_empty[st], ((is / kBStages) & 1) ^ 1, sm, a.status))) break;
          mbar_expect_tx(&sm->b_full[st], 2 * n16 * 16 * kChunk);
          tma_load_3d(sB + st * kBStage, bm, 0, td.y, s * (kSK / kChunk), &sm->b_full[st]);
        }
      }
      if (!ok) {
        for (int j = 0; j < kBStages && is > 0; ++j, --is) {
          const uint32_t q = is - 1;
          for (uint32_t i = 0; i < (1u << 16) && !mbar_try(&sm->b_full[q % kBStages], (q / kBStages) & 1); ++i) {
          }
        }
      }
    }
  } else if (warp == kWarpMma) {
    uint32_t is = 0, ic = 0;
    bool ok = true;
    int4 td_next = load_tile(a, blockIdx.x, n_items, MB);
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++ic) {
      const int4 td = td_next;
      td_next = load_tile(a, item + gridDim.x, n_items, MB);
      const int n = (td.z + 15) & ~15;
      const uint32_t idesc = idesc_f32acc(kBM, n);
      const int d = ic & 1;
      if (!(ok = warp_wait(&sm->acc_empty[d], ((ic >> 1) & 1) ^ 1, sm, a.status))) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem + d * kBN;
      for (int s = 0; s < KS; ++s, ++is) {
        const int sa = is % kAStages, sb = is % kBStages;
        if (!(ok = warp_wait(&sm->a_full[sa], (is / kAStages) & 1, sm, a.status))) break;
        if (!(ok = warp_wait(&sm->b_full[sb], (is / kBStages) & 1, sm, a.status))) break;
        tc_fence_after();
        if (elect_one()) {
          const uint32_t a_addr = smem_u32(sA + sa * kAStage);
          const uint32_t b_addr = smem_u32(sB + sb * kBStage);
#pragma unroll
          for (int c = 0; c < kSK / kChunk; ++c) {
#pragma unroll
            for (int kk = 0; kk < kChunk / 32; ++kk) {   // K = 32 e4m3 per MMA (32 bytes of the row)
              const uint64_t ad = smem_desc_sw128(a_addr + c * (kBM * kChunk) + kk * 32);
              const uint64_t bd = smem_desc_sw128(b_addr + c * (n * kChunk) + kk * 32);
              mma_f8(d_tmem, ad, bd, idesc, (s | c | kk) != 0);
            }
          }
          tc_commit(&sm->a_empty[sa]);
          tc_commit(&sm->b_empty[sb]);
        }
        __syncwarp();
      }
      if (ok) {
        if (elect_one()) tc_commit(&sm->acc_full[d]);
        __syncwarp();
      }
    }
    if (elect_one()) {   // every MMA issued completes before TMEM is released (bounded)
      tc_commit(&sm->drain);
      for (uint32_t i = 0; i < kSpinLimit && !mbar_try(&sm->drain, 0); ++i) {
      }
    }
    __syncwarp();
  } else if (warp >= kWarpEpi) {
    const int q = warp & 3;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t ic = 0;
    bool ok = true;
    int4 td_next = load_tile(a, blockIdx.x, n_items, MB);
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++ic) {
      const int4 td = td_next;
      td_next = load_tile(a, item + gridDim.x, n_items, MB);
      const int mb = item % MB;
      const int d = ic & 1;
      // this lane's weight row and its factor scale2 x row scale; the activation-row scales of
      // columns l, l + 32, l + 64, l + 96
      int wrow, j = 0;
      bool is_gate = true;
      if (kGateUp) {
        is_gate = lane < 16;
        j = mb * (kBM / 2) + q * 16 + (lane & 15);            // intermediate column
        wrow = is_gate ? j : (a.Nw / 2) + j;
      } else {
        wrow = mb * kBM + q * 32 + lane;
      }
      const float rowf = __ldg(a.scale2 + td.x) * __ldg(a.row_scale + static_cast<int64_t>(td.x) * a.Nw + wrow);
      float cf[kBN / 32];
#pragma unroll
      for (int i = 0; i < kBN / 32; ++i) cf[i] = (32 * i + lane < td.z) ? __ldg(a.act_scale + td.y + 32 * i + lane) : 0.0f;
      if (!kGateUp && a.y16 && mb == 0 && q == 0) {   // the tile's row factors for the combine
        const float s2 = __ldg(a.scale2 + td.x);
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
        TC_LD16(t_lane + d * kBN + c0, v);
        const int cr = c0 >> 5;
        const float colf = cr == 0 ? cf[0] : cr == 1 ? cf[1] : cr == 2 ? cf[2] : cf[3];
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (kGateUp) {
          // a gate lane finishes columns c0..c0+7 and its up partner (lane ^ 16) c0+8..c0+15,
          // each receiving the other's scaled half by one exchange
          const int cb = is_gate ? 0 : 8;
          float gv[8], uv[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float mine0 = __uint_as_float(v[i]) * rowf, mine1 = __uint_as_float(v[8 + i]) * rowf;
            const float other = __shfl_xor_sync(0xffffffffu, is_gate ? mine1 : mine0, 16);
            const float sc = __shfl_sync(0xffffffffu, colf, (c0 & 31) + cb + i);
            gv[i] = (is_gate ? mine0 : other) * sc;
            uv[i] = (is_gate ? other : mine1) * sc;
          }
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
          // compact y: the accumulator times the weight row's scale and a fixed power of two, as
          // f16 (the combine applies scale2 and the activation row's scale)
          const float f = __ldg(a.row_scale + static_cast<int64_t>(td.x) * a.Nw + wrow) * a.y16_scale;
          uint16_t* yh = a.y16 + static_cast<int64_t>(td.y + c0) * a.out_ld + wrow;
          if (c0 + 16 <= td.z) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              yh[static_cast<int64_t>(i) * a.out_ld] = __half_as_ushort(__float2half_rn(__uint_as_float(v[i]) * f));
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (c0 + i < td.z)
                yh[static_cast<int64_t>(i) * a.out_ld] = __half_as_ushort(__float2half_rn(__uint_as_float(v[i]) * f));
          }
        } else {
          // the column factors first, then the stores: unguarded for a full 16-column chunk (a
          // store guarded per element inside the shuffle sequence cost as much as the MMAs)
          float* yrow = static_cast<float*>(a.out) + static_cast<int64_t>(td.y + c0) * a.out_ld + wrow;
          float sc[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) sc[i] = __shfl_sync(0xffffffffu, colf, (c0 & 31) + i) * rowf;
          if (c0 + 16 <= td.z) {
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
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpAlloc) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

constexpr size_t kSmemBytes = 1024 + kAStages * kAStage + kBStages * kBStage + sizeof(F8Smem);
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

template <bool kGateUp>
cudaError_t launch_fp8(const GroupedFp8Args& g, cudaStream_t st) {
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(grouped_gemm_fp8_kernel<kGateUp>),
                                      static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  int n_sm = 0;
  if ((e = current_sm_count(&n_sm)) != cudaSuccess) return e;
  const uint64_t G = static_cast<uint64_t>(g.E) + 1;
  const uint64_t K = static_cast<uint64_t>(g.K);
  const uint64_t act_rows = static_cast<uint64_t>(g.S) + g.T;
  F8Maps maps;
  bool ok = true;
  if (kGateUp) {
    // {128 B, 16 rows, 2 halves (I rows apart), 16-row blocks, 128-byte chunks}; the block count
    // stops I rows early so that the up half of every valid box stays inside the tensor
    const uint64_t half = static_cast<uint64_t>(g.N / 2);
    const uint64_t blocks = (G * g.N - half) / 16;
    const uint64_t dims[5] = {static_cast<uint64_t>(kChunk), 16, 2, blocks, K / kChunk};
    const uint64_t strides[4] = {K, half * K, 16 * K, static_cast<uint64_t>(kChunk)};
    const uint32_t box[5] = {kChunk, 16, 2, 4, kSK / kChunk};
    ok = make_tensor_map(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, g.codes, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    const uint64_t dims[3] = {static_cast<uint64_t>(kChunk), G * g.N, K / kChunk};
    const uint64_t strides[2] = {K, static_cast<uint64_t>(kChunk)};
    const uint32_t box[3] = {kChunk, kBM, kSK / kChunk};
    ok = make_tensor_map(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, g.codes, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B);
  }
  for (int i = 0; ok && i < kBN / 16; ++i) {
    const uint64_t dims[3] = {static_cast<uint64_t>(kChunk), act_rows, K / kChunk};
    const uint64_t strides[2] = {K, static_cast<uint64_t>(kChunk)};
    const uint32_t box[3] = {kChunk, static_cast<uint32_t>(16 * (i + 1)), kSK / kChunk};
    ok = make_tensor_map(&maps.b[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, g.act, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (!ok) return cudaErrorInvalidValue;
  F8Args a;
  a.scale2 = g.scale2;
  a.row_scale = g.row_scale;
  a.Nw = g.N;
  a.K = g.K;
  a.tiles = g.tiles;
  a.meta = g.meta;
  a.out = g.out;
  a.out_ld = kGateUp ? g.N / 2 : g.N;
  a.act_scale = g.act_scale;
  a.status = g.status;
  a.y16 = kGateUp ? nullptr : g.y16;
  a.y16_scale = g.y16_scale;
  a.y16_rowf = g.y16_rowf;
  const int64_t items_max = g.max_tiles * (g.N / kBM);
  const int grid = static_cast<int>(std::min<int64_t>(items_max, n_sm));
  grouped_gemm_fp8_kernel<kGateUp><<<grid, kThreads, kSmemBytes, st>>>(maps, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gate_up_fp8(const GroupedFp8Args& a, cudaStream_t st) { return launch_fp8<true>(a, st); }
cudaError_t launch_down_fp8(const GroupedFp8Args& a, cudaStream_t st) { return launch_fp8<false>(a, st); }

}  // namespace moe
