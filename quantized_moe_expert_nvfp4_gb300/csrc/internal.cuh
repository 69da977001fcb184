// Internal declarations of the NVFP4 routed-MoE library (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>
#include <utility>

#include "moe_nvfp4.h"

namespace moe {

// ------------------------------------------------------------------ limits and arm choice
constexpr int kMaxK = 16;
constexpr int kMaxE = 1024;
constexpr int kDecodeMaxT = 64;        // moe_forward uses the grouped-GEMV arm up to this T
constexpr int kSimtTileRows = 64;      // rows per work item of the SIMT grouped GEMM
constexpr int kTcTileRows = 128;       // tokens per work item of the tcgen05 grouped GEMM
constexpr int kPermuteMaxGrid = 256;   // CTAs of the one-launch permutation (histogram rows)
constexpr int kFdMaxT = 8;             // the fused single-launch decode kernel handles T <= 8
constexpr int kFdSlice = 64;           // intermediate columns of one work unit of that kernel
// its sync words: two units-done counters, one per launch parity, then per launch parity one
// gate_up-units-done counter per active expert (each launch zeroes the other parity's words)
constexpr int kFdSyncWords = 512;
constexpr int kFdMaxAct = 160;         // active experts of one decode launch (at most T * k + 1), rounded up

// ------------------------------------------------------------------ workspace layout
// All offsets are in bytes from the workspace base and 256-byte aligned.
struct WsLayout {
  size_t status;       // int32 device status word (+ padding)
  size_t meta;         // int32 meta[8]: [0] = number of work tiles, [2..3] 64-bit launch count
  size_t fdsync;       // uint32 [kFdSyncWords] one-launch decode arm: its units-done counters
                       // and per-expert h counters (each launch zeroes the next launch's)
  size_t ids;          // int32 [S]
  size_t w;            // fp32  [S]
  size_t counts;       // int32 [E]
  size_t offsets;      // int32 [E + 1]
  size_t sorted_slot;  // int32 [S]
  size_t slot_pos;     // int32 [S]
  size_t tiles;        // int4  [max_tiles] work items {group, row_begin, rows, 0}
  size_t hist;         // int32 [kPermuteMaxGrid, E] per-CTA expert histograms of the permutation
  size_t h;            // bf16  [S + T, I]  (moe_forward on arms 1-3)
  size_t y;            // fp32  [S + T, H]  (moe_forward on arms 2-3)
  size_t xf;           // f16   [S + T, H]  tensor-core arm: scaled rows of x in expert order
  size_t xe;           // fp32  [S + T]    2^e of each row of xf
  size_t hf;           // f16   [S + T, I]  tensor-core arm: scaled copy of h, and its row exponents
  size_t he;           // fp32  [S + T]    2^e of each row of hf
  size_t fdscr;        // one-launch decode arm: h [S + T][I] bf16, then y [S + T][H] fp32
  size_t rxf;          // f16   [T, H]  router GEMM on the tensor cores: scaled rows of x
  size_t rxe;          // fp32  [T]     and their factors 2^e
  size_t rlogits;      // fp32  [T, E]  moe_forward_routed: the router's logits
  size_t total;
  int64_t max_tiles;
};

WsLayout ws_layout(const moe_shape_t& s);
int64_t max_tiles_for(const moe_shape_t& s, int tile_rows);

// Codes a kernel writes into the workspace status word (first error wins).
enum DeviceError : int32_t {
  kDevOk = 0,
  kDevBadIndex = MOE_ERR_INVALID_ARG,   // an index array (offsets, sorted_slot, slot_pos) out of range
  kDevTimeout = MOE_ERR_DEVICE_TIMEOUT
};

// ------------------------------------------------------------------ device helpers
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Eight e2m1 codes in a 32-bit word (element i in bits 4i..4i+3) -> four f16x2 words holding
// elements (0, 1), (2, 3), (4, 5), (6, 7), the lower element in the low half; exact, since every
// e2m1 value is an f16 value.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// The same eight codes -> eight exact fp32 values.
__device__ __forceinline__ void e2m1x8_to_f32(uint32_t w, float (&v)[8]) {
  uint32_t h[4];
  e2m1x8_to_f16x2(w, h);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[i]));
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  const __half_raw hr = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(byte), __NV_E4M3);
  return __half2float(__half(hr));
}

// Programmatic dependent launch (the kernels of one layer call follow each other on a stream):
// a kernel launched with launch_pdl may start while the previous kernel drains; before touching
// global memory it waits for that kernel's completion and the visibility of its writes
// (griddepcontrol.wait, a no-op when the launch has no programmatic dependency).  Kernels of a
// single wave of CTAs (the persistent GEMMs, the small routing kernels) then let their successor
// be scheduled at once (pdl_wait_then_release), so that its launch and shared-memory / TMEM set-up
// overlap their work; kernels of many waves do not (pdl_wait), because a successor scheduled early
// would take the SM resources their later waves need.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_then_release() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launches kern, with a programmatic dependency on the stream's previous kernel when pdl is set
// (moe_forward sets it for batches of up to kDecodeMaxT tokens, where launch latency is a visible
// share of the layer; on larger batches the early-resident successors cost the GEMMs more than the
// overlap gains, measured on GB300).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

__device__ __forceinline__ float silu_f32(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ void report_device_error(int32_t* status, int32_t code) {
  atomicCAS(status, 0, code);
}

// ------------------------------------------------------------------ per-device host state
// SM count of the current device (cached per device).
cudaError_t current_sm_count(int* n);
// Raises `kernel`'s dynamic shared-memory limit on the current device to at least `bytes`, once
// per (device, kernel) and size; thread-safe.
cudaError_t ensure_dynamic_smem(const void* kernel, int bytes);

// ------------------------------------------------------------------ launchers
// Each returns cudaGetLastError() of its launches.
cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, bool pdl,
                              cudaStream_t st);
// Single-CTA routing + permutation + work list for small T (decode arm).
cudaError_t launch_route_permute_small(const float* logits, const int32_t* ids_in, int T, int E,
                                       int k, int has_shared, int32_t* ids, float* w,
                                       int32_t* counts, int32_t* offsets, int32_t* sorted_slot,
                                       int32_t* slot_pos, int4* tiles, int32_t* meta,
                                       int tile_rows, cudaStream_t st);
// One cooperative launch for any T: routing (logits != NULL) or given ids, counts, offsets, the
// stable permutation and the work list.  hist: [kPermuteMaxGrid, E]; meta[4..5] is its barrier
// counter (zero in a new workspace).
// After the top-k of a batch of T <= kDecodeMaxT tokens: permutation, work list and the
// expert-ordered f16 rows of x (as act_scatter_f16) in one launch of min(T, SMs) CTAs without a
// grid-wide wait.
cudaError_t launch_permute_gather_small(const int32_t* ids, const uint16_t* x, int T, int E, int k, int has_shared,
                                        int H, int32_t* counts, int32_t* offsets, int32_t* sorted_slot,
                                        int32_t* slot_pos, int4* tiles, int32_t* meta, int tile_rows, uint16_t* xf,
                                        float* xe, int32_t* status, cudaStream_t st);
cudaError_t launch_route_permute_large(const float* logits, const int32_t* ids_in, int T, int E, int k,
                                      int has_shared, int32_t* ids, float* w, int32_t* counts,
                                      int32_t* offsets, int32_t* sorted_slot, int32_t* slot_pos,
                                      int32_t* hist, int4* tiles, int32_t* meta, int tile_rows,
                                      int32_t* status, cudaStream_t st);
// Work list from offsets: one item per (group, run of <= tile_rows rows).
// Offsets that are not a valid exclusive prefix (offsets[0] = 0, non-decreasing, offsets[E] = S)
// produce no routed work and record kDevBadIndex.
cudaError_t launch_build_tiles(const int32_t* offsets, int T, int E, int k, int has_shared,
                               int tile_rows, int4* tiles, int32_t* meta, int32_t* status,
                               cudaStream_t st);

struct GroupedArgs {
  const uint8_t* packed;
  const uint8_t* scales;
  const float* scale2;
  int N, K;                     // weight rows and reduction length
  const uint16_t* act;          // x [T, H] (gate_up) or h [S + T, I] (down)
  const int32_t* sorted_slot;   // gate_up: routed row -> slot (token = slot / k)
  int T, k, S, E;
  const int4* tiles;
  const int32_t* meta;
  int64_t max_tiles;
  void* out;                    // h [S + T, I] bf16 (gate_up) or y [S + T, H] fp32 (down)
  int32_t* status;              // device status word (bad indices are clamped and reported)
  const float* act_factor;      // tensor-core arm: 2^e of each f16 act row
  int tile_rows = kTcTileRows;  // tensor-core arm: rows per work item of the list (64 or 128)
  // tensor-core down inside moe_forward: y stored compact as f16(acc * y16_scale), the raw fp32
  // accumulator times a power of two fixed by its bound, and per row the factor that restores it
  // (scale2 * activation row factor / y16_scale), for launch_combine_y16
  uint16_t* y16 = nullptr;
  float y16_scale = 0.0f;
  float* y16_rowf = nullptr;
  // tensor-core arm: work items of at most this many rows (<= 8) run on the dequant warps'
  // register arm inside the same launch (0: every item on tcgen05)
  int narrow_rows = 0;
  bool pdl = false;             // launched with a programmatic dependency (see launch_pdl)
};
cudaError_t launch_gate_up_simt(const GroupedArgs& a, cudaStream_t st);
cudaError_t launch_down_simt(const GroupedArgs& a, cudaStream_t st);
// bf16 rows -> f16 rows scaled by 2^-e[row] (e = floor(log2 max|row|) - 14), for the f16 MMAs.
cudaError_t launch_act_to_f16(const uint16_t* src, uint16_t* dst, float* factor, int64_t rows, int K, bool pdl,
                              cudaStream_t st);
// The same for the gate_up operand, gathered into expert order: row p < S of dst is token
// sorted_slot[p] / k of x, row S + t is token t (out-of-range slots are reported as kDevBadIndex).
cudaError_t launch_act_gather_f16(const uint16_t* x, const int32_t* sorted_slot, int T, int k, int K,
                                  uint16_t* dst, float* factor, int32_t* status, cudaStream_t st);
// The same rows written token-major from the inverse map (slot_pos): every x row is read once.
// k < 32.
cudaError_t launch_act_scatter_f16(const uint16_t* x, const int32_t* slot_pos, int T, int k, int K, uint16_t* dst,
                                   float* factor, int32_t* status, cudaStream_t st);
// tcgen05 grouped GEMM (work items from a tile list built with kTcTileRows rows); act is the
// expert-ordered f16 operand [S + T, K] (launch_act_gather_f16 for gate_up, launch_act_to_f16
// of h for down) and act_factor its row factors 2^e.
bool tc_supported(const moe_shape_t& s);
cudaError_t launch_gate_up_tc(const GroupedArgs& a, cudaStream_t st);
cudaError_t launch_down_tc(const GroupedArgs& a, cudaStream_t st);

// FP8-activation arm: e4m3 rows with one fp32 scale each (fp8_quant.cu) on tcgen05 kind::f8f6f4
// (gemm_fp8.cu).  Same work list as the f16 tensor-core arm.
struct GroupedFp8Args {
  const uint8_t* codes;         // weights [G, N, K] e4m3
  const float* row_scale;       // [G, N]
  const float* scale2;          // [G]
  int N, K;
  const uint8_t* act;           // expert-ordered activation codes [S + T, K]
  const float* act_scale;       // [S + T]
  int T, k, S, E;
  const int4* tiles;
  const int32_t* meta;
  int64_t max_tiles;
  void* out;                    // h [S + T, I] bf16 (gate_up) or y [S + T, H] fp32 (down)
  int32_t* status;
  // down inside moe_forward_fp8: y compact as f16(accumulator * weight-row scale * y16_scale),
  // and per row the factor that restores it (scale2 * activation row scale / y16_scale)
  uint16_t* y16 = nullptr;
  float y16_scale = 0.0f;
  float* y16_rowf = nullptr;
};
cudaError_t launch_gate_up_fp8(const GroupedFp8Args& a, cudaStream_t st);
cudaError_t launch_down_fp8(const GroupedFp8Args& a, cudaStream_t st);
// Weight rows [rows, K] (NVFP4 packed/scales) -> e4m3 codes [rows, K] and row scales [rows].
cudaError_t launch_prepare_fp8(const uint8_t* packed, const uint8_t* scales, int64_t rows, int K, uint8_t* codes,
                               float* row_scale, cudaStream_t st);
// bf16 rows -> e4m3 codes + row scales; with sorted_slot, gathered into expert order as
// launch_act_gather_f16 does.
cudaError_t launch_act_quant_fp8(const uint16_t* src, const int32_t* sorted_slot, int S, int k, int64_t rows, int K,
                                 uint8_t* dst, float* scale, int32_t* status, cudaStream_t st);
// Token-major from slot_pos, as launch_act_scatter_f16.  k < 32.
cudaError_t launch_act_scatter_fp8(const uint16_t* x, const int32_t* slot_pos, int T, int k, int K, uint8_t* dst,
                                   float* scale, int32_t* status, cudaStream_t st);

struct DownCombineArgs {
  const uint8_t* packed;
  const uint8_t* scales;
  const float* scale2;
  int H, I, T, k, S, E;
  const uint16_t* h;            // [S + T, I]
  const int32_t* slot_pos;
  const float* topk_w;
  const int4* tiles;
  const int32_t* meta;
  int64_t max_tiles;
  int has_shared;
  void* out;
  int out_is_fp32;
  int32_t* status;
};
cudaError_t launch_down_combine_gemv(const DownCombineArgs& a, cudaStream_t st);

// status may be NULL (bad slot positions are then clamped silently).
// Single-launch decode arm (route + gate_up + down + combine, cooperative, T <= kFdMaxT).
struct DecodeFusedArgs {
  const uint16_t* x;
  const float* logits;
  moe_nvfp4_weights_t gate_up, down;
  moe_shape_t shape;
  int32_t* ids;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted_slot;
  int32_t* slot_pos;
  void* scratch;                    // fd_scratch_bytes(shape): h and y of the launch, 256-byte aligned
  unsigned* sync;                   // [kFdSyncWords] its counters (the kernel zeroes them itself)
  void* out;
  int out_is_fp32;
  unsigned long long* grid_ctr;     // 64-bit launch count (zero in a new workspace)
  int32_t* status;
};
bool decode_fused_supported(const moe_shape_t& s);
// Bytes of scratch the one-launch decode kernel needs: h [S + T][I] bf16 and y [S + T][H] fp32
// (0 if unsupported).
size_t fd_scratch_bytes(const moe_shape_t& s);
// One warp running the decode kernel's bounded wait on a barrier nothing arrives at (test hook).
cudaError_t launch_fd_timeout_probe(int32_t* status, uint64_t limit_ns, cudaStream_t st);
cudaError_t launch_decode_fused(const DecodeFusedArgs& d, cudaStream_t st);

cudaError_t launch_combine(const float* y, const int32_t* slot_pos, const float* topk_w, int T,
                           int H, int k, int has_shared, void* out, int out_is_fp32,
                           int32_t* status, cudaStream_t st);
// The same sum over the tensor-core down's compact y: row p's values are f16 * rowf[p].
cudaError_t launch_combine_y16(const uint16_t* y16, const float* rowf, const int32_t* slot_pos, const float* topk_w,
                               int T, int H, int k, int has_shared, void* out, int out_is_fp32, int32_t* status,
                               bool pdl, cudaStream_t st);
// Router GEMM on the CUDA cores: logits [T, E] fp32 = scale2 * x . deq(W)^T, W one NVFP4
// projection of E rows of H (H % 16 == 0).
cudaError_t launch_router_simt(const uint16_t* x, const moe_nvfp4_weights_t& w, int T, int H, int E, float* logits,
                               cudaStream_t st);
// Work list of a one-group GEMM over rows [0, rows) in items of tile_rows (meta[0] = count).
cudaError_t launch_dense_tiles(int rows, int tile_rows, int4* tiles, int32_t* meta, cudaStream_t st);

cudaError_t launch_quantize(const float* w, int64_t G, int64_t N, int64_t K, uint8_t* packed,
                            uint8_t* scales, float* scale2, cudaStream_t st);

}  // namespace moe
