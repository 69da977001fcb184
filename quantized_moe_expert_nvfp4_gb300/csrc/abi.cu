// C ABI of the NVFP4 routed-MoE library: argument validation, workspace layout and the
// choice of arm.  Host code only; every stage runs in the kernels of the other files.
#include <algorithm>
#include <atomic>

#include <cmath>

#include "internal.cuh"

namespace moe {
namespace {

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status_t check_shape(const moe_shape_t* s) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (s->T < 0 || s->H < 128 || s->H > 16384 || s->H % 128 || s->I < 128 || s->I > 8192 ||
      s->I % 128 || s->E < 1 || s->E > kMaxE || s->k < 1 || s->k > kMaxK || s->k > s->E ||
      (s->has_shared != 0 && s->has_shared != 1))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<int64_t>(s->T) * (s->k + 1) >= (int64_t{1} << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

moe_status_t check_weights(const moe_nvfp4_weights_t* w, const moe_shape_t& s, bool gate_up) {
  if (!w || !aligned16(w->packed) || !aligned16(w->scales) || !aligned16(w->scale2))
    return MOE_ERR_INVALID_ARG;
  const int N = gate_up ? 2 * s.I : s.H, K = gate_up ? s.H : s.I;
  if (w->G != s.E + s.has_shared || w->N != N || w->K != K) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status_t check_ws(const void* ws, size_t ws_bytes, const moe_shape_t& s) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < ws_layout(s).total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return MOE_OK;
}

// The current device must be compute capability 10.3 (GB300).  Cached per device.
moe_status_t check_arch() {
  static std::atomic<int> cache[64];  // 0 unknown, 1 ok, 2 wrong arch
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c == 1) return MOE_OK;
    if (c == 2) return MOE_ERR_ARCH;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  const bool ok = (major == 10 && minor == 3);
  if (dev >= 0 && dev < 64) cache[dev].store(ok ? 1 : 2, std::memory_order_relaxed);
  return ok ? MOE_OK : MOE_ERR_ARCH;
}

// The current device must be compute capability 10.3 and `stream` must belong to it (a stream
// created on another device would run the launches there, against pointers of this one).  The
// legacy and per-thread default stream handles always name the current device.  A stream that
// is being captured is not asked (the query is not allowed during capture and would invalidate
// it); the graph's launches then run on whatever stream the graph is launched into.
moe_status_t check_device(void* stream) {
  moe_status_t st = check_arch();
  if (st != MOE_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (cs == nullptr || cs == cudaStreamLegacy || cs == cudaStreamPerThread) return MOE_OK;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(cs, &cap) != cudaSuccess) return MOE_ERR_INVALID_ARG;
  if (cap != cudaStreamCaptureStatusNone) return MOE_OK;
  int dev = 0, sdev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamGetDevice(cs, &sdev) != cudaSuccess) return MOE_ERR_INVALID_ARG;
  return sdev == dev ? MOE_OK : MOE_ERR_INVALID_ARG;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

struct Ws {
  int32_t* status;
  int32_t* meta;
  int32_t* ids;
  float* w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted_slot;
  int32_t* slot_pos;
  int4* tiles;
  int32_t* hist;
  uint16_t* h;
  float* y;
  uint16_t* xf;
  float* xe;
  uint16_t* hf;
  float* he;
  uint16_t* rxf;
  float* rxe;
  float* rlogits;
  WsLayout L;
};

Ws carve(void* ws, const moe_shape_t& s) {
  Ws r;
  r.L = ws_layout(s);
  char* b = static_cast<char*>(ws);
  r.status = reinterpret_cast<int32_t*>(b + r.L.status);
  r.meta = reinterpret_cast<int32_t*>(b + r.L.meta);
  r.ids = reinterpret_cast<int32_t*>(b + r.L.ids);
  r.w = reinterpret_cast<float*>(b + r.L.w);
  r.counts = reinterpret_cast<int32_t*>(b + r.L.counts);
  r.offsets = reinterpret_cast<int32_t*>(b + r.L.offsets);
  r.sorted_slot = reinterpret_cast<int32_t*>(b + r.L.sorted_slot);
  r.slot_pos = reinterpret_cast<int32_t*>(b + r.L.slot_pos);
  r.tiles = reinterpret_cast<int4*>(b + r.L.tiles);
  r.hist = reinterpret_cast<int32_t*>(b + r.L.hist);
  r.h = reinterpret_cast<uint16_t*>(b + r.L.h);
  r.y = reinterpret_cast<float*>(b + r.L.y);
  r.xf = reinterpret_cast<uint16_t*>(b + r.L.xf);
  r.xe = reinterpret_cast<float*>(b + r.L.xe);
  r.hf = reinterpret_cast<uint16_t*>(b + r.L.hf);
  r.he = reinterpret_cast<float*>(b + r.L.he);
  r.rxf = reinterpret_cast<uint16_t*>(b + r.L.rxf);
  r.rxe = reinterpret_cast<float*>(b + r.L.rxe);
  r.rlogits = reinterpret_cast<float*>(b + r.L.rlogits);
  return r;
}

// Arm of a shape: the grouped-GEMV decode arms for up to kFdMaxT tokens; above that the tcgen05
// grouped GEMM when H and I are multiples of 256 (it streams the selected experts' weights at
// least as fast as the GEMV arm once an expert sees more than a few tokens), else the CUDA-core
// GEMV arm up to kDecodeMaxT tokens and the CUDA-core grouped GEMM beyond.
enum class Arm { kDecode, kTc, kSimt };

Arm arm_for(const moe_shape_t& s) {
  if (s.T <= kFdMaxT) return Arm::kDecode;
  if (tc_supported(s)) return Arm::kTc;
  return s.T <= kDecodeMaxT ? Arm::kDecode : Arm::kSimt;
}

// Which kernels moe_forward runs for a shape (the value moe_forward_arm reports).
int forward_arm(const moe_shape_t& s) {
  switch (arm_for(s)) {
    case Arm::kDecode: return (s.T <= kFdMaxT && decode_fused_supported(s)) ? 0 : 1;
    case Arm::kTc: return 2;
    default: return 3;
  }
}

int tile_rows_for(const moe_shape_t& s) {
  switch (arm_for(s)) {
    case Arm::kDecode: return kDecodeMaxT;
    case Arm::kTc: return s.T <= kDecodeMaxT ? 64 : kTcTileRows;   // 64-row tiles for small batches
    default: return kSimtTileRows;
  }
}

// Row bound of the tensor-core arm's register arm (tiles of at most this many rows run on the
// dequant warps with mma.sync; set by moe_set_narrow_rows, -1 = the library's default).
std::atomic<int> g_narrow_rows{-1};
constexpr int kNarrowMaxRows = 8;

int narrow_rows_for(const moe_shape_t& s) {
  if (arm_for(s) != Arm::kTc) return 0;
  const int set = g_narrow_rows.load(std::memory_order_relaxed);
  if (set >= 0) return set;
  return 0;
}

// The tensor-core arm takes its activations as f16 rows with power-of-two row exponents, in
// expert order: x is gathered by sorted_slot and converted into the workspace first (h already
// is in order).  moe_forward writes the same rows token-major from the inverse map instead.
cudaError_t launch_gate_up(GroupedArgs a, const moe_shape_t& s, const Ws& ws, cudaStream_t cs) {
  if (arm_for(s) != Arm::kTc) return launch_gate_up_simt(a, cs);
  cudaError_t e = launch_act_gather_f16(a.act, a.sorted_slot, s.T, s.k, s.H, ws.xf, ws.xe, ws.status, cs);
  if (e != cudaSuccess) return e;
  a.act = ws.xf;
  a.act_factor = ws.xe;
  return launch_gate_up_tc(a, cs);
}

cudaError_t launch_down(GroupedArgs a, const moe_shape_t& s, const Ws& ws, cudaStream_t cs) {
  if (arm_for(s) != Arm::kTc) return launch_down_simt(a, cs);
  cudaError_t e = launch_act_to_f16(a.act, ws.hf, ws.he, static_cast<int64_t>(s.T) * s.k + s.T, s.I, a.pdl, cs);
  if (e != cudaSuccess) return e;
  a.act = ws.hf;
  a.act_factor = ws.he;
  return launch_down_tc(a, cs);
}

GroupedArgs grouped_args(const moe_nvfp4_weights_t& w, const moe_shape_t& s, const uint16_t* act,
                         const int32_t* sorted_slot, const Ws& ws, void* out) {
  GroupedArgs a;
  a.packed = w.packed;
  a.scales = w.scales;
  a.scale2 = w.scale2;
  a.N = w.N;
  a.K = w.K;
  a.act = act;
  a.sorted_slot = sorted_slot;
  a.T = s.T;
  a.k = s.k;
  a.S = s.T * s.k;
  a.E = s.E;
  a.tiles = ws.tiles;
  a.meta = ws.meta;
  a.max_tiles = max_tiles_for(s, tile_rows_for(s));
  a.tile_rows = tile_rows_for(s);
  a.narrow_rows = narrow_rows_for(s);
  a.out = out;
  a.status = ws.status;
  a.act_factor = nullptr;
  return a;
}

// Routing, permutation and work list of the grouped-GEMM arms: one cooperative launch.
cudaError_t launch_route_permute(const float* logits, const moe_shape_t& s, const Ws& w, int tile_rows,
                                 cudaStream_t cs) {
  return launch_route_permute_large(logits, nullptr, s.T, s.E, s.k, s.has_shared, w.ids, w.w, w.counts, w.offsets,
                                    w.sorted_slot, w.slot_pos, w.hist, w.tiles, w.meta, tile_rows, w.status, cs);
}

// The router GEMM runs on the tcgen05 grouped GEMM (one group of E weight rows) for batches
// above the decode sizes when E and H fit its tiles, else on the CUDA-core kernel.
// The CUDA-core router up to 32 tokens (measured on GB300 at H = 2048, E = 512: 5.8 us against
// 11.2 us for the tensor-core path's three launches at T = 8..32; 14.2 against 12.2 at T = 64).
constexpr int kRouterSimtMaxT = 32;
bool router_on_tc(const moe_shape_t& s) { return s.T > kRouterSimtMaxT && s.E % 128 == 0 && s.H % 256 == 0; }

moe_status_t check_router(const moe_nvfp4_weights_t* r, const moe_shape_t& s) {
  if (!r || !aligned16(r->packed) || !aligned16(r->scales) || !aligned16(r->scale2)) return MOE_ERR_INVALID_ARG;
  if (r->G != 1 || r->N != s.E || r->K != s.H) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

}  // namespace

// Work items of a shape: sum_e ceil(c_e / R) <= S / R + (number of non-empty experts), and the
// shared expert adds ceil(T / R).
int64_t max_tiles_for(const moe_shape_t& s, int tile_rows) {
  const int64_t S = static_cast<int64_t>(s.T) * s.k;
  const int64_t routed = S / tile_rows + std::min<int64_t>(S, s.E);
  const int64_t shared = s.has_shared ? (s.T + tile_rows - 1) / tile_rows : 0;
  return std::max<int64_t>(1, routed + shared);
}

WsLayout ws_layout(const moe_shape_t& s) {
  WsLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  const int64_t S = static_cast<int64_t>(s.T) * s.k;
  const int64_t R = S + s.T;
  L.status = take(256);
  L.meta = take(256);
  L.fdsync = take(4 * kFdSyncWords);
  L.ids = take(4 * S);
  L.w = take(4 * S);
  L.counts = take(4 * static_cast<size_t>(s.E));
  L.offsets = take(4 * static_cast<size_t>(s.E + 1));
  L.sorted_slot = take(4 * S);
  L.slot_pos = take(4 * S);
  L.max_tiles = std::max(max_tiles_for(s, kSimtTileRows), max_tiles_for(s, kDecodeMaxT));
  L.tiles = take(16 * static_cast<size_t>(L.max_tiles));
  L.hist = take(4 * static_cast<size_t>(kPermuteMaxGrid) * s.E);
  // moe_forward's intermediates, by arm: h for arms 1-3, fp32 y for arms 2-3, the f16 operands
  // for arm 2, the decode kernel's h and expert outputs for arm 0
  const int arm = forward_arm(s);
  L.h = take(arm != 0 ? 2 * static_cast<size_t>(R) * s.I : 0);
  L.y = take(arm >= 2 ? 4 * static_cast<size_t>(R) * s.H : 0);
  const size_t tc_rows = arm_for(s) == Arm::kTc ? static_cast<size_t>(R) : 0;   // tensor-core arm only
  L.xf = take(2 * tc_rows * s.H);
  L.xe = take(4 * tc_rows);
  L.hf = take(2 * tc_rows * s.I);
  L.he = take(4 * tc_rows);
  L.fdscr = take(arm == 0 ? fd_scratch_bytes(s) : 0);
  // the router GEMM (moe_router_logits, moe_forward_routed)
  L.rxf = take(router_on_tc(s) ? 2 * static_cast<size_t>(s.T) * s.H : 0);
  L.rxe = take(router_on_tc(s) ? 4 * static_cast<size_t>(s.T) : 0);
  L.rlogits = take(4 * static_cast<size_t>(s.T) * s.E);
  L.total = off;
  return L;
}

}  // namespace moe

namespace moe {
namespace {

// logits [T, E] of the router; ws is a checked workspace of the shape.
cudaError_t launch_router(const uint16_t* x, const moe_nvfp4_weights_t& r, const moe_shape_t& s, float* logits,
                          const Ws& w, cudaStream_t cs) {
  if (!router_on_tc(s)) return launch_router_simt(x, r, s.T, s.H, s.E, logits, cs);
  // one group of E weight rows against the T rows of x, f16 operands (x scaled per row)
  uint16_t* xf = w.rxf;
  float* xe = w.rxe;
  cudaError_t e = launch_act_to_f16(x, xf, xe, s.T, s.H, false, cs);
  if (e == cudaSuccess) e = launch_dense_tiles(s.T, kTcTileRows, w.tiles, w.meta, cs);
  if (e != cudaSuccess) return e;
  GroupedArgs a;
  a.packed = r.packed;
  a.scales = r.scales;
  a.scale2 = r.scale2;
  a.N = s.E;
  a.K = s.H;
  a.act = xf;
  a.sorted_slot = nullptr;
  a.T = s.T;
  a.k = 0;
  a.S = 0;
  a.E = 0;   // one group
  a.tiles = w.tiles;
  a.meta = w.meta;
  a.max_tiles = (s.T + kTcTileRows - 1) / kTcTileRows;
  a.out = logits;
  a.status = w.status;
  a.act_factor = xe;
  return launch_down_tc(a, cs);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

moe_status_t moe_set_narrow_rows(int rows) {
  if (rows < -1 || rows > kNarrowMaxRows) return MOE_ERR_INVALID_ARG;
  g_narrow_rows.store(rows, std::memory_order_relaxed);
  return MOE_OK;
}

size_t moe_workspace_size(const moe_shape_t* shape) {
  if (check_shape(shape) != MOE_OK) return 0;
  return ws_layout(*shape).total;
}

moe_status_t moe_route_topk(const float* logits, const moe_shape_t* shape, int32_t* topk_ids,
                            float* topk_w, void* stream) {
  moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (!aligned16(logits) || !aligned16(topk_ids) || !aligned16(topk_w)) return MOE_ERR_INVALID_ARG;
  if (shape->T == 0) return MOE_OK;
  if ((st = check_device(stream)) != MOE_OK) return st;
  return cuda_status(launch_route_topk(logits, shape->T, shape->E, shape->k, topk_ids, topk_w, false,
                                       static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_permute(const int32_t* topk_ids, const moe_shape_t* shape, int32_t* counts,
                         int32_t* offsets, int32_t* sorted_slot, int32_t* slot_pos, void* ws,
                         size_t ws_bytes, void* stream) {
  moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (!aligned16(topk_ids) || !aligned16(counts) || !aligned16(offsets) ||
      !aligned16(sorted_slot) || !aligned16(slot_pos))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(ws, ws_bytes, *shape)) != MOE_OK) return st;
  if ((st = check_device(stream)) != MOE_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const moe_shape_t& s = *shape;
  if (s.T == 0) {  // offsets of an empty batch are all zero
    cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * s.E, cs);
    if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (s.E + 1), cs);
    return cuda_status(e);
  }
  Ws w = carve(ws, s);
  if (s.T <= kDecodeMaxT)
    return cuda_status(launch_route_permute_small(nullptr, topk_ids, s.T, s.E, s.k, s.has_shared,
                                                  nullptr, nullptr, counts, offsets, sorted_slot,
                                                  slot_pos, w.tiles, w.meta, kDecodeMaxT, cs));
  return cuda_status(launch_route_permute_large(nullptr, topk_ids, s.T, s.E, s.k, s.has_shared, nullptr,
                                                nullptr, counts, offsets, sorted_slot, slot_pos, w.hist,
                                                w.tiles, w.meta, tile_rows_for(s), w.status, cs));
}

moe_status_t moe_grouped_gate_up(const uint16_t* x, const int32_t* sorted_slot,
                                 const int32_t* offsets, const moe_nvfp4_weights_t* gate_up,
                                 const moe_shape_t* shape, uint16_t* h, void* ws, size_t ws_bytes,
                                 void* stream) {
  moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (!aligned16(x) || !aligned16(sorted_slot) || !aligned16(offsets) || !aligned16(h))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_weights(gate_up, *shape, true)) != MOE_OK) return st;
  if ((st = check_ws(ws, ws_bytes, *shape)) != MOE_OK) return st;
  if (shape->T == 0) return MOE_OK;
  if ((st = check_device(stream)) != MOE_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const moe_shape_t& s = *shape;
  Ws w = carve(ws, s);
  cudaError_t e = launch_build_tiles(offsets, s.T, s.E, s.k, s.has_shared, tile_rows_for(s),
                                     w.tiles, w.meta, w.status, cs);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(launch_gate_up(grouped_args(*gate_up, s, x, sorted_slot, w, h), s, w, cs));
}

moe_status_t moe_grouped_down(const uint16_t* h, const int32_t* offsets,
                              const moe_nvfp4_weights_t* down, const moe_shape_t* shape,
                              float* y, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (!aligned16(h) || !aligned16(offsets) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  if ((st = check_weights(down, *shape, false)) != MOE_OK) return st;
  if ((st = check_ws(ws, ws_bytes, *shape)) != MOE_OK) return st;
  if (shape->T == 0) return MOE_OK;
  if ((st = check_device(stream)) != MOE_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const moe_shape_t& s = *shape;
  Ws w = carve(ws, s);
  cudaError_t e = launch_build_tiles(offsets, s.T, s.E, s.k, s.has_shared, tile_rows_for(s),
                                     w.tiles, w.meta, w.status, cs);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(launch_down(grouped_args(*down, s, h, nullptr, w, y), s, w, cs));
}

moe_status_t moe_combine(const float* y, const int32_t* slot_pos, const float* topk_w,
                         const moe_shape_t* shape, void* out, int out_is_fp32, void* stream) {
  moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (!aligned16(y) || !aligned16(slot_pos) || !aligned16(topk_w) || !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  if (out_is_fp32 != 0 && out_is_fp32 != 1) return MOE_ERR_INVALID_ARG;
  if (shape->T == 0) return MOE_OK;
  if ((st = check_device(stream)) != MOE_OK) return st;
  return cuda_status(launch_combine(y, slot_pos, topk_w, shape->T, shape->H, shape->k,
                                    shape->has_shared, out, out_is_fp32, nullptr,
                                    static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_forward(const uint16_t* x, const float* logits,
                         const moe_nvfp4_weights_t* gate_up, const moe_nvfp4_weights_t* down,
                         const moe_shape_t* shape, void* out, int out_is_fp32, void* ws,
                         size_t ws_bytes, void* stream) {
  return moe_forward_profiled(x, logits, gate_up, down, shape, out, out_is_fp32, ws, ws_bytes,
                              stream, nullptr);
}

moe_status_t moe_forward_profiled(const uint16_t* x, const float* logits,
                                  const moe_nvfp4_weights_t* gate_up,
                                  const moe_nvfp4_weights_t* down, const moe_shape_t* shape,
                                  void* out, int out_is_fp32, void* ws, size_t ws_bytes,
                                  void* stream, void* const* stage_events) {
  moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (!aligned16(x) || !aligned16(logits) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  if (out_is_fp32 != 0 && out_is_fp32 != 1) return MOE_ERR_INVALID_ARG;
  if ((st = check_weights(gate_up, *shape, true)) != MOE_OK) return st;
  if ((st = check_weights(down, *shape, false)) != MOE_OK) return st;
  if ((st = check_ws(ws, ws_bytes, *shape)) != MOE_OK) return st;
  if (shape->T == 0) return MOE_OK;
  if ((st = check_device(stream)) != MOE_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const moe_shape_t& s = *shape;
  Ws w = carve(ws, s);
  // Under stream capture the records become external event nodes of the graph; otherwise they
  // are plain records (the external flag is refused on the legacy default stream).
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (stage_events && cudaStreamIsCapturing(cs, &cap) != cudaSuccess) return MOE_ERR_CUDA;
  const unsigned rec_flags = cap == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
  auto mark = [&](int i) -> cudaError_t {
    return stage_events ? cudaEventRecordWithFlags(static_cast<cudaEvent_t>(stage_events[i]), cs, rec_flags)
                        : cudaSuccess;
  };
  cudaError_t e = mark(0);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (forward_arm(s) == 0) {
    // decode arm, one cooperative launch: route, permute, gate_up, down, combine
    DecodeFusedArgs f;
    f.x = x;
    f.logits = logits;
    f.gate_up = *gate_up;
    f.down = *down;
    f.shape = s;
    f.ids = w.ids;
    f.topk_w = w.w;
    f.counts = w.counts;
    f.offsets = w.offsets;
    f.sorted_slot = w.sorted_slot;
    f.slot_pos = w.slot_pos;
    f.scratch = reinterpret_cast<char*>(ws) + w.L.fdscr;
    f.sync = reinterpret_cast<unsigned*>(reinterpret_cast<char*>(ws) + w.L.fdsync);
    f.out = out;
    f.out_is_fp32 = out_is_fp32;
    f.grid_ctr = reinterpret_cast<unsigned long long*>(w.meta + 2);
    f.status = w.status;
    e = launch_decode_fused(f, cs);
    for (int i = 1; i <= 4 && e == cudaSuccess; ++i) e = mark(i);
    return cuda_status(e);
  }
  if (arm_for(s) == Arm::kDecode) {
    // decode arm for larger batches: 1) route + permute + work list, 2) gate_up GEMV (+SiLU*up)
    // of every active group incl. the shared expert, 3) down GEMV + fixed-order combine.
    e = launch_route_permute_small(logits, nullptr, s.T, s.E, s.k, s.has_shared, w.ids, w.w,
                                   w.counts, w.offsets, w.sorted_slot, w.slot_pos, w.tiles, w.meta,
                                   kDecodeMaxT, cs);
    if (e == cudaSuccess) e = mark(1);
    if (e == cudaSuccess) e = launch_gate_up_simt(grouped_args(*gate_up, s, x, w.sorted_slot, w, w.h), cs);
    if (e == cudaSuccess) e = mark(2);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    DownCombineArgs d;
    d.packed = down->packed;
    d.scales = down->scales;
    d.scale2 = down->scale2;
    d.H = s.H;
    d.I = s.I;
    d.T = s.T;
    d.k = s.k;
    d.S = s.T * s.k;
    d.E = s.E;
    d.h = w.h;
    d.slot_pos = w.slot_pos;
    d.topk_w = w.w;
    d.tiles = w.tiles;
    d.meta = w.meta;
    d.max_tiles = max_tiles_for(s, kDecodeMaxT);
    d.has_shared = s.has_shared;
    d.out = out;
    d.out_is_fp32 = out_is_fp32;
    d.status = w.status;
    e = launch_down_combine_gemv(d, cs);
    if (e == cudaSuccess) e = mark(3);
    if (e == cudaSuccess) e = mark(4);
    return cuda_status(e);
  }
  // grouped-GEMM arms: routing, permutation and work list in one cooperative launch
  // (on the tensor-core arm also the expert-ordered f16 rows of x, written token-major from the
  // inverse map so that each x row is read once; stage event 1 follows them)
  // (batches of up to kDecodeMaxT tokens on the tensor-core arm: the top-k, then permutation, work
  // list and the f16 rows of x in one launch whose CTAs each place the whole batch, with no
  // grid-wide wait)
  const bool tc = arm_for(s) == Arm::kTc;
  const bool small_tc = tc && s.T <= kDecodeMaxT;   // its kernels launch with programmatic dependencies
  if (small_tc) {
    e = launch_route_topk(logits, s.T, s.E, s.k, w.ids, w.w, true, cs);
    if (e == cudaSuccess)
      e = launch_permute_gather_small(w.ids, x, s.T, s.E, s.k, s.has_shared, s.H, w.counts, w.offsets, w.sorted_slot,
                                      w.slot_pos, w.tiles, w.meta, tile_rows_for(s), w.xf, w.xe, w.status, cs);
  } else {
    e = launch_route_permute(logits, s, w, tile_rows_for(s), cs);
    if (e == cudaSuccess && tc) e = launch_act_scatter_f16(x, w.slot_pos, s.T, s.k, s.H, w.xf, w.xe, w.status, cs);
  }
  if (e == cudaSuccess) e = mark(1);
  if (e == cudaSuccess) {
    GroupedArgs ga = grouped_args(*gate_up, s, x, w.sorted_slot, w, w.h);
    if (tc) {
      ga.act = w.xf;
      ga.act_factor = w.xe;
      ga.pdl = small_tc;
      e = launch_gate_up_tc(ga, cs);
    } else {
      e = launch_gate_up_simt(ga, cs);
    }
  }
  if (e == cudaSuccess) e = mark(2);
  // The tensor-core arm hands y to the combine compact: f16 of the raw down accumulator times
  // 2^-c, c fixed by the accumulator's bound (|e2m1 x e4m3| <= 2688 and the f16 rows of h below
  // 2^15, so |acc| <= I * 2688 * 2^15 and |acc| * 2^-c stays below f16's maximum); the values keep
  // f16's 11 significant bits, and the combine multiplies them by scale2 * (h row factor) * 2^c.
  const int64_t R = static_cast<int64_t>(s.T) * s.k + s.T;
  uint16_t* y16 = tc ? reinterpret_cast<uint16_t*>(w.y) : nullptr;
  float* rowf = tc ? reinterpret_cast<float*>(y16 + R * s.H) : nullptr;   // after the f16 rows, in the y region
  if (e == cudaSuccess) {
    GroupedArgs da = grouped_args(*down, s, w.h, nullptr, w, w.y);
    if (tc) {
      const int c = static_cast<int>(std::ceil(std::log2(static_cast<double>(s.I) * 2688.0 * 32768.0 / 65504.0)));
      da.y16 = y16;
      da.y16_scale = std::ldexp(1.0f, -c);
      da.y16_rowf = rowf;
      da.pdl = small_tc;
    }
    e = launch_down(da, s, w, cs);
  }
  if (e == cudaSuccess) e = mark(3);
  if (e == cudaSuccess)
    e = tc ? launch_combine_y16(y16, rowf, w.slot_pos, w.w, s.T, s.H, s.k, s.has_shared, out, out_is_fp32, w.status,
                                small_tc, cs)
           : launch_combine(w.y, w.slot_pos, w.w, s.T, s.H, s.k, s.has_shared, out, out_is_fp32, w.status, cs);
  if (e == cudaSuccess) e = mark(4);
  return cuda_status(e);
}


moe_status_t moe_router_logits(const uint16_t* x, const moe_nvfp4_weights_t* router, const moe_shape_t* shape,
                               float* logits, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (!aligned16(x) || !aligned16(logits)) return MOE_ERR_INVALID_ARG;
  if ((st = check_router(router, *shape)) != MOE_OK) return st;
  if ((st = check_ws(ws, ws_bytes, *shape)) != MOE_OK) return st;
  if (shape->T == 0) return MOE_OK;
  if ((st = check_device(stream)) != MOE_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  Ws w = carve(ws, *shape);
  return cuda_status(launch_router(x, *router, *shape, logits, w, cs));
}

moe_status_t moe_forward_routed(const uint16_t* x, const moe_nvfp4_weights_t* router,
                                const moe_nvfp4_weights_t* gate_up, const moe_nvfp4_weights_t* down,
                                const moe_shape_t* shape, void* out, int out_is_fp32, void* ws, size_t ws_bytes,
                                void* stream) {
  moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (!aligned16(x) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  if ((st = check_router(router, *shape)) != MOE_OK) return st;
  if ((st = check_ws(ws, ws_bytes, *shape)) != MOE_OK) return st;
  if (shape->T == 0) return MOE_OK;
  if ((st = check_device(stream)) != MOE_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  Ws w = carve(ws, *shape);
  if (launch_router(x, *router, *shape, w.rlogits, w, cs) != cudaSuccess) return MOE_ERR_CUDA;
  return moe_forward(x, w.rlogits, gate_up, down, shape, out, out_is_fp32, ws, ws_bytes, stream);
}

moe_status_t moe_prepare_fp8(const moe_nvfp4_weights_t* w, uint8_t* codes, float* row_scale, void* stream) {
  if (!w || !aligned16(w->packed) || !aligned16(w->scales) || !aligned16(codes) || !aligned16(row_scale))
    return MOE_ERR_INVALID_ARG;
  if (w->G < 1 || w->N < 1 || w->K < 256 || w->K % 256 || w->K > 16384) return MOE_ERR_UNSUPPORTED_SHAPE;
  moe_status_t st = check_device(stream);
  if (st != MOE_OK) return st;
  return cuda_status(launch_prepare_fp8(w->packed, w->scales, static_cast<int64_t>(w->G) * w->N, w->K, codes,
                                        row_scale, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_quantize_rows_e4m3(const uint16_t* x, int64_t rows, int32_t K, uint8_t* codes, float* scale,
                                    void* stream) {
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scale)) return MOE_ERR_INVALID_ARG;
  if (rows < 0 || K < 256 || K % 256 || K > 16384) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return MOE_OK;
  moe_status_t st = check_device(stream);
  if (st != MOE_OK) return st;
  return cuda_status(launch_act_quant_fp8(x, nullptr, 0, 1, rows, K, codes, scale, nullptr,
                                          static_cast<cudaStream_t>(stream)));
}

namespace {
moe_status_t check_fp8_weights(const moe_fp8_weights_t* w, const moe_shape_t& s, bool gate_up) {
  if (!w || !aligned16(w->codes) || !aligned16(w->row_scale) || !aligned16(w->scale2)) return MOE_ERR_INVALID_ARG;
  const int N = gate_up ? 2 * s.I : s.H, K = gate_up ? s.H : s.I;
  if (w->G != s.E + s.has_shared || w->N != N || w->K != K) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

GroupedFp8Args fp8_args(const moe_fp8_weights_t& w, const moe_shape_t& s, const Ws& ws, const uint8_t* act,
                        const float* act_scale, void* out) {
  GroupedFp8Args a;
  a.codes = w.codes;
  a.row_scale = w.row_scale;
  a.scale2 = w.scale2;
  a.N = w.N;
  a.K = w.K;
  a.act = act;
  a.act_scale = act_scale;
  a.T = s.T;
  a.k = s.k;
  a.S = s.T * s.k;
  a.E = s.E;
  a.tiles = ws.tiles;
  a.meta = ws.meta;
  a.max_tiles = max_tiles_for(s, kTcTileRows);
  a.out = out;
  a.status = ws.status;
  return a;
}
}  // namespace

moe_status_t moe_forward_fp8(const uint16_t* x, const float* logits, const moe_fp8_weights_t* gate_up,
                             const moe_fp8_weights_t* down, const moe_shape_t* shape, void* out, int out_is_fp32,
                             void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (arm_for(*shape) != Arm::kTc) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(logits) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  if (out_is_fp32 != 0 && out_is_fp32 != 1) return MOE_ERR_INVALID_ARG;
  if ((st = check_fp8_weights(gate_up, *shape, true)) != MOE_OK) return st;
  if ((st = check_fp8_weights(down, *shape, false)) != MOE_OK) return st;
  if ((st = check_ws(ws, ws_bytes, *shape)) != MOE_OK) return st;
  if ((st = check_device(stream)) != MOE_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const moe_shape_t& s = *shape;
  Ws w = carve(ws, s);
  // the e4m3 operands reuse the f16 operands' regions (one byte per element instead of two)
  uint8_t* xq = reinterpret_cast<uint8_t*>(w.xf);
  uint8_t* hq = reinterpret_cast<uint8_t*>(w.hf);
  const int S = s.T * s.k;
  const int64_t R = static_cast<int64_t>(S) + s.T;
  cudaError_t e = launch_route_permute(logits, s, w, kTcTileRows, cs);
  if (e == cudaSuccess) e = launch_act_scatter_fp8(x, w.slot_pos, s.T, s.k, s.H, xq, w.xe, w.status, cs);
  if (e == cudaSuccess) e = launch_gate_up_fp8(fp8_args(*gate_up, s, w, xq, w.xe, w.h), cs);
  if (e == cudaSuccess) e = launch_act_quant_fp8(w.h, nullptr, 0, 1, R, s.I, hq, w.he, w.status, cs);
  // y compact as on the W4A16 tensor-core arm: f16(acc * weight-row scale * 2^-c), with
  // |acc| <= I * 448^2 and the row scale <= 2688 / 448 (an NVFP4 row's largest value over 448)
  const int c = static_cast<int>(std::ceil(std::log2(static_cast<double>(s.I) * 448.0 * 448.0 * 6.0 / 65504.0)));
  uint16_t* y16 = reinterpret_cast<uint16_t*>(w.y);
  float* rowf = reinterpret_cast<float*>(y16 + R * s.H);
  if (e == cudaSuccess) {
    GroupedFp8Args da = fp8_args(*down, s, w, hq, w.he, w.y);
    da.y16 = y16;
    da.y16_scale = std::ldexp(1.0f, -c);
    da.y16_rowf = rowf;
    e = launch_down_fp8(da, cs);
  }
  if (e == cudaSuccess)
    e = launch_combine_y16(y16, rowf, w.slot_pos, w.w, s.T, s.H, s.k, s.has_shared, out, out_is_fp32, w.status, false,
                           cs);
  return cuda_status(e);
}

moe_status_t moe_quantize_nvfp4(const float* w, int64_t G, int64_t N, int64_t K, uint8_t* packed,
                                uint8_t* scales, float* scale2, void* stream) {
  if (!aligned16(w) || !aligned16(packed) || !aligned16(scales) || !aligned16(scale2))
    return MOE_ERR_INVALID_ARG;
  if (G < 1 || G > 65535 || N < 1 || K < 16 || K % 16 || N * K > (int64_t{1} << 40))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  moe_status_t st = check_device(stream);
  if (st != MOE_OK) return st;
  return cuda_status(launch_quantize(w, G, N, K, packed, scales, scale2,
                                     static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_get_device_status(void* ws, int32_t* status, void* stream) {
  if (!ws || !status || (reinterpret_cast<uintptr_t>(ws) & 255u)) return MOE_ERR_INVALID_ARG;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof(int32_t), cs);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  *status = v;
  return MOE_OK;
}

moe_status_t moe_debug_timeout_probe(void* ws, uint64_t limit_ns, void* stream) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return MOE_ERR_INVALID_ARG;
  if (limit_ns < 1 || limit_ns > 1000000000ull) return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_device(stream);
  if (st != MOE_OK) return st;
  return cuda_status(launch_fd_timeout_probe(static_cast<int32_t*>(ws), limit_ns, static_cast<cudaStream_t>(stream)));
}

int moe_forward_arm(const moe_shape_t* shape) {
  if (check_shape(shape) != MOE_OK) return -1;
  return forward_arm(*shape);
}

const char* moe_status_string(moe_status_t status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null/misaligned pointer or inconsistent struct)";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_ARCH: return "current device is not compute capability 10.3 (sm_103)";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side bounded wait timed out";
  }
  return "unknown status";
}

}  // extern "C"
