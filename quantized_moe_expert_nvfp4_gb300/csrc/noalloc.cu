// moe_forward_decode_static_scratch: the one-launch decode forward for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand the library a workspace: code that runs where cudaMalloc is
// not available or not allowed (for example inside a framework's memory-planning phase that
// forbids new allocations, inside a host callback, or a plugin whose host application owns
// every device allocation and only passes in tensor pointers).  For them this entry point keeps
// its scratch (routing results, the permutation, the decode kernel's h and expert outputs, the
// device status word and the kernel's counters) in one fixed-size array in device global
// memory, declared below at file scope.  It calls no allocator at all.
//
// Costs and rules, in plain terms:
//  - The array is kNoAllocScratchBytes (4 MiB) and exists on every GPU that loads this library,
//    for as long as the library stays loaded.  h and the expert outputs dominate the scratch:
//    T (k + 1) (2 I + 4 H) bytes, 0.8 MB for T = 8, k = 10, I = 512, H = 2048 and at most 2.5 MB
//    for a one-launch decode shape, so every such shape fits (a shape that did not would be
//    rejected).
//  - All calls on a device share the one array.  Calls whose work overlaps on the GPU (two
//    streams, or two host threads) race on it and produce garbage; serialize them.
//  - The first call in a context looks up the array's device address (cudaGetSymbolAddress); a
//    caller that makes another context current gets that context's own lookup.  Make that first
//    call outside any CUDA stream capture.
//  - A device reset is not supported: the library links its own static copy of the CUDA
//    runtime, which does not see a cudaDeviceReset (or primary-context reset) made by other code
//    in the process, so neither this array nor the library's kernels are reloaded after one.
//    The library must be unloaded (or the process restarted) after such a reset.
//  - Each call clears the status word, the launch counter and the decode kernel's other
//    synchronisation words at the start (an asynchronous memset on the caller's stream, not an allocation), so a
//    device-side timeout of one call does not poison the next; such a timeout is not reported
//    back by this entry point.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.cuh"

namespace moe {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t{4} << 20;

// The scratch itself.  In host code `g_noalloc_scratch` is only a host-side stand-in for the
// symbol; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

size_t up256(size_t x) { return (x + 255) & ~size_t{255}; }

struct Carve {
  size_t meta, fdsync, ids, w, counts, offsets, sorted, slot_pos, fdscr, total;
};

Carve carve_for(const moe_shape_t& s) {
  Carve c{};
  const size_t S = static_cast<size_t>(s.T) * s.k;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = up256(off + bytes);
    return o;
  };
  c.meta = take(256);        // [0] status word, [2..3] the decode kernel's 64-bit launch count
  c.fdsync = take(4 * static_cast<size_t>(kFdSyncWords));   // the decode kernel's sync words
  c.ids = take(4 * S);
  c.w = take(4 * S);
  c.counts = take(4 * static_cast<size_t>(s.E));
  c.offsets = take(4 * static_cast<size_t>(s.E + 1));
  c.sorted = take(4 * S);
  c.slot_pos = take(4 * S);
  c.fdscr = take(fd_scratch_bytes(s));   // the decode kernel's h and expert outputs
  c.total = off;
  return c;
}

bool ok16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The current context's unique id, or 0 when no context is current on this thread yet
// (cuCtxGetCurrent + cuCtxGetId, reached through the runtime's driver entry-point query, so the
// library needs no link against the driver library).
cudaError_t current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  *id = 0;
  if (!get_current || !get_id) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  if (!ctx) return cudaSuccess;
  return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

// Device address of the scratch array in the current context.  It is looked up once per device
// with that device current (cudaGetSymbolAddress) and kept together with the id of the context it
// was taken in: when a caller makes another context current (the module, and so the array, sits
// at another address there) the lookup is made again.
void* scratch_address(cudaError_t* err) {
  static std::mutex mu;
  static void* addr[64] = {};
  static unsigned long long ctx_of[64] = {};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess || dev < 0 || dev >= 64) {
    if (*err == cudaSuccess) *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  unsigned long long ctx = 0;
  if ((*err = current_context_id(&ctx)) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev] || ctx == 0 || ctx_of[dev] != ctx) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);   // binds the device's context if none was
    if (*err != cudaSuccess) return nullptr;
    if ((*err = current_context_id(&ctx)) != cudaSuccess) return nullptr;
    addr[dev] = p;
    ctx_of[dev] = ctx;
  }
  return addr[dev];
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_forward_decode_static_scratch(const uint16_t* x, const float* logits,
                                                          const moe_nvfp4_weights_t* gate_up,
                                                          const moe_nvfp4_weights_t* down,
                                                          const moe_shape_t* shape, void* out,
                                                          int out_is_fp32, void* stream) {
  if (!shape || !gate_up || !down) return MOE_ERR_INVALID_ARG;
  if (moe_workspace_size(shape) == 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  const moe_shape_t& s = *shape;
  if (s.T == 0) return MOE_OK;
  if (moe_forward_arm(shape) != 0) return MOE_ERR_UNSUPPORTED_SHAPE;   // one-launch decode shapes only
  if (!ok16(x) || !ok16(logits) || !ok16(out) || (out_is_fp32 != 0 && out_is_fp32 != 1))
    return MOE_ERR_INVALID_ARG;
  const int G = s.E + s.has_shared;
  if (!ok16(gate_up->packed) || !ok16(gate_up->scales) || !ok16(gate_up->scale2) || gate_up->G != G ||
      gate_up->N != 2 * s.I || gate_up->K != s.H)
    return MOE_ERR_INVALID_ARG;
  if (!ok16(down->packed) || !ok16(down->scales) || !ok16(down->scale2) || down->G != G || down->N != s.H ||
      down->K != s.I)
    return MOE_ERR_INVALID_ARG;
  const Carve c = carve_for(s);
  if (c.total > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED_SHAPE;   // scratch would not fit

  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return MOE_ERR_ARCH;
  {   // the stream must belong to the current device (the default stream handles always do; a
      // stream being captured is not asked: the query would invalidate the capture)
    const cudaStream_t cs0 = static_cast<cudaStream_t>(stream);
    int sdev = -1;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cs0 != nullptr && cs0 != cudaStreamLegacy && cs0 != cudaStreamPerThread) {
      if (cudaStreamIsCapturing(cs0, &cap) != cudaSuccess) return MOE_ERR_INVALID_ARG;
      if (cap == cudaStreamCaptureStatusNone && (cudaStreamGetDevice(cs0, &sdev) != cudaSuccess || sdev != dev))
        return MOE_ERR_INVALID_ARG;
    }
  }
  cudaError_t e = cudaSuccess;
  char* base = static_cast<char*>(scratch_address(&e));
  if (!base) return MOE_ERR_CUDA;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // the status word, the launch counter and the sync words must start at zero
  e = cudaMemsetAsync(base + c.meta, 0, c.ids - c.meta, cs);
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  DecodeFusedArgs f;
  f.x = x;
  f.logits = logits;
  f.gate_up = *gate_up;
  f.down = *down;
  f.shape = s;
  f.ids = reinterpret_cast<int32_t*>(base + c.ids);
  f.topk_w = reinterpret_cast<float*>(base + c.w);
  f.counts = reinterpret_cast<int32_t*>(base + c.counts);
  f.offsets = reinterpret_cast<int32_t*>(base + c.offsets);
  f.sorted_slot = reinterpret_cast<int32_t*>(base + c.sorted);
  f.slot_pos = reinterpret_cast<int32_t*>(base + c.slot_pos);
  f.scratch = base + c.fdscr;
  f.sync = reinterpret_cast<unsigned*>(base + c.fdsync);
  f.out = out;
  f.out_is_fp32 = out_is_fp32;
  f.grid_ctr = reinterpret_cast<unsigned long long*>(base + c.meta + 8);
  f.status = reinterpret_cast<int32_t*>(base + c.meta);
  return launch_decode_fused(f, cs) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
