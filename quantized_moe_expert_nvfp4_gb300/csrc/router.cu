// Router GEMM in front of the top-k: logits[t, e] = scale2 * (x[t] . deq(W_r[e])), fp32.
//
// The "long-context cold prefill to SGLang parity" issue counts the router GEMM among the MoE's
// logit-changing operations and its nsys table times the router as a W4A16 GEMM; here the router
// weights are one NVFP4 projection (E rows of H, the experts' layout) and the activations bf16.
// Large batches run on the tcgen05 grouped GEMM as one group of E weight rows (see abi.cu); this
// file holds the CUDA-core kernel for the other shapes (decode batches, E or H not multiples of
// the tensor-core tiles) and the work list of the one-group GEMM.
#include "internal.cuh"

namespace moe {
namespace {

constexpr int kRtWarps = 8;     // router rows per CTA (one warp each)
constexpr int kRtTokens = 4;    // tokens per CTA

// One warp per router row e, four tokens; lane l takes the 16-element blocks l, l + 32, ...;
// each block: the 16 exact e2m1 values times the e4m3 scale, dotted with the bf16 activations
// in fp32, then the warp's partial sums meet in a butterfly.
__global__ void __launch_bounds__(kRtWarps * 32) router_simt_kernel(const uint16_t* __restrict__ x,
                                                                    const uint8_t* __restrict__ packed,
                                                                    const uint8_t* __restrict__ scales,
                                                                    const float* __restrict__ scale2, int T,
                                                                    int H, int E, float* __restrict__ logits) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRtWarps + warp;
  const int t0 = blockIdx.y * kRtTokens;
  if (e >= E) return;
  const int nt = min(kRtTokens, T - t0);
  const int nblk = H / 16;
  const uint8_t* prow = packed + static_cast<int64_t>(e) * (H / 2);
  const uint8_t* srow = scales + static_cast<int64_t>(e) * nblk;
  float acc[kRtTokens] = {0.0f, 0.0f, 0.0f, 0.0f};
  // four blocks per lane and pass, their weight and scale loads issued together
  for (int b0 = lane; b0 < nblk; b0 += 4 * 32) {
    uint2 q[4];
    uint32_t sb[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int b = b0 + 32 * u;
      q[u] = b < nblk ? __ldg(reinterpret_cast<const uint2*>(prow) + b) : make_uint2(0u, 0u);
      sb[u] = b < nblk ? __ldg(srow + b) : 0u;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int b = b0 + 32 * u;
      if (b >= nblk) break;
      const float s = e4m3_to_f32(sb[u]);
      float w[16];
      {
        float lo[8], hi[8];
        e2m1x8_to_f32(q[u].x, lo);
        e2m1x8_to_f32(q[u].y, hi);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          w[i] = lo[i];
          w[8 + i] = hi[i];
        }
      }
#pragma unroll
      for (int t = 0; t < kRtTokens; ++t) {
        if (t < nt) {
          const uint4* xp = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t0 + t) * H + 16 * b);
          const uint4 a0 = __ldg(xp), a1 = __ldg(xp + 1);
          const uint32_t v[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
          float d = 0.0f;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            d = fmaf(w[2 * i], bf16_bits_to_f32(v[i] & 0xffffu), d);
            d = fmaf(w[2 * i + 1], bf16_bits_to_f32(v[i] >> 16), d);
          }
          acc[t] = fmaf(d, s, acc[t]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kRtTokens; ++t)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
  if (lane < nt) {
    const float s2 = __ldg(scale2);
    float v = acc[0];
#pragma unroll
    for (int t = 1; t < kRtTokens; ++t)
      if (lane == t) v = acc[t];
    logits[static_cast<int64_t>(t0 + lane) * E + e] = v * s2;
  }
}

// Work list of a one-group GEMM over rows [0, rows): items {0, 128 i, rows in the item, 0}.
__global__ void __launch_bounds__(256) dense_tiles_kernel(int rows, int tile_rows, int4* __restrict__ tiles,
                                                          int32_t* __restrict__ meta) {
  const int n = (rows + tile_rows - 1) / tile_rows;
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    tiles[i] = make_int4(0, i * tile_rows, min(tile_rows, rows - i * tile_rows), 0);
  if (threadIdx.x == 0) meta[0] = n;
}

}  // namespace

cudaError_t launch_router_simt(const uint16_t* x, const moe_nvfp4_weights_t& w, int T, int H, int E, float* logits,
                               cudaStream_t st) {
  const dim3 grid((E + kRtWarps - 1) / kRtWarps, (T + kRtTokens - 1) / kRtTokens);
  router_simt_kernel<<<grid, kRtWarps * 32, 0, st>>>(x, w.packed, w.scales, w.scale2, T, H, E, logits);
  return cudaGetLastError();
}

cudaError_t launch_dense_tiles(int rows, int tile_rows, int4* tiles, int32_t* meta, cudaStream_t st) {
  dense_tiles_kernel<<<1, 256, 0, st>>>(rows, tile_rows, tiles, meta);
  return cudaGetLastError();
}

}  // namespace moe
