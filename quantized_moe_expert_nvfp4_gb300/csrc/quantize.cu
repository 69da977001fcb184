// Load-time NVFP4 quantizer with the recipe of the benchmark configurations (per-tensor
// scale2 = amax / (448*6); per-16-block e4m3 scale = block amax / 6 / scale2; e2m1 codes by
// round-to-nearest-even of w / (e4m3(scale) * scale2)).  Every step is one IEEE fp32 operation
// (explicit _rn intrinsics, no contraction) so the codes are reproducible bit for bit.
#include <algorithm>

#include "internal.cuh"

namespace moe {
namespace {

// e2m1 round-to-nearest-even with saturation at 6, from the midpoints of the magnitudes
// {0, .5, 1, 1.5, 2, 3, 4, 6}: a midpoint goes to the neighbour whose mantissa bit is 0.
__device__ __forceinline__ uint32_t e2m1_rne(float v) {
  const float a = fabsf(v);
  uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
               (a >= 3.5f) + (a > 5.0f);
  return c | (signbit(v) ? 8u : 0u);
}

__global__ void amax_kernel(const float* __restrict__ w, int64_t per_group,
                            unsigned int* __restrict__ amax_bits) {
  const int g = blockIdx.y;
  const float* wg = w + static_cast<int64_t>(g) * per_group;
  float m = 0.0f;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < per_group;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    m = fmaxf(m, fabsf(wg[i]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0) atomicMax(amax_bits + g, __float_as_uint(m));  // m >= 0
}

__global__ void scale2_kernel(float* scale2, int64_t G) {
  const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (g < G) scale2[g] = __fdiv_rn(__uint_as_float(__float_as_uint(scale2[g])), 2688.0f);
}

// One thread per 16-element block.
__global__ void quantize_blocks_kernel(const float* __restrict__ w, int64_t G, int64_t N,
                                       int64_t K, const float* __restrict__ scale2,
                                       uint8_t* __restrict__ packed, uint8_t* __restrict__ scales) {
  const int64_t nb = K / 16;
  const int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (b >= G * N * nb) return;
  const int64_t g = b / (N * nb);
  const float s2 = scale2[g];
  const float4* src = reinterpret_cast<const float4*>(w + b * 16);
  float v[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 f = src[i];
    v[4 * i] = f.x;
    v[4 * i + 1] = f.y;
    v[4 * i + 2] = f.z;
    v[4 * i + 3] = f.w;
  }
  float bamax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) bamax = fmaxf(bamax, fabsf(v[i]));
  uint32_t sc = 0;
  if (s2 > 0.0f) {
    const float ratio = __fdiv_rn(__fdiv_rn(bamax, 6.0f), s2);
    sc = __nv_cvt_float_to_fp8(ratio, __NV_SATFINITE, __NV_E4M3);
  }
  scales[b] = static_cast<uint8_t>(sc);
  const float d = __fmul_rn(e4m3_to_f32(sc), s2);
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t c = (d != 0.0f) ? e2m1_rne(__fdiv_rn(v[i], d)) : 0u;
    if (i < 8)
      lo |= c << (4 * i);
    else
      hi |= c << (4 * (i - 8));
  }
  *reinterpret_cast<uint2*>(packed + b * 8) = make_uint2(lo, hi);
}

}  // namespace

cudaError_t launch_quantize(const float* w, int64_t G, int64_t N, int64_t K, uint8_t* packed,
                            uint8_t* scales, float* scale2, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(scale2, 0, sizeof(float) * G, st);
  if (e != cudaSuccess) return e;
  const int64_t per_group = N * K;
  const unsigned bx = static_cast<unsigned>(std::min<int64_t>(1024, (per_group + 255) / 256));
  amax_kernel<<<dim3(bx, static_cast<unsigned>(G)), 256, 0, st>>>(
      w, per_group, reinterpret_cast<unsigned int*>(scale2));
  scale2_kernel<<<static_cast<unsigned>((G + 255) / 256), 256, 0, st>>>(scale2, G);
  const int64_t nblocks = G * N * (K / 16);
  quantize_blocks_kernel<<<static_cast<unsigned>((nblocks + 255) / 256), 256, 0, st>>>(
      w, G, N, K, scale2, packed, scales);
  return cudaGetLastError();
}

}  // namespace moe
