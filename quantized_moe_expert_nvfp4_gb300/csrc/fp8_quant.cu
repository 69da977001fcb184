// Quantizers of the FP8-activation arm.
//
// The "long-context cold prefill to SGLang parity" issue runs its transposed prefill kernels as
// e4m3 x e4m3: the NVFP4 weights re-quantized to e4m3 and e4m3 activations; its fix option (a)
// gives every token row its own scale (the row absmax, computed in the gather) and applies it in
// the f32 epilogue.  Both operands here follow one row rule:
//   amax = max |v| over the row, inv = 448 / amax and scale = amax / 448 (one IEEE fp32
//   division each; a row whose amax is 0 or not finite gets inv = scale = 1),
//   code = e4m3 round-to-nearest-even, saturating at 448, of the fp32 product v * inv,
// so the row's value is scale * e4m3(code).  A weight row's values are the exact NVFP4 values
// e2m1 x e4m3(block scale); the group's scale2 stays a separate fp32 factor of the epilogue.
// Every step is one IEEE operation (explicit _rn intrinsics), so the codes are reproducible
// bit for bit.
#include "internal.cuh"

namespace moe {
namespace {

__device__ __forceinline__ void row_rule(float amax, float& inv, float& scale) {
  if (amax > 0.0f && amax <= 3.402823466e38f) {
    inv = __fdiv_rn(448.0f, amax);
    scale = __fdiv_rn(amax, 448.0f);
  } else {
    inv = 1.0f;
    scale = 1.0f;
  }
}

// Two fp32 values times inv -> two e4m3 codes (nearest even, saturating), first in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b, float inv) {
  const float2 q = make_float2(__fmul_rn(a, inv), __fmul_rn(b, inv));
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(q, __NV_SATFINITE, __NV_E4M3));
}

// One warp per weight row of [G, N, K] (K % 256 == 0): two passes over the row's packed codes
// and block scales, the amax of the exact values, then the codes.
__global__ void __launch_bounds__(256) prepare_fp8_kernel(const uint8_t* __restrict__ packed,
                                                          const uint8_t* __restrict__ scales, int64_t rows, int K,
                                                          uint8_t* __restrict__ codes, float* __restrict__ row_scale) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (r >= rows) return;
  const uint2* pr = reinterpret_cast<const uint2*>(packed + r * (K / 2));   // one 16-element block per uint2
  const uint8_t* sr = scales + r * (K / 16);
  const int nblk = K / 16;
  float m = 0.0f;
  for (int b = lane; b < nblk; b += 32) {
    const uint2 q = __ldg(pr + b);
    const float s = e4m3_to_f32(__ldg(sr + b));
    float lo[8], hi[8];
    e2m1x8_to_f32(q.x, lo);
    e2m1x8_to_f32(q.y, hi);
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fmaxf(fabsf(lo[i] * s), fabsf(hi[i] * s)));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float inv, scale;
  row_rule(m, inv, scale);
  if (lane == 0) row_scale[r] = scale;
  uint4* dst = reinterpret_cast<uint4*>(codes + r * K);
  for (int b = lane; b < nblk; b += 32) {
    const uint2 q = __ldg(pr + b);
    const float s = e4m3_to_f32(__ldg(sr + b));
    float lo[8], hi[8];
    e2m1x8_to_f32(q.x, lo);
    e2m1x8_to_f32(q.y, hi);
    float v[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {   // e2m1 x e4m3 is exact in fp32
      v[i] = lo[i] * s;
      v[8 + i] = hi[i] * s;
    }
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = e4m3x2(v[4 * i], v[4 * i + 1], inv) | (e4m3x2(v[4 * i + 2], v[4 * i + 3], inv) << 16);
    dst[b] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// One warp per output row of bf16 activations (K % 256 == 0).  With sorted_slot set, output row
// p < S is token sorted_slot[p] / k of the source (the routed rows in expert order) and row
// S + t is token t (the shared expert's rows); without it row p is source row p.
__global__ void __launch_bounds__(256) act_quant_fp8_kernel(const uint16_t* __restrict__ src,
                                                            const int32_t* __restrict__ sorted_slot, int S, int k,
                                                            uint8_t* __restrict__ dst, float* __restrict__ scale,
                                                            int64_t rows, int K, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (r >= rows) return;
  int64_t srow = r;
  if (sorted_slot) {
    if (r < S) {
      int slot = __ldg(sorted_slot + r);
      if (static_cast<unsigned>(slot) >= static_cast<unsigned>(S)) {
        if (lane == 0) report_device_error(status, kDevBadIndex);
        slot = 0;
      }
      srow = slot / k;
    } else {
      srow = r - S;
    }
  }
  const uint4* s = reinterpret_cast<const uint4*>(src + srow * K);
  float m = 0.0f;
  for (int c = lane; c < K / 8; c += 32) {
    const uint4 v = __ldg(s + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fabsf(bf16_bits_to_f32(w[i] & 0xffffu)), fabsf(bf16_bits_to_f32(w[i] >> 16))));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float inv, sc;
  row_rule(m, inv, sc);
  if (lane == 0) scale[r] = sc;
  uint2* d = reinterpret_cast<uint2*>(dst + r * K);
  for (int c = lane; c < K / 8; c += 32) {
    const uint4 v = __ldg(s + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[2];
#pragma unroll
    for (int i = 0; i < 2; ++i)
      o[i] = e4m3x2(bf16_bits_to_f32(w[2 * i] & 0xffffu), bf16_bits_to_f32(w[2 * i] >> 16), inv) |
             (e4m3x2(bf16_bits_to_f32(w[2 * i + 1] & 0xffffu), bf16_bits_to_f32(w[2 * i + 1] >> 16), inv) << 16);
    d[c] = make_uint2(o[0], o[1]);
  }
}

// Token-major version of the gathered quantization (see act_scatter_f16_kernel): one warp per
// token reads its row once and writes the codes and the scale to every expert-ordered row of the
// token (its k ranks' rows slot_pos[t k + j] and the shared expert's row S + t).
__global__ void __launch_bounds__(256) act_scatter_fp8_kernel(const uint16_t* __restrict__ src,
                                                              const int32_t* __restrict__ slot_pos, int T, int k,
                                                              uint8_t* __restrict__ dst, float* __restrict__ scale,
                                                              int K, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int t = static_cast<int>((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  if (t >= T) return;
  const int S = T * k;
  int p = -1;
  if (lane < k) {
    p = __ldg(slot_pos + static_cast<int64_t>(t) * k + lane);
    if (static_cast<unsigned>(p) >= static_cast<unsigned>(S)) {
      report_device_error(status, kDevBadIndex);
      p = -1;
    }
  } else if (lane == k) {
    p = S + t;
  }
  const uint4* s = reinterpret_cast<const uint4*>(src + static_cast<int64_t>(t) * K);
  float m = 0.0f;
  for (int c = lane; c < K / 8; c += 32) {
    const uint4 v = __ldg(s + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fabsf(bf16_bits_to_f32(w[i] & 0xffffu)), fabsf(bf16_bits_to_f32(w[i] >> 16))));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float inv, sc;
  row_rule(m, inv, sc);
  if (p >= 0) scale[p] = sc;
  for (int c = lane; c < K / 8; c += 32) {
    const uint4 v = __ldg(s + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[2];
#pragma unroll
    for (int i = 0; i < 2; ++i)
      o[i] = e4m3x2(bf16_bits_to_f32(w[2 * i] & 0xffffu), bf16_bits_to_f32(w[2 * i] >> 16), inv) |
             (e4m3x2(bf16_bits_to_f32(w[2 * i + 1] & 0xffffu), bf16_bits_to_f32(w[2 * i + 1] >> 16), inv) << 16);
    const uint2 ov = make_uint2(o[0], o[1]);
    for (int j = 0; j <= k; ++j) {
      const int pj = __shfl_sync(0xffffffffu, p, j);
      if (pj >= 0) reinterpret_cast<uint2*>(dst + static_cast<int64_t>(pj) * K)[c] = ov;
    }
  }
}

}  // namespace

cudaError_t launch_act_scatter_fp8(const uint16_t* x, const int32_t* slot_pos, int T, int k, int K, uint8_t* dst,
                                   float* scale, int32_t* status, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  act_scatter_fp8_kernel<<<static_cast<unsigned>((static_cast<int64_t>(T) + 7) / 8), 256, 0, st>>>(
      x, slot_pos, T, k, dst, scale, K, status);
  return cudaGetLastError();
}

cudaError_t launch_prepare_fp8(const uint8_t* packed, const uint8_t* scales, int64_t rows, int K, uint8_t* codes,
                               float* row_scale, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  prepare_fp8_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(packed, scales, rows, K, codes, row_scale);
  return cudaGetLastError();
}

cudaError_t launch_act_quant_fp8(const uint16_t* src, const int32_t* sorted_slot, int S, int k, int64_t rows, int K,
                                 uint8_t* dst, float* scale, int32_t* status, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  act_quant_fp8_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(src, sorted_slot, S, k, dst, scale,
                                                                              rows, K, status);
  return cudaGetLastError();
}

}  // namespace moe
