// bf16 activation rows -> f16 rows with a per-row power-of-two scale, for the f16 tensor-core
// GEMMs of the prefill arm.
//
// Row r is written as f16(x[r] * 2^-e[r]) with e[r] = floor(log2(max |x[r]|)) - 14, at least
// -126 (and the factor 2^e[r] as a float for the GEMM epilogue), so the row's largest element
// lands in [2^14, 2^15), well inside f16's range.  A bf16 value has 8 significant
// bits and f16 11, so every element of at least 2^-31 of the row maximum converts exactly; only
// smaller ones (below f16's subnormal grid) are rounded.  The GEMM epilogue multiplies the fp32
// accumulator by 2^e[r] again, so the products are the bf16 activations' own.
#include "internal.cuh"

namespace moe {
namespace {

// One warp per output row; K % 256 == 0 (eight bf16 per lane per step).  With sorted_slot set,
// output row p < S is the token sorted_slot[p] / k of the source (the routed rows in expert
// order) and row S + t is token t (the shared expert's rows); without it row p is source row p.
__global__ void __launch_bounds__(256) act_to_f16_kernel(const uint16_t* __restrict__ src,
                                                         const int32_t* __restrict__ sorted_slot,
                                                         int S, int k, uint16_t* __restrict__ dst,
                                                         float* __restrict__ factor, int64_t rows,
                                                         int K, int32_t* status) {
  pdl_wait();
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
  // rows of K <= 2048 stay in registers between their maximum and their conversion (one read)
  constexpr int kHeld = 8;   // 16-byte pieces per lane held in registers
  const bool held = K % 256 == 0 && K <= 256 * kHeld;
  uint4 hv[kHeld];
  float m = 0.0f;
  if (held) {
#pragma unroll
    for (int i = 0; i < kHeld; ++i) {
      if (i < K / 256) {
        hv[i] = __ldg(s + i * 32 + lane);
        const uint32_t w[4] = {hv[i].x, hv[i].y, hv[i].z, hv[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          m = fmaxf(m, fabsf(__uint_as_float(w[j] << 16)));
          m = fmaxf(m, fabsf(__uint_as_float(w[j] & 0xffff0000u)));
        }
      }
    }
  } else {
    for (int c = lane; c < K / 8; c += 32) {
      const uint4 v = __ldg(s + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        m = fmaxf(m, fabsf(__uint_as_float(w[i] << 16)));
        m = fmaxf(m, fabsf(__uint_as_float(w[i] & 0xffff0000u)));
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  // e >= -126 keeps 2^-e a normal float (a row whose maximum is below 2^-112 is scaled less)
  const int e = (m > 0.0f && m <= 3.4e38f) ? max(ilogbf(m) - 14, -126) : 0;
  const float inv = __int_as_float((127 - e) << 23);           // 2^-e, exactly
  if (lane == 0) factor[r] = __int_as_float((127 + e) << 23);  // the epilogue's 2^e
  uint4* d = reinterpret_cast<uint4*>(dst + r * K);
  if (held) {
#pragma unroll
    for (int i = 0; i < kHeld; ++i) {
      if (i < K / 256) {
        const uint32_t w[4] = {hv[i].x, hv[i].y, hv[i].z, hv[i].w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const __half2 h = __floats2half2_rn(__uint_as_float(w[j] << 16) * inv, __uint_as_float(w[j] & 0xffff0000u) * inv);
          o[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
        d[i * 32 + lane] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    return;
  }
  for (int c = lane; c < K / 8; c += 32) {
    const uint4 v = __ldg(s + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float lo = __uint_as_float(w[i] << 16) * inv;
      const float hi = __uint_as_float(w[i] & 0xffff0000u) * inv;
      const __half2 h = __floats2half2_rn(lo, hi);
      o[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    d[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Token-major version of the expert-order gather: a warp reads its token's row and writes the
// f16 row to every expert-ordered row that holds the token (slot_pos[t k + j] for its k ranks,
// and S + t for the shared expert).  Each token row is read from memory once instead of k + 1
// times (a 32k-token batch of x is larger than L2).  For small batches `slices` warps share a
// token, each taking the row maximum over the whole row and then converting and writing its
// 1 / slices of the columns (K / 256 divisible by slices).
__global__ void __launch_bounds__(256) act_scatter_f16_kernel(const uint16_t* __restrict__ src,
                                                              const int32_t* __restrict__ slot_pos, int T, int k,
                                                              uint16_t* __restrict__ dst, float* __restrict__ factor,
                                                              int K, int slices, int32_t* status) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int t = static_cast<int>(gw / slices), sl = static_cast<int>(gw % slices);
  if (t >= T) return;
  const int S = T * k;
  // destination rows: lane j < k holds rank j's row, lane k the shared expert's row S + t
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
  // a whole row handled by one warp with K <= 2048 stays in registers between its maximum and its
  // conversion (one read of the row); otherwise the slice is read again after the maximum
  constexpr int kHeld = 8;   // 16-byte pieces per lane held in registers
  const bool held = slices == 1 && K % 256 == 0 && K <= 256 * kHeld;
  uint4 hv[kHeld];
  float m = 0.0f;
  if (held) {
#pragma unroll
    for (int i = 0; i < kHeld; ++i) {
      if (i < K / 256) {
        hv[i] = __ldg(s + i * 32 + lane);
        const uint32_t w[4] = {hv[i].x, hv[i].y, hv[i].z, hv[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          m = fmaxf(m, fabsf(__uint_as_float(w[j] << 16)));
          m = fmaxf(m, fabsf(__uint_as_float(w[j] & 0xffff0000u)));
        }
      }
    }
  } else {
    for (int c = lane; c < K / 8; c += 32) {
      const uint4 v = __ldg(s + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        m = fmaxf(m, fabsf(__uint_as_float(w[i] << 16)));
        m = fmaxf(m, fabsf(__uint_as_float(w[i] & 0xffff0000u)));
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  const int e = (m > 0.0f && m <= 3.4e38f) ? max(ilogbf(m) - 14, -126) : 0;
  const float inv = __int_as_float((127 - e) << 23);
  if (p >= 0 && sl == 0) factor[p] = __int_as_float((127 + e) << 23);
  if (held) {
#pragma unroll
    for (int i = 0; i < kHeld; ++i) {
      if (i < K / 256) {
        const uint32_t w[4] = {hv[i].x, hv[i].y, hv[i].z, hv[i].w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const __half2 h = __floats2half2_rn(__uint_as_float(w[j] << 16) * inv, __uint_as_float(w[j] & 0xffff0000u) * inv);
          o[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
        const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
        for (int jj = 0; jj <= k; ++jj) {
          const int pj = __shfl_sync(0xffffffffu, p, jj);
          if (pj >= 0) reinterpret_cast<uint4*>(dst + static_cast<int64_t>(pj) * K)[i * 32 + lane] = ov;
        }
      }
    }
    return;
  }
  const int per = K / 8 / slices;   // uint4 columns of this warp's slice
  for (int c = sl * per + lane; c < (sl + 1) * per; c += 32) {
    const uint4 v = __ldg(s + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 h = __floats2half2_rn(__uint_as_float(w[i] << 16) * inv, __uint_as_float(w[i] & 0xffff0000u) * inv);
      o[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
    for (int j = 0; j <= k; ++j) {
      const int pj = __shfl_sync(0xffffffffu, p, j);
      if (pj >= 0) reinterpret_cast<uint4*>(dst + static_cast<int64_t>(pj) * K)[c] = ov;
    }
  }
}

}  // namespace

cudaError_t launch_act_scatter_f16(const uint16_t* x, const int32_t* slot_pos, int T, int k, int K, uint16_t* dst,
                                   float* factor, int32_t* status, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  // slices per token: enough warps for about 16 per SM on a 152-SM GPU, at most K / 256
  int slices = 1;
  while (slices * 2 <= K / 256 && static_cast<int64_t>(T) * slices < 152 * 16) slices *= 2;
  while ((K / 256) % slices) slices /= 2;
  const int64_t warps = static_cast<int64_t>(T) * slices;
  return launch_pdl(false, act_scatter_f16_kernel, dim3(static_cast<unsigned>((warps + 7) / 8)), dim3(256), 0, st, x, slot_pos,
                    T, k, dst, factor, K, slices, status);
}

cudaError_t launch_act_to_f16(const uint16_t* src, uint16_t* dst, float* factor, int64_t rows, int K, bool pdl,
                              cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const int64_t blocks = (rows + 7) / 8;
  return launch_pdl(pdl, act_to_f16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, src,
                    static_cast<const int32_t*>(nullptr), 0, 1, dst, factor, rows, K, static_cast<int32_t*>(nullptr));
}

cudaError_t launch_act_gather_f16(const uint16_t* x, const int32_t* sorted_slot, int T, int k, int K,
                                  uint16_t* dst, float* factor, int32_t* status, cudaStream_t st) {
  const int S = T * k;
  const int64_t rows = static_cast<int64_t>(S) + T;
  if (rows <= 0) return cudaSuccess;
  const int64_t blocks = (rows + 7) / 8;
  act_to_f16_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(x, sorted_slot, S, k, dst, factor, rows, K,
                                                                     status);
  return cudaGetLastError();
}

}  // namespace moe
