// fp32 weighted unpermute/combine of the staged path (fp32 expert outputs y):
// out[t] = sum_j w[t, j] * y[slot_pos[t*k+j]]
// + y[S + t], accumulated in fp32 in rank order then the shared expert (the "fp32 weighted sum"
// of the "long-context cold prefill to SGLang parity" issue's kernel table; the fixed order is
// the one-rank reduction order the TensorFold sm_120 issue requires of expert parallelism).
#include <algorithm>

#include "internal.cuh"

namespace moe {
namespace {

__device__ __forceinline__ void load8(const float* p, float (&f)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// One thread per (token, 8 consecutive hidden columns).
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y,
                                                      const int32_t* __restrict__ slot_pos,
                                                      const float* __restrict__ topk_w, int T,
                                                      int H, int k, int has_shared, void* out,
                                                      int out_is_fp32, int32_t* status) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int cpr = H / 8;
  if (idx >= static_cast<int64_t>(T) * cpr) return;
  const int t = static_cast<int>(idx / cpr);
  const int c = static_cast<int>(idx % cpr) * 8;
  const int64_t S = static_cast<int64_t>(T) * k;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  // ranks in groups of four: the group's row loads are issued together, then summed in rank order
  for (int j0 = 0; j0 < k; j0 += 4) {
    float v[4][8], wj[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (j0 + q < k) {
        int64_t p = __ldg(slot_pos + static_cast<int64_t>(t) * k + j0 + q);
        if (p < 0 || p >= S) {  // caller-provided index
          if (status) report_device_error(status, kDevBadIndex);
          p = 0;
        }
        wj[q] = __ldg(topk_w + static_cast<int64_t>(t) * k + j0 + q);
        load8(y + p * H + c, v[q]);
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (j0 + q < k)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj[q], v[q][i], acc[i]);
  }
  if (has_shared) {
    float v[8];
    load8(y + (S + t) * H + c, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += v[i];
  }
  const int64_t o = static_cast<int64_t>(t) * H + c;
  if (out_is_fp32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + o);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  } else {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = static_cast<uint32_t>(f32_to_bf16_bits(acc[2 * i])) |
             (static_cast<uint32_t>(f32_to_bf16_bits(acc[2 * i + 1])) << 16);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + o) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// The same sum over the compact y of the tensor-core down: row p's values are f16 * rowf[p],
// rowf written by the down epilogue (the factor the fp32 path applies to the accumulator, times
// the power of two the compact form removed).  A unit is (token, 8 consecutive columns); the grid
// is resident (a few CTAs per SM) and thread i takes units i, i + n, i + 2n, ... (n threads in the
// grid).  For each unit every rank's row (raw f16 words and its row factor) and the shared
// expert's are loaded before any is used, then the unit's weights and the next unit's slot
// positions while those rows are in flight, so a unit costs about one memory round trip; the sum
// runs in rank order, then the shared expert.  KC >= k bounds the per-rank register arrays; up to
// 10 ranks two CTAs stay resident per SM, above that one.
template <int KC>
constexpr int combine_ctas_per_sm() { return KC <= 10 ? 2 : 1; }

template <int KC>
__global__ void __launch_bounds__(256, combine_ctas_per_sm<KC>()) combine_y16_kernel(const uint16_t* __restrict__ y16,
                                                             const float* __restrict__ rowf,
                                                             const int32_t* __restrict__ slot_pos,
                                                             const float* __restrict__ topk_w, int T, int H, int k,
                                                             int has_shared, void* out, int out_is_fp32,
                                                             int32_t* status) {
  pdl_wait();
  const int cpr = H / 8;
  const int64_t units = static_cast<int64_t>(T) * cpr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (u >= units) return;
  const int64_t S = static_cast<int64_t>(T) * k;
  int p[KC];
  auto load_slots = [&](int64_t unit) {
    const int64_t s0 = (unit / cpr) * k;
#pragma unroll
    for (int q = 0; q < KC; ++q)
      if (q < k) p[q] = __ldg(slot_pos + s0 + q);
  };
  load_slots(u);
  for (;;) {
    const int t = static_cast<int>(u / cpr);
    const int c = static_cast<int>(u % cpr) * 8;
    // out-of-range positions read row 0 and are reported once, after every load is issued (no
    // branch between the loads)
    bool bad = false;
#pragma unroll
    for (int q = 0; q < KC; ++q) {
      if (q < k) {
        const bool out = p[q] < 0 || p[q] >= S;
        bad |= out;
        p[q] = out ? 0 : p[q];
      }
    }
    uint4 hv[KC];
    float fr[KC];
#pragma unroll
    for (int q = 0; q < KC; ++q) {
      if (q < k) {
        hv[q] = __ldg(reinterpret_cast<const uint4*>(y16 + static_cast<int64_t>(p[q]) * H + c));
        fr[q] = __ldg(rowf + p[q]);
      }
    }
    uint4 hs = make_uint4(0u, 0u, 0u, 0u);
    float frs = 0.0f;
    if (has_shared) {
      hs = __ldg(reinterpret_cast<const uint4*>(y16 + (S + t) * H + c));
      frs = __ldg(rowf + S + t);
    }
    if (bad && status) report_device_error(status, kDevBadIndex);
    float wj[KC];
#pragma unroll
    for (int q = 0; q < KC; ++q)
      if (q < k) wj[q] = __ldg(topk_w + static_cast<int64_t>(t) * k + q);
    // the next unit's slot positions (this unit's rows are already addressed)
    const int64_t un = u + stride;
    if (un < units) load_slots(un);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int q = 0; q < KC; ++q) {
      if (q < k) {
        const uint32_t w[4] = {hv[q].x, hv[q].y, hv[q].z, hv[q].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = fmaf(wj[q], __half2float(__ushort_as_half(static_cast<uint16_t>(w[i] & 0xffffu))) * fr[q], acc[2 * i]);
          acc[2 * i + 1] = fmaf(wj[q], __half2float(__ushort_as_half(static_cast<uint16_t>(w[i] >> 16))) * fr[q], acc[2 * i + 1]);
        }
      }
    }
    if (has_shared) {
      const uint32_t w[4] = {hs.x, hs.y, hs.z, hs.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] += __half2float(__ushort_as_half(static_cast<uint16_t>(w[i] & 0xffffu))) * frs;
        acc[2 * i + 1] += __half2float(__ushort_as_half(static_cast<uint16_t>(w[i] >> 16))) * frs;
      }
    }
    const int64_t o = static_cast<int64_t>(t) * H + c;
    if (out_is_fp32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + o);
      dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        w[i] = static_cast<uint32_t>(f32_to_bf16_bits(acc[2 * i])) |
               (static_cast<uint32_t>(f32_to_bf16_bits(acc[2 * i + 1])) << 16);
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + o) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (un >= units) break;
    u = un;
  }
}

}  // namespace

cudaError_t launch_combine_y16(const uint16_t* y16, const float* rowf, const int32_t* slot_pos, const float* topk_w,
                               int T, int H, int k, int has_shared, void* out, int out_is_fp32, int32_t* status,
                               bool pdl, cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(T) * (H / 8);
  if (n == 0) return cudaSuccess;
  int n_sm = 0;
  const cudaError_t e = current_sm_count(&n_sm);
  if (e != cudaSuccess) return e;
  if (k < 1 || k > kMaxK) return cudaErrorInvalidValue;
  // the resident CTAs of the kernel's launch bounds on every SM, fewer when there are fewer units
  const bool lean = k <= 10;
  const int64_t resident = static_cast<int64_t>(n_sm) * (lean ? combine_ctas_per_sm<10>() : combine_ctas_per_sm<kMaxK>());
  const unsigned blocks = static_cast<unsigned>(std::min<int64_t>((n + 255) / 256, resident));
  return launch_pdl(pdl, lean ? combine_y16_kernel<10> : combine_y16_kernel<kMaxK>, dim3(blocks), dim3(256), 0, st, y16,
                    rowf, slot_pos, topk_w, T, H, k, has_shared, out, out_is_fp32, status);
}

cudaError_t launch_combine(const float* y, const int32_t* slot_pos, const float* topk_w, int T,
                           int H, int k, int has_shared, void* out, int out_is_fp32,
                           int32_t* status, cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(T) * (H / 8);
  const unsigned blocks = static_cast<unsigned>((n + 255) / 256);
  combine_kernel<<<blocks, 256, 0, st>>>(y, slot_pos, topk_w, T, H, k, has_shared, out,
                                         out_is_fp32, status);
  return cudaGetLastError();
}

}  // namespace moe
