// Grouped NVFP4 x bf16 GEMMs on the CUDA cores: the decode arm's GEMVs and the general
// staged path.
//
// W4A16 as in the untransposed column of the "long-context cold prefill to SGLang parity"
// issue's kernel table: bf16 activations, e2m1 x e4m3 block weights dequantized exactly,
// fp32 accumulation, scale2 applied to the fp32 sum, SiLU(gate)*up rounded to bf16.  The
// decode shape (one launch per projection, routed top-k and the shared expert together,
// gate+up fused, silu+down fused) is the two-launch structure the "handover briefs" page
// asks of a vectorised NVFP4 decode GEMV; weights are read with coalesced 8-byte loads of
// the resident [N, K/2] layout and dequantized in registers.
#include "internal.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void load_bf16x16(const uint16_t* p, float (&x)[16]) {
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
  const uint4 b = __ldg(reinterpret_cast<const uint4*>(p) + 1);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// One 16-element NVFP4 block of one weight row against TB activation vectors:
// acc[t] += e4m3(scale) * sum_i e2m1(q_i) * x[t][i]   (the block sum is exact-order fp32).
template <int TB>
__device__ __forceinline__ void block_dot(uint2 q, uint32_t scale_byte, const float (&x)[TB][16],
                                          float (&acc)[TB]) {
  float v[16];
  float lo[8], hi[8];
  e2m1x8_to_f32(q.x, lo);
  e2m1x8_to_f32(q.y, hi);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[i] = lo[i];
    v[8 + i] = hi[i];
  }
  const float s = e4m3_to_f32(scale_byte);
#pragma unroll
  for (int t = 0; t < TB; ++t) {
    float d = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) d = fmaf(v[i], x[t][i], d);
    acc[t] = fmaf(d, s, acc[t]);
  }
}

template <int R, int TB>
__device__ __forceinline__ void warp_allreduce(float (&acc)[R][TB]) {
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int t = 0; t < TB; ++t)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[r][t] += __shfl_xor_sync(kFull, acc[r][t], off);
}

// Activation row of permuted row p: gate_up gathers x[sorted_slot[p] / k] (routed) or x[p - S]
// (shared); down reads h[p].
__device__ __forceinline__ int64_t act_row(const GroupedArgs& a, bool gate_up, int p) {
  if (!gate_up) return p;
  if (p >= a.S) return p - a.S;
  int slot = __ldg(a.sorted_slot + p);
  if (static_cast<unsigned>(slot) >= static_cast<unsigned>(a.S)) {  // caller-provided index
    report_device_error(a.status, kDevBadIndex);
    slot = 0;
  }
  return slot / a.k;
}

// R weight rows (wrow) x TB permuted rows starting at p0 (nt of them live) for one warp.
template <bool kGateUp, int TB>
__device__ __forceinline__ void rows_pass(const GroupedArgs& a, const uint8_t* P, const uint8_t* Sc,
                                          const int (&wrow)[8], int p0, int nt, int lane,
                                          float (&acc)[8][TB]) {
  const int nchunk = a.K / 16;
  const uint16_t* arow[TB];
#pragma unroll
  for (int t = 0; t < TB; ++t) arow[t] = a.act + act_row(a, kGateUp, p0 + min(t, nt - 1)) * a.K;
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int t = 0; t < TB; ++t) acc[r][t] = 0.0f;
#pragma unroll 2
  for (int c = lane; c < nchunk; c += 32) {
    float x[TB][16];
#pragma unroll
    for (int t = 0; t < TB; ++t) load_bf16x16(arow[t] + c * 16, x[t]);
    uint2 q[8];
    uint32_t sb[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      q[r] = __ldg(reinterpret_cast<const uint2*>(P + static_cast<int64_t>(wrow[r]) * (a.K / 2)) + c);
      sb[r] = __ldg(Sc + static_cast<int64_t>(wrow[r]) * nchunk + c);
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      float part[TB];
#pragma unroll
      for (int t = 0; t < TB; ++t) part[t] = acc[r][t];
      block_dot<TB>(q[r], sb[r], x, part);
#pragma unroll
      for (int t = 0; t < TB; ++t) acc[r][t] = part[t];
    }
  }
  warp_allreduce<8, TB>(acc);
}

template <bool kGateUp, int TB>
__device__ __forceinline__ void store_rows(const GroupedArgs& a, const float (&acc)[8][TB], float s2,
                                           int wbase, int p0, int nt, int lane) {
  if (kGateUp) {
    const int I = a.N / 2;
    // rows 0..3 of the warp are gate columns wbase..wbase+3, rows 4..7 the matching up rows
#pragma unroll
    for (int t = 0; t < TB; ++t)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (lane == i + 4 * t && t < nt) {
          const float g = acc[i][t] * s2, u = acc[4 + i][t] * s2;
          static_cast<uint16_t*>(a.out)[static_cast<int64_t>(p0 + t) * I + wbase + i] =
              f32_to_bf16_bits(silu_f32(g) * u);
        }
  } else {
#pragma unroll
    for (int t = 0; t < TB; ++t)
#pragma unroll
      for (int r = 0; r < 8; ++r)
        if (lane == r + 8 * (t & 3) && t < nt)
          static_cast<float*>(a.out)[static_cast<int64_t>(p0 + t) * a.N + wbase + r] = acc[r][t] * s2;
  }
}

// grid.x = work item (tile), grid.y = block of 16 gate/up column pairs (gate_up) or 32 output
// rows (down); 4 warps, each owning 8 weight rows.
template <bool kGateUp>
__global__ void __launch_bounds__(128) grouped_simt_kernel(GroupedArgs a) {
  const int tile = blockIdx.x;
  if (tile >= __ldg(a.meta)) return;
  const int4 td = __ldg(a.tiles + tile);
  const int g = td.x, row0 = td.y, nrows = td.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int wrow[8];
  int wbase;
  if (kGateUp) {
    const int I = a.N / 2;
    wbase = blockIdx.y * 16 + warp * 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      wrow[i] = wbase + i;
      wrow[4 + i] = I + wbase + i;
    }
  } else {
    wbase = blockIdx.y * 32 + warp * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) wrow[i] = wbase + i;
  }
  const uint8_t* P = a.packed + static_cast<int64_t>(g) * a.N * (a.K / 2);
  const uint8_t* Sc = a.scales + static_cast<int64_t>(g) * a.N * (a.K / 16);
  const float s2 = __ldg(a.scale2 + g);
  int r0 = 0;
  for (; r0 + 4 <= nrows; r0 += 4) {
    float acc[8][4];
    rows_pass<kGateUp, 4>(a, P, Sc, wrow, row0 + r0, 4, lane, acc);
    store_rows<kGateUp, 4>(a, acc, s2, wbase, row0 + r0, 4, lane);
  }
  for (; r0 < nrows; ++r0) {
    float acc[8][1];
    rows_pass<kGateUp, 1>(a, P, Sc, wrow, row0 + r0, 1, lane, acc);
    store_rows<kGateUp, 1>(a, acc, s2, wbase, row0 + r0, 1, lane);
  }
}

// Decode arm, second launch: down projection of every active group for 8 output rows, then the
// fixed-order fp32 combine of those rows for every token.  grid.x = H / 8, 8 warps.
constexpr int kDcRows = 8;

__global__ void __launch_bounds__(256) down_combine_gemv_kernel(DownCombineArgs a) {
  extern __shared__ float ybuf[];  // [(S + T) rows][kDcRows]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kDcRows;
  const int n_tiles = __ldg(a.meta);
  const int nchunk = a.I / 16;
  for (int u = warp; u < n_tiles; u += 8) {
    const int4 td = __ldg(a.tiles + u);
    const int g = td.x, row0 = td.y, nrows = td.z;
    const uint8_t* P = a.packed + (static_cast<int64_t>(g) * a.H + n0) * (a.I / 2);
    const uint8_t* Sc = a.scales + (static_cast<int64_t>(g) * a.H + n0) * nchunk;
    const float s2 = __ldg(a.scale2 + g);
    for (int r0 = 0; r0 < nrows; ++r0) {
      float acc[kDcRows][1];
#pragma unroll
      for (int r = 0; r < kDcRows; ++r) acc[r][0] = 0.0f;
      const uint16_t* hrow = a.h + static_cast<int64_t>(row0 + r0) * a.I;
      for (int c = lane; c < nchunk; c += 32) {
        float x[1][16];
        load_bf16x16(hrow + c * 16, x[0]);
        uint2 q[kDcRows];
        uint32_t sb[kDcRows];
#pragma unroll
        for (int r = 0; r < kDcRows; ++r) {
          q[r] = __ldg(reinterpret_cast<const uint2*>(P + static_cast<int64_t>(r) * (a.I / 2)) + c);
          sb[r] = __ldg(Sc + static_cast<int64_t>(r) * nchunk + c);
        }
#pragma unroll
        for (int r = 0; r < kDcRows; ++r) {
          float part[1] = {acc[r][0]};
          block_dot<1>(q[r], sb[r], x, part);
          acc[r][0] = part[0];
        }
      }
      warp_allreduce<kDcRows, 1>(acc);
#pragma unroll
      for (int r = 0; r < kDcRows; ++r)
        if (lane == r) ybuf[static_cast<int64_t>(row0 + r0) * kDcRows + r] = acc[r][0] * s2;
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < a.T * kDcRows; idx += blockDim.x) {
    const int t = idx / kDcRows, r = idx % kDcRows;
    float s = 0.0f;
    for (int j = 0; j < a.k; ++j) {
      int p = __ldg(a.slot_pos + t * a.k + j);
      if (static_cast<unsigned>(p) >= static_cast<unsigned>(a.S)) {
        report_device_error(a.status, kDevBadIndex);
        p = 0;
      }
      s = fmaf(__ldg(a.topk_w + t * a.k + j), ybuf[p * kDcRows + r], s);
    }
    if (a.has_shared) s += ybuf[(a.S + t) * kDcRows + r];
    const int64_t o = static_cast<int64_t>(t) * a.H + n0 + r;
    if (a.out_is_fp32)
      static_cast<float*>(a.out)[o] = s;
    else
      static_cast<uint16_t*>(a.out)[o] = f32_to_bf16_bits(s);
  }
}

}  // namespace

cudaError_t launch_gate_up_simt(const GroupedArgs& a, cudaStream_t st) {
  dim3 grid(static_cast<unsigned>(a.max_tiles), static_cast<unsigned>(a.N / 2 / 16));
  grouped_simt_kernel<true><<<grid, 128, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_down_simt(const GroupedArgs& a, cudaStream_t st) {
  dim3 grid(static_cast<unsigned>(a.max_tiles), static_cast<unsigned>(a.N / 32));
  grouped_simt_kernel<false><<<grid, 128, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_down_combine_gemv(const DownCombineArgs& a, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(a.S + a.T) * kDcRows * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(down_combine_gemv_kernel),
                                        static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  down_combine_gemv_kernel<<<a.H / kDcRows, 256, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
