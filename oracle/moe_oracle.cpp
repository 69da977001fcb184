// CPU oracle of the NVFP4 routed-MoE layer -- TEST INFRASTRUCTURE ONLY (see moe_oracle.h).
//
// Plain, slow, obviously-correct restatement of what the layer computes.  Built with
// -O2 -ffp-contract=off and no fast-math so that every float/double operation is the single
// IEEE operation written here.
#include "moe_oracle.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------------------------------
// Element formats.  NVFP4 = e2m1 values x one e4m3 scale per 16-element block x one fp32
// per-tensor scale2 ("long-context cold prefill" issue, kernel comparison table, "weights"
// row).  e2m1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit, no inf/NaN.  e4m3: 1 sign,
// 4 exponent bits (bias 7), 3 mantissa bits, no inf, S.1111.111 is NaN; largest finite 448
// and smallest normal 2^-6 (the same table row: "saturation at +-448", "subnormals below
// 2^-6").
// ---------------------------------------------------------------------------------------
double e2m1_value(unsigned c) {
  const unsigned s = (c >> 3) & 1u, e = (c >> 1) & 3u, m = c & 1u;
  const double mag = (e == 0) ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, static_cast<int>(e) - 1);
  return s ? -mag : mag;
}

double e4m3_value(unsigned c) {
  const unsigned s = (c >> 7) & 1u, e = (c >> 3) & 15u, m = c & 7u;
  if (e == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
  const double mag = (e == 0) ? std::ldexp(m / 8.0, -6)
                              : std::ldexp(1.0 + m / 8.0, static_cast<int>(e) - 7);
  return s ? -mag : mag;
}

// Round a non-negative finite value to the nearest entry of an increasing table of the
// format's non-negative values (index == code), ties to the even code, saturating at the
// last entry.  All differences are exact in double (values are short dyadic numbers and
// v is an fp32 value).
int round_to_table(double v, const double* table, int n) {
  if (!(v > 0.0)) return 0;
  if (v >= table[n - 1]) return n - 1;
  int lo = 0;
  while (lo + 1 < n && table[lo + 1] <= v) ++lo;  // largest entry <= v
  const int hi = lo + 1;
  const double dlo = v - table[lo], dhi = table[hi] - v;
  if (dlo < dhi) return lo;
  if (dhi < dlo) return hi;
  return (lo % 2 == 0) ? lo : hi;
}

struct Tables {
  double e2m1_pos[8];
  double e4m3_pos[127];  // codes 0x00..0x7E
  double e2m1_all[16];   // every code's value, for the dequantizer
  double e4m3_all[256];
  Tables() {
    for (int c = 0; c < 8; ++c) e2m1_pos[c] = e2m1_value(c);
    for (int c = 0; c < 127; ++c) e4m3_pos[c] = e4m3_value(c);
    for (int c = 0; c < 16; ++c) e2m1_all[c] = e2m1_value(c);
    for (int c = 0; c < 256; ++c) e4m3_all[c] = e4m3_value(c);
  }
};
const Tables& tables() {
  static const Tables t;
  return t;
}

int e2m1_encode(float v) {
  const int sign = std::signbit(v) ? 8 : 0;
  return sign | round_to_table(std::fabs(static_cast<double>(v)), tables().e2m1_pos, 8);
}

int e4m3_encode(float v) {
  const int sign = std::signbit(v) ? 0x80 : 0;
  return sign | round_to_table(std::fabs(static_cast<double>(v)), tables().e4m3_pos, 127);
}

double bf16_value(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

// Logit as used for selection: NaN never wins, so it counts as -inf.
double sel_key(float l) {
  return std::isnan(l) ? -std::numeric_limits<double>::infinity() : static_cast<double>(l);
}

double silu(double g) { return g / (1.0 + std::exp(-g)); }

unsigned thread_count(int n_threads) {
  if (n_threads > 0) return static_cast<unsigned>(n_threads);
  const unsigned hc = std::thread::hardware_concurrency();
  return hc ? hc : 1u;
}

template <class F>
void parallel_for(int64_t n, unsigned nt, F&& f) {
  std::atomic<int64_t> next{0};
  auto worker = [&]() {
    for (int64_t i = next.fetch_add(1); i < n; i = next.fetch_add(1)) f(i);
  };
  if (nt <= 1 || n <= 1) {
    worker();
    return;
  }
  std::vector<std::thread> pool;
  for (unsigned t = 0; t < nt; ++t) pool.emplace_back(worker);
  for (auto& th : pool) th.join();
}

// Exact dequantization of one [N, K] matrix of one group into fp64:
// w[n, k] = e2m1(q[n, k]) * e4m3(s[n, k/16]) * scale2.  The code values are read from tables
// filled by e2m1_value / e4m3_value above (the same values, looked up instead of recomputed).
void dequant_matrix(const uint8_t* packed, const uint8_t* scales, float scale2, int64_t N,
                    int64_t K, double* out) {
  const Tables& tb = tables();
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t kk = 0; kk < K; ++kk) {
      const uint8_t byte = packed[n * (K / 2) + kk / 2];
      const unsigned code = (kk % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
      const double s = tb.e4m3_all[scales[n * (K / 16) + kk / 16]];
      out[n * K + kk] = tb.e2m1_all[code] * s * static_cast<double>(scale2);
    }
  }
}

}  // namespace

extern "C" {

double orc_e2m1_value(int code) { return e2m1_value(static_cast<unsigned>(code) & 0xFu); }
double orc_e4m3_value(int code) { return e4m3_value(static_cast<unsigned>(code) & 0xFFu); }
int orc_e2m1_encode(float v) { return e2m1_encode(v); }
int orc_e4m3_encode(float v) { return e4m3_encode(v); }

// NVFP4 quantizer of the benchmark configurations: per-tensor scale2 = amax / (448*6);
// per-16-block e4m3 scale = block amax / 6 / scale2, rounded to nearest even and saturated;
// element code = e2m1 round-to-nearest-even of w / (e4m3(scale) * scale2).  Each step is one
// fp32 operation in the order written.  A block whose decoded scale is 0 stores code +0.
int orc_quantize(const float* w, int64_t G, int64_t N, int64_t K, uint8_t* packed,
                 uint8_t* scales, float* scale2) {
  if (!w || !packed || !scales || !scale2 || G < 0 || N < 0 || K <= 0 || K % 16) return -1;
  for (int64_t g = 0; g < G; ++g) {
    const float* wg = w + g * N * K;
    float amax = 0.0f;
    for (int64_t i = 0; i < N * K; ++i) amax = std::max(amax, std::fabs(wg[i]));
    const float s2 = amax / 2688.0f;
    scale2[g] = s2;
    for (int64_t n = 0; n < N; ++n) {
      for (int64_t b = 0; b < K / 16; ++b) {
        const float* blk = wg + n * K + b * 16;
        float bamax = 0.0f;
        for (int i = 0; i < 16; ++i) bamax = std::max(bamax, std::fabs(blk[i]));
        int sc = 0;
        if (s2 > 0.0f) {
          const float ratio = (bamax / 6.0f) / s2;
          sc = e4m3_encode(ratio);
        }
        scales[(g * N + n) * (K / 16) + b] = static_cast<uint8_t>(sc);
        const float d = static_cast<float>(e4m3_value(sc)) * s2;
        for (int i = 0; i < 16; i += 2) {
          int c0 = 0, c1 = 0;
          if (d != 0.0f) {
            c0 = e2m1_encode(blk[i] / d);
            c1 = e2m1_encode(blk[i + 1] / d);
          }
          packed[(g * N + n) * (K / 2) + b * 8 + i / 2] = static_cast<uint8_t>(c0 | (c1 << 4));
        }
      }
    }
  }
  return 0;
}

int orc_dequantize(const uint8_t* packed, const uint8_t* scales, const float* scale2, int64_t G,
                   int64_t N, int64_t K, double* out) {
  if (!packed || !scales || !scale2 || !out || K <= 0 || K % 16) return -1;
  for (int64_t g = 0; g < G; ++g)
    dequant_matrix(packed + g * N * (K / 2), scales + g * N * (K / 16), scale2[g], N, K,
                   out + g * N * K);
  return 0;
}

// Router GEMM: logit[t, e] = sum_h x[t, h] * w[e, h] in fp64, w dequantized exactly (one group of E
// rows), each row's products summed in h order.
int orc_router_logits(const uint16_t* x, const uint8_t* packed, const uint8_t* scales, const float* scale2,
                      int T, int H, int E, double* logits) {
  if (!x || !packed || !scales || !scale2 || !logits || T < 0 || H <= 0 || H % 16 || E <= 0) return -1;
  std::vector<double> w(static_cast<size_t>(E) * H);
  dequant_matrix(packed, scales, scale2[0], E, H, w.data());
  std::vector<double> xv(H);
  for (int t = 0; t < T; ++t) {
    for (int c = 0; c < H; ++c) xv[c] = bf16_value(x[static_cast<int64_t>(t) * H + c]);
    for (int e = 0; e < E; ++e) {
      double s = 0.0;
      const double* we = &w[static_cast<size_t>(e) * H];
      for (int c = 0; c < H; ++c) s += we[c] * xv[c];
      logits[static_cast<int64_t>(t) * E + e] = s;
    }
  }
  return 0;
}

// Routing: softmax over all E logits, top-k by (logit descending, index ascending) with NaN
// counted as -inf, then the k probabilities renormalised to sum to 1.  Selection is made on
// the logits themselves (softmax is monotone).  Where the softmax has no value (every logit
// -inf or NaN) the weights are 0; +inf logits share the mass equally (the limit).
int orc_route(const float* logits, int T, int E, int k, int32_t* ids, double* w) {
  if (!logits || !ids || !w || T < 0 || E <= 0 || k <= 0 || k > E) return -1;
  std::vector<int> order(E);
  std::vector<double> p(E);
  const double inf = std::numeric_limits<double>::infinity();
  for (int t = 0; t < T; ++t) {
    const float* l = logits + static_cast<int64_t>(t) * E;
    for (int e = 0; e < E; ++e) order[e] = e;
    std::stable_sort(order.begin(), order.end(),
                     [&](int a, int b) { return sel_key(l[a]) > sel_key(l[b]); });
    double m = -inf;
    for (int e = 0; e < E; ++e) m = std::max(m, sel_key(l[e]));
    if (m == -inf) {
      std::fill(p.begin(), p.end(), 0.0);
    } else if (m == inf) {
      double n_inf = 0;
      for (int e = 0; e < E; ++e) n_inf += (sel_key(l[e]) == inf) ? 1.0 : 0.0;
      for (int e = 0; e < E; ++e) p[e] = (sel_key(l[e]) == inf) ? 1.0 / n_inf : 0.0;
    } else {
      double z = 0.0;
      for (int e = 0; e < E; ++e) z += std::exp(sel_key(l[e]) - m);
      for (int e = 0; e < E; ++e) p[e] = std::exp(sel_key(l[e]) - m) / z;
    }
    double zk = 0.0;
    for (int j = 0; j < k; ++j) zk += p[order[j]];
    for (int j = 0; j < k; ++j) {
      ids[static_cast<int64_t>(t) * k + j] = order[j];
      w[static_cast<int64_t>(t) * k + j] = (zk > 0.0) ? p[order[j]] / zk : 0.0;
    }
  }
  return 0;
}

// Permutation: counts per expert, exclusive prefix offsets (E+1 entries), slots stably
// sorted by expert (ascending slot id inside an expert) and the inverse map.
int orc_permute(const int32_t* ids, int T, int E, int k, int32_t* counts, int32_t* offsets,
                int32_t* sorted_slot, int32_t* slot_pos) {
  if (!ids || !counts || !offsets || !sorted_slot || !slot_pos || T < 0 || E <= 0 || k <= 0)
    return -1;
  const int64_t S = static_cast<int64_t>(T) * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t s = 0; s < S; ++s) {
    if (ids[s] < 0 || ids[s] >= E) return -1;
    counts[ids[s]]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  std::vector<int32_t> fill(offsets, offsets + E);
  for (int64_t s = 0; s < S; ++s) {
    const int32_t p = fill[ids[s]]++;
    sorted_slot[p] = static_cast<int32_t>(s);
    slot_pos[s] = p;
  }
  return 0;
}

int orc_moe_forward(const uint16_t* x, const float* logits, const uint8_t* gu_packed,
                    const uint8_t* gu_scales, const float* gu_scale2, const uint8_t* dn_packed,
                    const uint8_t* dn_scales, const float* dn_scale2, int T, int H, int I, int E,
                    int k, int has_shared, const int32_t* tokens, int n_tok, double* out,
                    double* h, double* y, int n_threads) {
  if (!x || !logits || !gu_packed || !gu_scales || !gu_scale2 || !dn_packed || !dn_scales ||
      !dn_scale2 || !out || T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || k > E ||
      H % 16 || I % 16)
    return -1;
  std::vector<int32_t> tok;
  if (tokens) {
    tok.assign(tokens, tokens + n_tok);
    for (int32_t t : tok)
      if (t < 0 || t >= T) return -1;
  } else {
    tok.resize(T);
    for (int t = 0; t < T; ++t) tok[t] = t;
  }
  const int64_t n = static_cast<int64_t>(tok.size());
  const int J = k + (has_shared ? 1 : 0);

  std::vector<int32_t> ids(static_cast<size_t>(T) * k);
  std::vector<double> rw(static_cast<size_t>(T) * k);
  if (orc_route(logits, T, E, k, ids.data(), rw.data())) return -1;

  // Work list per group: (evaluated-token index i, rank j).
  const int G = E + (has_shared ? 1 : 0);
  std::vector<std::vector<std::pair<int64_t, int>>> work(G);
  for (int64_t i = 0; i < n; ++i) {
    for (int j = 0; j < k; ++j) work[ids[static_cast<size_t>(tok[i]) * k + j]].push_back({i, j});
    if (has_shared) work[E].push_back({i, k});
  }

  std::vector<double> ybuf(static_cast<size_t>(n) * J * H, 0.0);
  std::vector<double> hbuf(h ? static_cast<size_t>(n) * J * I : 0, 0.0);
  const int64_t gu_N = 2LL * I, gu_K = H, dn_N = H, dn_K = I;

  // Tasks: consecutive runs of at most kChunk work items of one group, so that a group with
  // many tokens (the shared expert, a popular expert) is spread over the threads.  Every item
  // is still computed on its own, exactly as below; only the split of the loop changes.
  constexpr size_t kChunk = 64;
  std::vector<std::pair<int, size_t>> tasks;   // (group, first item)
  for (int g = 0; g < G; ++g)
    for (size_t b = 0; b < work[g].size(); b += kChunk) tasks.push_back({g, b});

  parallel_for(static_cast<int64_t>(tasks.size()), thread_count(n_threads), [&](int64_t ti) {
    const int64_t g = tasks[ti].first;
    const size_t b0 = tasks[ti].second, b1 = std::min(work[g].size(), b0 + kChunk);
    std::vector<double> wgu(static_cast<size_t>(gu_N * gu_K)), wdn(static_cast<size_t>(dn_N * dn_K));
    dequant_matrix(gu_packed + g * gu_N * (gu_K / 2), gu_scales + g * gu_N * (gu_K / 16),
                   gu_scale2[g], gu_N, gu_K, wgu.data());
    dequant_matrix(dn_packed + g * dn_N * (dn_K / 2), dn_scales + g * dn_N * (dn_K / 16),
                   dn_scale2[g], dn_N, dn_K, wdn.data());
    std::vector<double> xv(H), a(I);
    for (size_t wi = b0; wi < b1; ++wi) {
      const auto& item = work[g][wi];
      const int64_t i = item.first;
      const int j = item.second;
      const uint16_t* xr = x + static_cast<int64_t>(tok[i]) * H;
      for (int c = 0; c < H; ++c) xv[c] = bf16_value(xr[c]);
      // gate row r and up row I + r of the gate_up projection
      for (int r = 0; r < I; ++r) {
        double gsum = 0.0, usum = 0.0;
        const double* wg = &wgu[static_cast<size_t>(r) * H];
        const double* wu = &wgu[static_cast<size_t>(I + r) * H];
        for (int c = 0; c < H; ++c) gsum += wg[c] * xv[c];
        for (int c = 0; c < H; ++c) usum += wu[c] * xv[c];
        a[r] = silu(gsum) * usum;
      }
      if (h) std::memcpy(&hbuf[(static_cast<size_t>(i) * J + j) * I], a.data(), sizeof(double) * I);
      double* yr = &ybuf[(static_cast<size_t>(i) * J + j) * H];
      for (int r = 0; r < H; ++r) {
        double s = 0.0;
        const double* wd = &wdn[static_cast<size_t>(r) * I];
        for (int c = 0; c < I; ++c) s += wd[c] * a[c];
        yr[r] = s;
      }
    }
  });

  // Combine: out[t] = sum_j w[t, j] * y[t, j] (j in rank order) + y_shared[t], in fp64.
  for (int64_t i = 0; i < n; ++i) {
    for (int c = 0; c < H; ++c) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j)
        acc += rw[static_cast<size_t>(tok[i]) * k + j] * ybuf[(static_cast<size_t>(i) * J + j) * H + c];
      if (has_shared) acc += ybuf[(static_cast<size_t>(i) * J + k) * H + c];
      out[i * H + c] = acc;
    }
  }
  if (h) std::memcpy(h, hbuf.data(), sizeof(double) * hbuf.size());
  if (y) std::memcpy(y, ybuf.data(), sizeof(double) * ybuf.size());
  return 0;
}

}  // extern "C"

// ---------------------------------------------------------------------------------------
// FP8-activation arm.  The "long-context cold prefill" issue of the Atlas project describes
// its transposed prefill kernels as e4m3 x e4m3: the weights re-quantized to e4m3 (a second
// rounding of the NVFP4 values) and the activations in e4m3; its fix option (a) scales each
// token row into the e4m3 range (row absmax, computed in the gather) and applies the scale in
// the f32 epilogue.  Readings (the issue leaves them open): the weights are re-quantized per
// output row with the same rule as an activation row, from their exact values e2m1 x e4m3
// block scale (scale2 stays the group's fp32 factor); the SiLU(g) * u intermediate is rounded to
// bf16 as on the W4A16 path and then quantized per row like x before the down projection.
// ---------------------------------------------------------------------------------------

// e4m3 quantization of one row of fp32 values: amax = max |v|; inv = 448 / amax and
// scale = amax / 448, one fp32 division each (a row whose amax is 0 or not finite gets
// inv = scale = 1); code = e4m3 round-to-nearest-even, saturating at 448, of the fp32 product
// v * inv.  The row's value is then scale * e4m3(code).
void quant_row_e4m3(const float* v, int64_t K, uint8_t* codes, float* scale) {
  float amax = 0.0f;
  for (int64_t i = 0; i < K; ++i) amax = std::max(amax, std::fabs(v[i]));
  float inv = 1.0f, sc = 1.0f;
  if (amax > 0.0f && std::isfinite(amax)) {
    inv = 448.0f / amax;
    sc = amax / 448.0f;
  }
  for (int64_t i = 0; i < K; ++i) {
    const float q = v[i] * inv;
    codes[i] = static_cast<uint8_t>(e4m3_encode(q));
  }
  *scale = sc;
}

// Round a double to bf16 (8 significant bits, ties to even), returned as a double.
double round_bf16(double a) {
  if (a == 0.0 || !std::isfinite(a)) return a;
  const double tiny = std::ldexp(1.0, -126);
  if (std::fabs(a) < tiny) {   // bf16 subnormals: multiples of 2^-133
    const double q = std::ldexp(1.0, -133);
    return std::nearbyint(a / q) * q;
  }
  int e = 0;
  const double m = std::frexp(a, &e);   // a = m 2^e, 0.5 <= |m| < 1
  return std::ldexp(std::nearbyint(std::ldexp(m, 8)), e - 8);
}

extern "C" {

int orc_quant_rows_e4m3(const float* v, int64_t rows, int64_t K, uint8_t* codes, float* scale) {
  if (!v || !codes || !scale || rows < 0 || K <= 0) return -1;
  for (int64_t r = 0; r < rows; ++r) quant_row_e4m3(v + r * K, K, codes + r * K, scale + r);
  return 0;
}

int orc_prepare_fp8(const uint8_t* packed, const uint8_t* scales, int64_t G, int64_t N, int64_t K,
                    uint8_t* codes, float* row_scale) {
  if (!packed || !scales || !codes || !row_scale || G <= 0 || N <= 0 || K <= 0 || K % 16) return -1;
  const Tables& tb = tables();
  // rows are independent: blocks of 64 rows over the threads
  const int64_t rows = G * N, nb = (rows + 63) / 64;
  parallel_for(nb, thread_count(0), [&](int64_t b) {
    std::vector<float> w(static_cast<size_t>(K));
    for (int64_t r = b * 64; r < std::min(rows, b * 64 + 64); ++r) {
      const uint8_t* pr = packed + r * (K / 2);
      const uint8_t* sr = scales + r * (K / 16);
      for (int64_t c = 0; c < K; ++c) {
        const unsigned code = (c & 1) ? (pr[c / 2] >> 4) : (pr[c / 2] & 0xF);
        // e2m1 x e4m3 has at most 6 significant bits: exact in fp32
        w[c] = static_cast<float>(tb.e2m1_all[code] * tb.e4m3_all[sr[c / 16]]);
      }
      quant_row_e4m3(w.data(), K, codes + r * K, row_scale + r);
    }
  });
  return 0;
}

int orc_moe_forward_fp8(const uint16_t* x, const float* logits, const uint8_t* gu_codes,
                        const float* gu_rs, const float* gu_scale2, const uint8_t* dn_codes,
                        const float* dn_rs, const float* dn_scale2, int T, int H, int I, int E, int k,
                        int has_shared, const int32_t* tokens, int n_tok, double* out, double* h,
                        double* y, int n_threads) {
  if (!x || !logits || !gu_codes || !gu_rs || !gu_scale2 || !dn_codes || !dn_rs || !dn_scale2 ||
      !out || T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || k > E)
    return -1;
  std::vector<int32_t> tok;
  if (tokens) {
    tok.assign(tokens, tokens + n_tok);
    for (int32_t t : tok)
      if (t < 0 || t >= T) return -1;
  } else {
    tok.resize(T);
    for (int t = 0; t < T; ++t) tok[t] = t;
  }
  const int64_t n = static_cast<int64_t>(tok.size());
  const int J = k + (has_shared ? 1 : 0);
  std::vector<int32_t> ids(static_cast<size_t>(T) * k);
  std::vector<double> rw(static_cast<size_t>(T) * k);
  if (orc_route(logits, T, E, k, ids.data(), rw.data())) return -1;
  const int G = E + (has_shared ? 1 : 0);
  std::vector<std::vector<std::pair<int64_t, int>>> work(G);
  for (int64_t i = 0; i < n; ++i) {
    for (int j = 0; j < k; ++j) work[ids[static_cast<size_t>(tok[i]) * k + j]].push_back({i, j});
    if (has_shared) work[E].push_back({i, k});
  }
  // x rows quantized once per evaluated token (every expert of the token sees the same codes)
  std::vector<uint8_t> xq(static_cast<size_t>(n) * H);
  std::vector<float> xs(static_cast<size_t>(n));
  {
    std::vector<float> xf(H);
    for (int64_t i = 0; i < n; ++i) {
      const uint16_t* xr = x + static_cast<int64_t>(tok[i]) * H;
      for (int c = 0; c < H; ++c) xf[c] = static_cast<float>(bf16_value(xr[c]));
      quant_row_e4m3(xf.data(), H, &xq[static_cast<size_t>(i) * H], &xs[i]);
    }
  }
  std::vector<double> ybuf(static_cast<size_t>(n) * J * H, 0.0);
  std::vector<double> hbuf(h ? static_cast<size_t>(n) * J * I : 0, 0.0);
  const Tables& tb = tables();
  constexpr size_t kChunk = 64;
  std::vector<std::pair<int, size_t>> tasks;
  for (int g = 0; g < G; ++g)
    for (size_t b = 0; b < work[g].size(); b += kChunk) tasks.push_back({g, b});
  parallel_for(static_cast<int64_t>(tasks.size()), thread_count(n_threads), [&](int64_t ti) {
    const int64_t g = tasks[ti].first;
    const size_t b0 = tasks[ti].second, b1 = std::min(work[g].size(), b0 + kChunk);
    const uint8_t* wgu = gu_codes + g * (2LL * I) * H;
    const uint8_t* wdn = dn_codes + g * static_cast<int64_t>(H) * I;
    std::vector<double> xv(H), a(I);
    std::vector<float> hf(I);
    std::vector<uint8_t> hq(I);
    for (size_t wi = b0; wi < b1; ++wi) {
      const int64_t i = work[g][wi].first;
      const int j = work[g][wi].second;
      for (int c = 0; c < H; ++c) xv[c] = tb.e4m3_all[xq[static_cast<size_t>(i) * H + c]];
      for (int r = 0; r < I; ++r) {
        double gsum = 0.0, usum = 0.0;
        const uint8_t* wg = wgu + static_cast<int64_t>(r) * H;
        const uint8_t* wu = wgu + static_cast<int64_t>(I + r) * H;
        for (int c = 0; c < H; ++c) gsum += tb.e4m3_all[wg[c]] * xv[c];
        for (int c = 0; c < H; ++c) usum += tb.e4m3_all[wu[c]] * xv[c];
        const double gv = gsum * gu_rs[g * 2LL * I + r] * xs[i] * gu_scale2[g];
        const double uv = usum * gu_rs[g * 2LL * I + I + r] * xs[i] * gu_scale2[g];
        a[r] = silu(gv) * uv;
      }
      if (h) std::memcpy(&hbuf[(static_cast<size_t>(i) * J + j) * I], a.data(), sizeof(double) * I);
      // h as bf16, then quantized per row like x
      for (int r = 0; r < I; ++r) hf[r] = static_cast<float>(round_bf16(a[r]));
      float hs = 1.0f;
      quant_row_e4m3(hf.data(), I, hq.data(), &hs);
      double* yr = &ybuf[(static_cast<size_t>(i) * J + j) * H];
      for (int r = 0; r < H; ++r) {
        double s = 0.0;
        const uint8_t* wd = wdn + static_cast<int64_t>(r) * I;
        for (int c = 0; c < I; ++c) s += tb.e4m3_all[wd[c]] * tb.e4m3_all[hq[c]];
        yr[r] = s * dn_rs[g * static_cast<int64_t>(H) + r] * hs * dn_scale2[g];
      }
    }
  });
  for (int64_t i = 0; i < n; ++i) {
    for (int c = 0; c < H; ++c) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j)
        acc += rw[static_cast<size_t>(tok[i]) * k + j] * ybuf[(static_cast<size_t>(i) * J + j) * H + c];
      if (has_shared) acc += ybuf[(static_cast<size_t>(i) * J + k) * H + c];
      out[i * H + c] = acc;
    }
  }
  if (h) std::memcpy(h, hbuf.data(), sizeof(double) * hbuf.size());
  if (y) std::memcpy(y, ybuf.data(), sizeof(double) * ybuf.size());
  return 0;
}

}  // extern "C"
