/*
 * CPU oracle of the NVFP4 routed-MoE layer -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg use this code.
 * It shares no source, header, table or helper with the CUDA library; the two meet only in
 * the seeded inputs that the `synth` module draws.
 *
 * The layer it computes (W4A16 routed mixture of experts with NVFP4 expert weights) is the
 * one the "long-context cold prefill to SGLang parity" issue of the Atlas project states in
 * its kernel comparison table (untransposed column: bf16 activations, e2m1 x e4m3 block x
 * scale2 weights, f32 accumulation, SiLU intermediate, fp32 weighted unpermute/combine) and
 * in its op-dump list (router logits, top-k ids/weights, token permutation, shared-expert
 * in/out, routed outputs before combine, combine result).  Routing ties follow the
 * "handover briefs" page (device-side indexer selection: lower index wins, NaN never wins).
 *
 * Every function computes the plain definition: no blocking, no fusion, fp64 arithmetic for
 * the layer.  The quantizer is the exception: its inputs are fp32 weights and the recipe it
 * follows (scale2 = amax / (448*6), block scale = block amax / 6 / scale2, code = w / (block
 * scale * scale2)) is stated on those fp32 values, so each of its steps is one fp32 operation
 * on fp32 data, taken in the order the recipe writes them.
 *
 * Status: 0 = ok, -1 = invalid argument.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* --- NVFP4 element formats (from their bit definitions) --- */
double orc_e2m1_value(int code);        /* 4-bit code -> value, -0 for code 8 */
double orc_e4m3_value(int code);        /* 8-bit E4M3 (no inf) -> value, NaN for 0x7F/0xFF */
int orc_e2m1_encode(float v);           /* round to nearest, ties to even code, saturate at 6 */
int orc_e4m3_encode(float v);           /* round to nearest, ties to even code, saturate at 448 */

/* --- NVFP4 quantizer: w fp32 [G, N, K] -> packed [G, N, K/2] (low nibble = even k),
 *     scales [G, N, K/16] e4m3, scale2 [G] fp32.  K % 16 == 0. --- */
int orc_quantize(const float* w, int64_t G, int64_t N, int64_t K,
                 uint8_t* packed, uint8_t* scales, float* scale2);
/* exact fp64 dequantization of the same layout -> out [G, N, K] */
int orc_dequantize(const uint8_t* packed, const uint8_t* scales, const float* scale2,
                   int64_t G, int64_t N, int64_t K, double* out);

/* --- router GEMM: logits fp64 [T, E] = x (bf16 bit patterns [T, H]) . deq(W_r)^T, with the
 *     router weights one NVFP4 projection (packed [E, H/2], scales [E, H/16], scale2 [1]), the
 *     layout of the experts' weights.  The "long-context cold prefill" issue of the Atlas project
 *     counts the router GEMM among the MoE's logit-changing operations, and its nsys table times
 *     the router as a W4A16 GEMM.  H % 16 == 0. --- */
int orc_router_logits(const uint16_t* x, const uint8_t* packed, const uint8_t* scales, const float* scale2,
                      int T, int H, int E, double* logits);

/* --- routing: logits fp32 [T, E] -> ids int32 [T, k] (rank order), w fp64 [T, k] --- */
int orc_route(const float* logits, int T, int E, int k, int32_t* ids, double* w);

/* --- permutation: stable counting sort of slots s = t*k + j by expert --- */
int orc_permute(const int32_t* ids, int T, int E, int k, int32_t* counts, int32_t* offsets,
                int32_t* sorted_slot, int32_t* slot_pos);

/* --- layer forward in fp64.
 * x: bf16 bit patterns [T, H]; logits fp32 [T, E].
 * gate_up: packed [G, 2I, H/2], scales [G, 2I, H/16], scale2 [G]; rows 0..I-1 gate, I..2I-1 up.
 * down:    packed [G, H, I/2],  scales [G, H, I/16],  scale2 [G].
 * G = E + has_shared (the shared expert is group E).
 * tokens: the n_tok token indices to evaluate (NULL = all T, in order).
 * out fp64 [n_tok, H].  Optional dumps (may be NULL), per evaluated token i and rank j
 * (j = k is the shared expert):  h fp64 [n_tok, k+1, I],  y fp64 [n_tok, k+1, H].
 * n_threads <= 0 uses every hardware thread. --- */
int orc_moe_forward(const uint16_t* x, const float* logits,
                    const uint8_t* gu_packed, const uint8_t* gu_scales, const float* gu_scale2,
                    const uint8_t* dn_packed, const uint8_t* dn_scales, const float* dn_scale2,
                    int T, int H, int I, int E, int k, int has_shared,
                    const int32_t* tokens, int n_tok, double* out, double* h, double* y,
                    int n_threads);

/* --- FP8-activation arm (the "long-context cold prefill" issue: its transposed prefill kernels run
 * e4m3 x e4m3 with the weights re-quantized to e4m3, and its option (a) gives each token row an
 * e4m3 scale, applied in the f32 epilogue).
 * Row rule: amax = max |v|, inv = 448 / amax and scale = amax / 448 (fp32 divisions; amax 0 or
 * not finite -> inv = scale = 1), code = e4m3 nearest-even saturating of the fp32 product v * inv.
 * orc_quant_rows_e4m3: v fp32 [rows, K] -> codes [rows, K], scale [rows].
 * orc_prepare_fp8: NVFP4 packed/scales [G, N, ..] -> codes [G, N, K], row_scale [G, N]: each row's
 *   exact values e2m1 x e4m3(block scale) under the row rule (scale2 stays the group factor).
 * orc_moe_forward_fp8: the layer of orc_moe_forward with x rows quantized by the row rule,
 *   gate/up = scale2 * row_scale * x_scale * sum(e4m3 w * e4m3 x) in fp64, h = SiLU(g) * u
 *   rounded to bf16 and quantized by the row rule, y = scale2 * row_scale * h_scale *
 *   sum(e4m3 w * e4m3 h), combine as orc_moe_forward.  Dumps: h before rounding, y. --- */
int orc_quant_rows_e4m3(const float* v, int64_t rows, int64_t K, uint8_t* codes, float* scale);
int orc_prepare_fp8(const uint8_t* packed, const uint8_t* scales, int64_t G, int64_t N, int64_t K,
                    uint8_t* codes, float* row_scale);
int orc_moe_forward_fp8(const uint16_t* x, const float* logits,
                        const uint8_t* gu_codes, const float* gu_rs, const float* gu_scale2,
                        const uint8_t* dn_codes, const float* dn_rs, const float* dn_scale2,
                        int T, int H, int I, int E, int k, int has_shared,
                        const int32_t* tokens, int n_tok, double* out, double* h, double* y,
                        int n_threads);

#ifdef __cplusplus
}
#endif
#endif
