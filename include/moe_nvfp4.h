/*
 * moe_nvfp4.h -- C ABI of the GB300 (sm_103a) NVFP4 routed mixture-of-experts layer.
 *
 * The layer is the one the Atlas project's "long-context cold prefill to SGLang parity" issue
 * states for NVFP4 checkpoints (kernel comparison table, untransposed W4A16 column):
 *   bf16 activations; expert weights stored as e2m1 values x one e4m3 scale per 16-element
 *   K block x one fp32 per-tensor scale2; f32 accumulation; SiLU(gate)*up intermediate in
 *   bf16; an fp32 weighted unpermute/combine; an always-on shared expert.
 * Its stages are the tensors the same issue's op-dump list names (router logits, top-k ids and
 * weights, the token permutation, shared-expert in/out, routed outputs before combine, the
 * combine result), and each stage is one call below.  `moe_forward` runs them all.
 *
 * Conventions for every call
 *  - Memory: every tensor argument is DEVICE memory owned by the caller.  The library never
 *    allocates or frees.  Scratch comes from the caller's workspace `ws` (size from
 *    moe_workspace_size), which the call may overwrite; 256-byte alignment is required for
 *    `ws` and 16-byte alignment for every other device pointer.  The first 4 bytes of `ws` hold
 *    the device status word: zero-fill a new workspace once before its first use, and again
 *    after a call reported MOE_ERR_DEVICE_TIMEOUT (the one-launch decode kernel keeps a grid
 *    barrier counter in the workspace, which a timed-out launch may leave mid-instance).
 *  - Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls only
 *    enqueue work; none synchronizes the host, none copies device data to the host (the
 *    route and permutation results stay on the device, so no host round trip breaks stream
 *    capture, as the "handover briefs" page requires of its device-side selection), so a
 *    call sequence can be captured in a CUDA graph.
 *  - Errors: argument and shape errors are returned before anything is enqueued.  A failed
 *    launch returns MOE_ERR_CUDA.  Errors detected on the device (a bounded wait that ran
 *    out) are written to a status word in `ws`; read it with moe_get_device_status.
 *  - Sizes: T >= 0 tokens (T = 0 enqueues nothing); H % 128 == 0, 128 <= H <= 16384;
 *    I % 128 == 0, 128 <= I <= 8192; 1 <= E <= 1024; 1 <= k <= min(E, 16);
 *    T * (k + 1) < 2^31.  The shared expert, when present, has the routed experts' I.
 *  - Data types: bf16 tensors are passed as their 16-bit patterns (uint16_t).
 *
 * Weight layout (one projection, all groups): the resident [N, K/2] layout that the issue prices
 * as the option without a dequantization pass or a transpose:
 *    packed [G, N, K/2] bytes, element k of row n in byte k/2, even k in the low nibble;
 *    scales [G, N, K/16] e4m3 bytes, one per 16 consecutive k of a row;
 *    scale2 [G] fp32, one per group and projection;
 *    G = E + has_shared groups, the shared expert is group E.
 *  gate_up: N = 2I, K = H (rows 0..I-1 are gate, rows I..2I-1 are up).  down: N = H, K = I.
 *
 * Row conventions of the staged tensors: S = T*k slots, slot s = t*k + j for rank j of
 * token t.  h [S+T, I] (bf16) and y [S+T, H] (fp32) hold the routed slots in permuted order
 * (row p is slot sorted_slot[p]) followed by one shared-expert row per token (row S + t).
 * h is bf16 because the issue's table fixes the SiLU intermediate as bf16; the expert outputs y
 * feed an fp32 weighted sum and are kept in fp32 (rounding them to bf16 before the combine
 * costs up to ~2.5% of a row's RMS in the worst element).
 */
#ifndef MOE_NVFP4_H
#define MOE_NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,          /* null/misaligned pointer, inconsistent struct */
  MOE_ERR_UNSUPPORTED_SHAPE = -2,    /* sizes outside the supported ranges above */
  MOE_ERR_WORKSPACE_TOO_SMALL = -3,  /* ws_bytes < moe_workspace_size(shape) */
  MOE_ERR_ARCH = -4,                 /* current device is not compute capability 10.3 */
  MOE_ERR_CUDA = -5,                 /* a CUDA runtime call or launch failed */
  MOE_ERR_DEVICE_TIMEOUT = -6        /* a device-side bounded wait ran out */
} moe_status_t;

/* Sizes of one MoE layer. */
typedef struct {
  int32_t T;           /* tokens (rows of x) */
  int32_t H;           /* hidden size */
  int32_t I;           /* expert intermediate size (routed and shared) */
  int32_t E;           /* routed experts */
  int32_t k;           /* experts per token */
  int32_t has_shared;  /* 1: an always-on shared expert is group E; 0: none */
} moe_shape_t;

/* One NVFP4 projection of every group (device pointers, caller-owned; layout above). */
typedef struct {
  const uint8_t* packed;
  const uint8_t* scales;
  const float* scale2;
  int32_t G, N, K;
} moe_nvfp4_weights_t;

/* Bytes of workspace every call below needs for this shape (0 on an unsupported shape). */
size_t moe_workspace_size(const moe_shape_t* shape);

/* Router top-k (the top-k after the router GEMM, in the issue's list of logit-changing ops; the
 * tie rule is the handover briefs' device selection: lower index wins, NaN never wins).
 *   logits   fp32 [T, E]
 *   topk_ids int32 [T, k]: experts ordered by (logit descending, index ascending), NaN as -inf
 *   topk_w   fp32 [T, k]: softmax over all E, restricted to the k picks and renormalised to
 *            sum 1 (= a softmax over the k selected logits).  A token whose logits are all
 *            -inf/NaN gets weights 0; +inf logits share the mass equally. */
moe_status_t moe_route_topk(const float* logits, const moe_shape_t* shape, int32_t* topk_ids,
                            float* topk_w, void* stream);

/* Token permutation by expert (the issue's "token permutation" dump), built on the device.
 *   topk_ids    int32 [T, k] (values in [0, E))
 *   counts      int32 [E]     slots routed to each expert
 *   offsets     int32 [E + 1] exclusive prefix sum of counts (offsets[E] = S)
 *   sorted_slot int32 [S]     slot ids sorted by expert, ascending slot id within an expert
 *   slot_pos    int32 [S]     inverse: sorted_slot[slot_pos[s]] == s
 * Bit-exact and deterministic. */
moe_status_t moe_permute(const int32_t* topk_ids, const moe_shape_t* shape, int32_t* counts,
                         int32_t* offsets, int32_t* sorted_slot, int32_t* slot_pos, void* ws,
                         size_t ws_bytes, void* stream);

/* Grouped gate_up GEMM with SiLU(gate)*up fused (the issue's fused gate_up kernel, W4A16):
 * for routed row p (expert e with offsets[e] <= p < offsets[e+1]) and x row t = sorted_slot[p]/k,
 *   g = scale2_e * (x_t . deq(W_e[r]))   for gate rows r < I,  u likewise for up rows I + r,
 *   h[p, r] = bf16(SiLU(g) * u), accumulated in fp32;
 * and the shared expert (group E) for h rows S + t over every token t.
 *   x [T, H] bf16; h [S + T, I] bf16 (shared rows written only when has_shared). */
moe_status_t moe_grouped_gate_up(const uint16_t* x, const int32_t* sorted_slot,
                                 const int32_t* offsets, const moe_nvfp4_weights_t* gate_up,
                                 const moe_shape_t* shape, uint16_t* h, void* ws, size_t ws_bytes,
                                 void* stream);

/* Grouped down GEMM (the issue's pointer-table grouped GEMM): y[p] = scale2 * (h[p] .
 * deq(Wd_e)^T) accumulated in fp32 for every routed row p of expert e and, for the shared
 * expert, rows S + t.   h [S + T, I] bf16 -> y [S + T, H] fp32. */
moe_status_t moe_grouped_down(const uint16_t* h, const int32_t* offsets,
                              const moe_nvfp4_weights_t* down, const moe_shape_t* shape,
                              float* y, void* ws, size_t ws_bytes, void* stream);

/* fp32 weighted unpermute/combine ("fp32 weighted sum" of the issue's table; fixed summation
 * order as in the expert-parallel discussion of the TensorFold sm_120 issue):
 *   out[t] = (sum_{j=0..k-1} topk_w[t, j] * y[slot_pos[t*k + j]]) + y[S + t]
 * summed in fp32 in exactly that order, then written as bf16 (out_is_fp32 = 0) or fp32. */
moe_status_t moe_combine(const float* y, const int32_t* slot_pos, const float* topk_w,
                         const moe_shape_t* shape, void* out, int out_is_fp32, void* stream);

/* The whole layer: route, permute, grouped gate_up(+SiLU), grouped down, combine, with the
 * shared expert.  Same numerics contract as the stage calls; out is [T, H] bf16 or fp32.  The
 * arm depends on the shape (see moe_forward_arm): decode/verify batches stream only the
 * selected experts' bytes through grouped GEMVs, prefill batches run the grouped GEMM on the
 * tensor cores. */
moe_status_t moe_forward(const uint16_t* x, const float* logits,
                         const moe_nvfp4_weights_t* gate_up, const moe_nvfp4_weights_t* down,
                         const moe_shape_t* shape, void* out, int out_is_fp32, void* ws,
                         size_t ws_bytes, void* stream);

/* moe_forward with per-stage timing (the per-stage microsecond hooks of the handover briefs'
 * measure-first steps, as CUDA events).  stage_events, when not NULL, points to 5 cudaEvent_t
 * (created with timing enabled) that are recorded on `stream`: [0] before routing, [1] after
 * the permutation and work list (on arm 2 also the expert-ordered f16 copy of x), [2] after the
 * gate_up GEMM, [3] after down (on arm 2 with the f16 conversion of h), [4] after combine.  On the
 * decode arm down and combine are one kernel, so [3] and [4] are recorded together; on arm 0
 * (see moe_forward_arm) the whole layer is one kernel and [1]..[4] follow it.  With
 * stage_events == NULL this is moe_forward. */
moe_status_t moe_forward_profiled(const uint16_t* x, const float* logits,
                                  const moe_nvfp4_weights_t* gate_up,
                                  const moe_nvfp4_weights_t* down, const moe_shape_t* shape,
                                  void* out, int out_is_fp32, void* ws, size_t ws_bytes,
                                  void* stream, void* const* stage_events);

/* Router GEMM in front of the top-k (the issue's list of logit-changing operations includes the
 * router GEMM; its nsys table times the router as a W4A16 GEMM):
 *   logits[t, e] = scale2 * (x[t] . deq(W_r[e])), accumulated in fp32, written fp32 [T, E].
 *   router: one NVFP4 projection of the experts' layout with G = 1, N = E rows, K = H.
 * Batches above 8 tokens with E % 128 == 0 and H % 256 == 0 run on the tcgen05 grouped GEMM
 * (x converted to f16 rows scaled by a power of two, as in that arm); other shapes on a CUDA-core
 * kernel.  ws as for moe_forward (its size covers this call). */
moe_status_t moe_router_logits(const uint16_t* x, const moe_nvfp4_weights_t* router, const moe_shape_t* shape,
                               float* logits, void* ws, size_t ws_bytes, void* stream);

/* moe_router_logits into the workspace, then moe_forward on those logits: the layer from x
 * alone.  Same numerics and arms as moe_forward; the routing decisions are taken on the fp32
 * logits the router GEMM produced. */
moe_status_t moe_forward_routed(const uint16_t* x, const moe_nvfp4_weights_t* router,
                                const moe_nvfp4_weights_t* gate_up, const moe_nvfp4_weights_t* down,
                                const moe_shape_t* shape, void* out, int out_is_fp32, void* ws, size_t ws_bytes,
                                void* stream);

/* The one-launch decode forward (moe_forward_arm == 0 shapes: T <= 8, H % 512 == 0, H <= 4096,
 * I % 256 == 0, I <= 1024) for callers that cannot allocate device memory -- code running where
 * cudaMalloc is not allowed or not available, such as inside a framework's memory-planning phase,
 * a host callback, or a plugin whose host application owns every device allocation and only
 * passes in tensor pointers.  No workspace argument: the scratch (routing results, permutation,
 * the layer's h and expert outputs, the status word and the decode kernel's counters) lives in
 * one 4 MiB array in device global memory that the library declares at file scope; every GPU that
 * loads the library holds it until the library is unloaded.  The pages have no counterpart to
 * this call; it is a deployment aid.
 *   - Inputs, weights and out are as for moe_forward; nothing is allocated or freed.
 *   - Shapes outside arm 0 return MOE_ERR_UNSUPPORTED_SHAPE, and so would a shape whose scratch
 *     exceeded 4 MiB (h and the expert outputs take T (k+1) (2 I + 4 H) bytes, at most 2.5 MB on
 *     arm-0 shapes, so every arm-0 shape fits).
 *   - All calls on a device share the array: calls that overlap on the GPU (other streams or
 *     threads) race and corrupt each other; serialize them.
 *   - The first call in a context looks up the array's device address (a caller that makes
 *     another context current gets that context's own lookup); make the first call outside any
 *     CUDA stream capture.
 *   - Not supported across a device reset.  The library carries its own copy of the CUDA
 *     runtime, so a cudaDeviceReset (or a reset of the primary context) made by other code in
 *     the process is not seen by it, and its kernels and this array are not reloaded: after such
 *     a reset, unload the library (or restart the process) before calling it again.
 *   - Each call first clears the status word, the launch count and the decode kernel's counters
 *     on `stream` (an asynchronous memset).
 *     Device-side timeouts are not reported back by this call. */
moe_status_t moe_forward_decode_static_scratch(const uint16_t* x, const float* logits,
                                               const moe_nvfp4_weights_t* gate_up,
                                               const moe_nvfp4_weights_t* down,
                                               const moe_shape_t* shape, void* out,
                                               int out_is_fp32, void* stream);

/* Load-time NVFP4 quantizer of fp32 weights [G, N, K] (K % 16 == 0, finite values) into the
 * layout above, with the recipe of the benchmark configurations: scale2 = amax / (448 * 6);
 * block scale = e4m3_rne_satfinite(block_amax / 6 / scale2); code = e2m1_rne_satfinite(
 * w / (e4m3(scale) * scale2)); every step one fp32 operation; a block whose scale decodes to 0
 * stores code 0.  Not on the hot path (weights are quantized once, at load). */
moe_status_t moe_quantize_nvfp4(const float* w, int64_t G, int64_t N, int64_t K, uint8_t* packed,
                                uint8_t* scales, float* scale2, void* stream);

/* Reads (and clears) the device status word of a workspace: *status receives MOE_OK or the
 * first device-side error recorded since the last read.  Synchronizes `stream`. */
moe_status_t moe_get_device_status(void* ws, int32_t* status, void* stream);

/* Test hook for the device-side timeout path (the pages have no counterpart): one warp waits,
 * with the one-launch decode kernel's bounded wait, on a shared-memory barrier that nothing
 * arrives at, for limit_ns nanoseconds of the global timer (1 .. 1e9).  The wait runs out and
 * records MOE_ERR_DEVICE_TIMEOUT in the workspace status word, as a stalled wait inside a
 * forward would; nothing faults or hangs.  ws: a workspace (256-byte aligned; only its status
 * word is written).  Returns MOE_OK once the probe is launched on `stream`; read the result
 * with moe_get_device_status. */
moe_status_t moe_debug_timeout_probe(void* ws, uint64_t limit_ns, void* stream);

/* ---------------------------------------------------------------------------------------------
 * FP8-activation prefill arm (a separate arm with its own numerics).  The "long-context cold
 * prefill to SGLang parity" issue runs its transposed prefill kernels as e4m3 x e4m3 (weights
 * re-quantized to e4m3, a second rounding) and lists as fix (a) a per-token-row e4m3 activation
 * scale computed in the gather and applied in the f32 epilogue.  Every e4m3 operand row here
 * carries one fp32 scale under one rule:
 *   amax = max |v| over the row; inv = 448 / amax, scale = amax / 448 (IEEE fp32 divisions; a row
 *   whose amax is 0 or not finite gets inv = scale = 1); code = e4m3 round-to-nearest-even,
 *   saturating at 448, of the fp32 product v * inv.  The row's value is scale * e4m3(code).
 * Weight rows are re-quantized from their exact NVFP4 values (e2m1 x e4m3 block scale; scale2
 * stays the group's factor); x rows are quantized per token; h = SiLU(g) * u is rounded to bf16
 * as on the W4A16 path and then quantized per row before down.
 * ------------------------------------------------------------------------------------------- */

/* One e4m3 projection of every group (device pointers, caller-owned). */
typedef struct {
  const uint8_t* codes;      /* [G, N, K] e4m3, row-major */
  const float* row_scale;    /* [G, N] fp32 */
  const float* scale2;       /* [G] fp32, the NVFP4 projection's own */
  int32_t G, N, K;
} moe_fp8_weights_t;

/* Load-time re-quantization of an NVFP4 projection: codes [G, N, K] and row_scale [G, N] (the
 * caller's device buffers, 16-byte aligned) by the row rule above; scale2 is not touched (point
 * the fp8 weights at the NVFP4 scale2).  K % 256 == 0.  Asynchronous on stream. */
moe_status_t moe_prepare_fp8(const moe_nvfp4_weights_t* w, uint8_t* codes, float* row_scale, void* stream);

/* The row rule on bf16 rows: x [rows, K] -> codes [rows, K] e4m3, scale [rows] fp32 (the
 * quantization the FP8 arm applies to activation rows).  K % 256 == 0. */
moe_status_t moe_quantize_rows_e4m3(const uint16_t* x, int64_t rows, int32_t K, uint8_t* codes, float* scale,
                                    void* stream);

/* The whole layer on the FP8-activation arm: route and permute as moe_forward, x rows
 * quantized per token and gathered into expert order, e4m3 x e4m3 grouped gate_up on the tensor
 * cores (fp32 accumulation, epilogue x scale2 x weight-row scale x x-row scale, SiLU(g) * u ->
 * bf16 h), h rows quantized, grouped down (-> fp32 y), then moe_combine's fixed-order sum.
 * Shapes of moe_forward_arm 2 only (T > 8, H and I multiples of 256); the workspace is
 * moe_workspace_size(shape). */
moe_status_t moe_forward_fp8(const uint16_t* x, const float* logits, const moe_fp8_weights_t* gate_up,
                             const moe_fp8_weights_t* down, const moe_shape_t* shape, void* out, int out_is_fp32,
                             void* ws, size_t ws_bytes, void* stream);

/* Which kernels moe_forward runs for a shape (-1 for an unsupported shape):
 *   0  T <= 8 (H % 512 == 0, H <= 4096, I % 256 == 0, I <= 1024, and room in shared memory for
 *      a ring of three slots): one cooperative launch that routes, streams the active experts'
 *      weights with TMA copies, multiplies on the tensor cores and combines;
 *   1  T <= 8 otherwise, and 8 < T <= 64 when H or I is not a multiple of 256: three launches
 *      (route+permute, gate_up GEMV, down GEMV + combine);
 *   2  T > 8, H and I multiples of 256: tcgen05 grouped GEMMs (batched decode and prefill);
 *   3  T > 64 otherwise: CUDA-core grouped GEMMs. */
int moe_forward_arm(const moe_shape_t* shape);

/* Per-expert choice inside the arm-2 grouped GEMMs (the handover briefs' MoE decode-arm brief
 * wants the grouped arm to engage only where a group is wide and tiny groups to take a GEMV-like
 * path, decided on the device): a work item whose expert group has at most `rows` token rows runs
 * on the dequant warps of the same persistent launch as a register-operand mma.sync product with
 * the group's tokens as the 8 MMA columns, instead of TMEM staging and tcgen05; wider groups stay
 * on tcgen05.  The choice is made per item on the device from the permutation's counts.
 *   rows  0 (every item on tcgen05), 1..8, or -1 (the library's default for the shape).
 * Process-wide; takes effect for calls issued afterwards (a captured CUDA graph keeps the value
 * it was captured with).  Returns MOE_ERR_INVALID_ARG outside [-1, 8].  Numerics are those of
 * the grouped GEMMs (exact f16 operands, fp32 accumulation); only the accumulation order of the
 * MMA differs between the two arms. */
moe_status_t moe_set_narrow_rows(int rows);

/* Static description of a status code. */
const char* moe_status_string(moe_status_t status);

#ifdef __cplusplus
}
#endif
#endif /* MOE_NVFP4_H */
