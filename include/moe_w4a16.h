/*
 * moe_w4a16.h -- C ABI of the routed-expert W4A16 MoE layer for GB300 (sm_103a).
 *
 * What the layer computes (sources are the pages describing the model):
 *   - Shapes and weight format: "Kimi-K2.6" (model-catalog page), GEOMETRY,
 *     QUANT and PARAMS paragraphs -- hidden 7168, 384 routed experts, 8 per
 *     token, moe_intermediate_size 2048; the routed experts are an INT4 bank
 *     (compressed-tensors, pack-quantized, symmetric, group size 32, int4
 *     weights in int32 containers); one shared expert kept in higher precision.
 *   - The routed MoE with its routing and W4A16 expert kernels:
 *     "feat(pytorch): support Kimi K2.6", Motivation and Changes.
 *   The pages do not spell out the router, the nibble order or the activation;
 *   the readings this library implements are:
 *     score_e = sigmoid(logit_e) in fp32 (a fixed sequence of IEEE fp32
 *       operations, identical on every run and every device: see moe_route);
 *     top-k by score, lowest expert index first on ties, weights renormalised
 *       to sum to 1;
 *     weight q in [-8, 7] stored as nibble q + 8, input 8c + j of a row in bits
 *       4j..4j+3 of the row's int32 word c; one bf16 scale per 32 inputs;
 *     expert(x) = W2 * (SiLU(W_gate x) .* (W_up x)),
 *     out[t] = sum_j w[t,j] * expert_{id[t,j]}(x[t]) (+ shared(x[t])).
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers unless the name ends in _host. bf16 values
 *     travel as uint16_t bit patterns. Arrays are row-major, C-contiguous, the
 *     input (K) dimension innermost. Device pointers must be 16-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Every
 *     call is asynchronous and stream-ordered, unless documented otherwise.
 *   - The caller owns every buffer. The library allocates no device memory,
 *     keeps no per-call state, and holds only a per-device cache of device
 *     properties and a process-wide launch counter.
 *   - Argument and shape errors are returned synchronously, before anything
 *     is launched. A failed launch returns MOE_ERR_CUDA. Errors found on the
 *     device (an expert id out of range, a bounded wait that expired) are
 *     recorded in the workspace status word and reported by moe_check_status.
 *   - T == 0 is a no-op that returns MOE_OK.
 *   - Shape rules: 1 <= top_k <= E <= 1024; H and I multiples of 32 in
 *     [32, 32768]; group == 32; 0 <= T and T * top_k <= 2^24.
 */
#ifndef MOE_W4A16_H
#define MOE_W4A16_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,          /* null pointer, negative size, bad op code    */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,    /* violates the shape rules above              */
  MOE_ERR_WORKSPACE_TOO_SMALL = 3,  /* ws_bytes < moe_workspace_size(...)          */
  MOE_ERR_CUDA = 4,                 /* a CUDA runtime/driver call failed           */
  MOE_ERR_DEVICE_TIMEOUT = 5,       /* a bounded device wait expired (status word) */
  MOE_ERR_DEVICE_BOUNDS = 6,        /* an expert id outside [0, E) (status word)   */
  MOE_ERR_UNSUPPORTED_DEVICE = 7    /* not a compute capability 10.3 device        */
} moe_status_t;

/* Layer dimensions. group must be 32. */
typedef struct {
  int32_t E;      /* routed experts                    */
  int32_t top_k;  /* experts per token                 */
  int32_t H;      /* hidden size                       */
  int32_t I;      /* expert intermediate size          */
  int32_t group;  /* inputs per scale (32)             */
} moe_dims_t;

/* Weights of one layer (device pointers). Per expert e:
 *   w13_packed[e] : int32 [2I][H/8]  rows 0..I-1 = gate, rows I..2I-1 = up
 *   w13_scale[e]  : bf16  [2I][H/32]
 *   w2_packed[e]  : int32 [H][I/8]
 *   w2_scale[e]   : bf16  [H][I/32]
 * Optional dense bf16 shared expert (both NULL and shared_I == 0 if absent):
 *   shared_wgu    : bf16  [2*shared_I][H]  gate rows first
 *   shared_wd     : bf16  [H][shared_I]
 * shared_I must be a multiple of 64. */
typedef struct {
  const int32_t* w13_packed;
  const uint16_t* w13_scale;
  const int32_t* w2_packed;
  const uint16_t* w2_scale;
  const uint16_t* shared_wgu;
  const uint16_t* shared_wd;
  int32_t shared_I;
} moe_weights_t;

/* Weights of one layer in the 4-bit float format (NVFP4-style checkpoints).
 * Passage: "Kimi k2.5 MLA based eagle3", test plan (an NVFP4 checkpoint of the
 * model family) and "Probing the Depths: Verifying SGLang Compatibility for
 * Kimi K2.6 Deployment", Assumption 2 (nvfp4_pack_quantized). The pages name
 * the format without spelling it out; the reading is the published NVFP4
 * layout. Per expert e:
 *   w13_packed[e] : int32 [2I][H/8]  E2M1 codes (sign, 2 exponent bits with
 *                   bias 1, 1 mantissa bit) in the INT4 bank's nibble places
 *   w13_scale[e]  : uint8 [2I][H/16] FP8 E4M3 scale of each 16 inputs
 *   w13_gscale[e] : fp32             scale of the whole matrix
 *   w2_packed[e]  : int32 [H][I/8], w2_scale[e] : uint8 [H][I/16], w2_gscale[e]
 *   W[n][i] = e2m1(code) * e4m3(scale[n][i/16]) * gscale
 * The shared expert is the bf16 one of moe_weights_t. moe_dims_t.group must
 * be 16 for this format. */
typedef struct {
  const int32_t* w13_packed;
  const uint8_t* w13_scale;
  const float* w13_gscale;
  const int32_t* w2_packed;
  const uint8_t* w2_scale;
  const float* w2_gscale;
  const uint16_t* shared_wgu;
  const uint16_t* shared_wd;
  int32_t shared_I;
} moe_weights_fp4_t;

/* Grouped GEMM operations. */
#define MOE_GEMM_GATEUP_SILU 0   /* h[r, :] = SiLU(W_gate a[r]) .* (W_up a[r]), out [R][I] */
#define MOE_GEMM_DOWN 1          /* y[r, :] = W2 a[r],                          out [R][H] */

/* Flags (bitwise OR). 0 selects the default tensor-core path. */
#define MOE_FLAG_GEMM_SIMT 0x1u  /* grouped GEMMs on the CUDA-core baseline kernel        */
#define MOE_FLAG_A_SMEM 0x2u     /* stage dequantised weights in shared memory, not TMEM  */
/* Activation rows exchanged between the steps are stored in the tensor-core
 * GEMM's K order: inside every block of 8 consecutive inputs, position p holds
 * input [0,4,1,5,2,6,3,7][p]. With this flag moe_permute writes x_perm that way
 * and moe_w4a16_grouped_gemm reads a_rows that way and (gate/up) writes h that
 * way, so the calls chain exactly as moe_forward runs them; without it every
 * row is in natural order. */
#define MOE_FLAG_ROWS_MMA_ORDER 0x4u
/* The down projection (moe_w4a16_grouped_gemm with MOE_GEMM_DOWN, and the
 * shared expert) writes its rows in fp32 instead of bf16: out_rows / out are
 * then float arrays of the same shape, to be summed by moe_combine_f32.
 * moe_forward keeps these rows in fp32 internally: the layer output is then
 * rounded to bf16 once, in the combine. Not valid with MOE_GEMM_GATEUP_SILU. */
#define MOE_FLAG_OUT_F32 0x8u
/* Run the int4 grouped GEMMs on CTA pairs: one tensor-core MMA (M = 256)
 * covers the weight rows of two SMs, each SM dequantising its own 128 rows and
 * loading half of the token rows. Same results as the one-SM kernel up to the
 * order of fp32 additions inside the tensor cores. Ignored with
 * MOE_FLAG_GEMM_SIMT or MOE_FLAG_A_SMEM. */
#define MOE_FLAG_GEMM_PAIR 0x10u
/* moe_workspace_size(..., MOE_FLAG_ROUTER_PROJECT) sizes the workspace of
 * moe_forward_project (the layer plus the router's logits). */
#define MOE_FLAG_ROUTER_PROJECT 0x20u
/* Bits 8..15: token rows per tile of the tensor-core GEMM: 16, 32, 64 or 128
 * (16 or 32 with MOE_FLAG_A_SMEM); 0 lets the library choose from T * top_k / E.
 * Any other value makes the GEMM calls return MOE_ERR_UNSUPPORTED_SHAPE. */
#define MOE_FLAG_TOKENS_PER_TILE(n) ((uint32_t)(n) << 8)

/* Text of a status code (static storage; never NULL). */
MOE_API const char* moe_status_string(moe_status_t s);

/* Bytes of workspace that moe_forward / moe_forward_host need for T tokens
 * (shared_I = 0 without a shared expert). A workspace of this size also serves
 * every other entry point for the same dims and T. Returns 0 for invalid dims.
 * Before its first use the first 256 bytes of a workspace must be zero. */
MOE_API size_t moe_workspace_size(moe_dims_t d, int32_t T, int32_t shared_I, uint32_t flags);

/* Step 1, routing. Passage: "feat(pytorch): support Kimi K2.6", Motivation and
 * Changes ("MoE routing"); "Kimi-K2.6" catalog page, GEOMETRY ("384 routed
 * experts, 8 per token"). The pages name routing but not its function; the
 * sigmoid / top-k / renormalise reading is the one stated at the top.
 * logits fp32 [T][E] -> topk_ids int32 [T][k] and topk_w fp32
 * [T][k], in rank order (score descending, expert index ascending on ties).
 * score = 1 / (1 + e(-logit)), every operation one IEEE fp32 operation rounded
 * to nearest even, with e(t) = p(r) * 2^n, n = rint(t * log2 e),
 * r = (t - n * LN2_HI) - n * LN2_LO (Cody-Waite split of ln 2, LN2_HI the
 * multiple of 2^-14 nearest ln 2), p the degree-7 Taylor polynomial of exp in
 * Horner form; e(t) = +inf for t > 88 and 0 for t < -87. NaN scores rank below
 * all numbers. w_j = s_j / (s_0 + ... + s_{k-1}) (sum in rank order); all
 * weights are 1/k when that sum is 0. Bit-identical on every device. */
MOE_API moe_status_t moe_route(const float* logits, int32_t T, int32_t E, int32_t k,
                       int32_t* topk_ids, float* topk_w, void* stream);

/* The router's logit projection. Passage: "feat(pytorch): support Kimi K2.6",
 * Motivation and Changes ("MoE routing"); "Kimi-K2.6" catalog page, GEOMETRY
 * (hidden 7168, 384 routed experts). The pages print no router; the reading
 * is the plain linear gate of a routed MoE:
 *   logits fp32 [T][E] = x bf16 [T][H] . w_gate^T, w_gate bf16 [E][H],
 * products of bf16 values summed in fp32 on the tensor cores (the order of
 * the fp32 additions is the hardware's: logits agree with an fp32 reference
 * to rounding, not bit for bit). H a multiple of 32, 1 <= E <= 1024.
 * ws: the status word in its first 256 bytes, then the K-slice sums of small
 * batches; ws_bytes >= moe_router_workspace_size(T, E, H). flags:
 * MOE_FLAG_GEMM_SIMT runs the CUDA-core kernel instead. */
MOE_API size_t moe_router_workspace_size(int32_t T, int32_t E, int32_t H);
MOE_API moe_status_t moe_router_logits(const uint16_t* x, const uint16_t* w_gate, int32_t T, int32_t E,
                               int32_t H, float* logits, void* ws, size_t ws_bytes, uint32_t flags,
                               void* stream);

/* moe_router_logits, then moe_route on those logits: topk_ids, topk_w as
 * moe_route gives them (the selection is bit-exact for the logits written). */
MOE_API moe_status_t moe_route_project(const uint16_t* x, const uint16_t* w_gate, int32_t T, int32_t E,
                               int32_t H, int32_t k, float* logits, int32_t* topk_ids, float* topk_w,
                               void* ws, size_t ws_bytes, uint32_t flags, void* stream);

/* The router's score function alone, element-wise: scores[i] = score(logits[i]). */
MOE_API moe_status_t moe_sigmoid_scores(const float* logits, int64_t n, float* scores, void* stream);

/* Step 2, expert-sorted permutation. Passage: "Kimi-K2.6" catalog page,
 * GEOMETRY (8 of 384 experts per token) and "feat(pytorch): support Kimi
 * K2.6", Changes (W4A16 MoE kernels). The pages print no permutation: this
 * step is the design choice that groups each expert's rows so its int4
 * weights are read once per batch by one grouped GEMM. Assignment i = t*k + j goes to row
 * inv_perm[i]; rows are grouped by expert, expert e owning rows
 * [expert_offsets[e], expert_offsets[e+1]), and within an expert ordered by
 * increasing i (a stable sort). sorted_token_ids[row] = the row's token.
 *   topk_ids int32 [T][k] -> expert_offsets int32 [E+1], sorted_token_ids
 *   int32 [T*k], inv_perm int32 [T*k].
 * If x (bf16 [T][H]) and x_perm (bf16 [T*k][H]) are both non-NULL, also
 * gathers x_perm[row] = x[sorted_token_ids[row]]. An id outside [0, E) sets
 * MOE_ERR_DEVICE_BOUNDS in the status word and that assignment is left out
 * (its inv_perm entry is -1; no out-of-bounds access). Deterministic: no
 * result depends on timing. ws: status word in its first 256 bytes, then
 * 4 * E * ceil(T*k / 4096) bytes of scratch (a moe_workspace_size workspace
 * is large enough). flags: MOE_FLAG_ROWS_MMA_ORDER stores x_perm rows in the
 * tensor-core K order. */
MOE_API moe_status_t moe_permute(const int32_t* topk_ids, int32_t T, int32_t E, int32_t k,
                         int32_t* expert_offsets, int32_t* sorted_token_ids, int32_t* inv_perm,
                         const uint16_t* x, int32_t H, uint16_t* x_perm,
                         void* ws, size_t ws_bytes, uint32_t flags, void* stream);

/* moe_permute for callers that have no device memory to give and may not
 * allocate any: a hook inside an engine that reserved all of HBM for its own
 * pool, or a latency-critical path where cudaMalloc/cudaFree (which can
 * synchronise the device) are not allowed. The pages describing the method
 * have no counterpart of this call; it exists only for such callers.
 *
 * Same arguments, results and rules as moe_permute, except that the
 * histograms come from a fixed array of MOE_PERMUTE_STATIC_SCRATCH_BYTES of
 * device memory inside the library image (loaded once on every device that
 * uses it, held until the process exits) and no workspace is passed. The call
 * allocates nothing. It returns MOE_ERR_WORKSPACE_TOO_SMALL when the
 * histograms, 4 * E * ceil(T*k / 4096) bytes, would exceed that array (with
 * E = 384, T*k up to 2,793,472 fits; with E = 1024, up to 1,048,576).
 *
 * status: a caller-owned device int32 that must be 0 before the first call;
 * an id outside [0, E) sets MOE_ERR_DEVICE_BOUNDS in it (read and reset it
 * with moe_check_status(status, stream)). May be NULL: such ids are then
 * still left out (inv_perm entry -1) but not reported. Nothing in the
 * library's own array has to start at zero.
 *
 * Set-up: the first call on a device, with that device current, looks up the
 * array's device address (this can load the library's module onto the
 * device) and checks the device; make that first call before any stream
 * capture. Later calls on the device only launch kernels. A set-up that
 * failed (MOE_ERR_CUDA, for instance inside a capture) is not remembered:
 * the next call on that device tries again. MOE_ERR_UNSUPPORTED_DEVICE is
 * final for that device.
 *
 * Every call on a device uses the same array: calls whose kernels overlap on
 * the GPU (other streams, other host threads, without ordering between them)
 * race and give wrong results. Calls on one stream are ordered and safe. */
#define MOE_PERMUTE_STATIC_SCRATCH_BYTES (1u << 20)
MOE_API moe_status_t moe_permute_static_scratch(const int32_t* topk_ids, int32_t T, int32_t E, int32_t k,
                                        int32_t* expert_offsets, int32_t* sorted_token_ids,
                                        int32_t* inv_perm, const uint16_t* x, int32_t H,
                                        uint16_t* x_perm, int32_t* status, uint32_t flags,
                                        void* stream);

/* Steps 3 and 4, the grouped W4A16 GEMMs over expert-sorted rows. Passage:
 * "Kimi-K2.6" catalog page, QUANT and PARAMS (INT4 via compressed-tensors,
 * group size 32, pack-quantized, symmetric, int4 weights in int32 containers)
 * and GEOMETRY (hidden 7168, moe_intermediate_size 2048; three H x I matrices
 * per expert by the I32 parameter count); "feat(pytorch): support Kimi
 * K2.6", Changes ("compressed-tensors W4A16 MoE"). Row r of
 * a_rows (bf16 [R][K], R = T*k) belongs to the expert e with
 * expert_offsets[e] <= r < expert_offsets[e+1]. Each weight is dequantised as
 * bf16(q * scale) and the products accumulate in fp32 on the tensor cores.
 *   op = MOE_GEMM_GATEUP_SILU: K = H, out_rows bf16 [R][I],
 *        out = bf16(SiLU(g) * u), g and u the gate and up rows of W13_e.
 *   op = MOE_GEMM_DOWN:        K = I, out_rows bf16 [R][H], out = bf16(W2_e a).
 * flags: MOE_FLAG_GEMM_SIMT, MOE_FLAG_A_SMEM, MOE_FLAG_TOKENS_PER_TILE(n),
 * MOE_FLAG_ROWS_MMA_ORDER (a_rows and, for gate/up, out_rows in the tensor-core
 * K order), MOE_FLAG_OUT_F32 (down only: out_rows is fp32 [R][H]). ws: the status word in its first 256 bytes; the tensor-core path
 * with natural-order rows also rewrites a_rows into the K order right after
 * it, so ws_bytes >= 256 + R*K*2 (rounded up to 256) unless
 * MOE_FLAG_ROWS_MMA_ORDER or MOE_FLAG_GEMM_SIMT is set. */
MOE_API moe_status_t moe_w4a16_grouped_gemm(int32_t op, moe_dims_t d, const moe_weights_t* w,
                                    const uint16_t* a_rows, int32_t T,
                                    const int32_t* expert_offsets, uint16_t* out_rows,
                                    void* ws, size_t ws_bytes, uint32_t flags, void* stream);

/* moe_w4a16_grouped_gemm over 4-bit float weights (moe_weights_fp4_t, group
 * 16): each E2M1 code times its E4M3 scale is exact in bf16, the products sum
 * in fp32 on the tensor cores and the matrix scale multiplies the fp32 sums.
 * Same arguments, flags and workspace as moe_w4a16_grouped_gemm, except that
 * MOE_FLAG_GEMM_SIMT and MOE_FLAG_A_SMEM return MOE_ERR_UNSUPPORTED_SHAPE. */
MOE_API moe_status_t moe_fp4_grouped_gemm(int32_t op, moe_dims_t d, const moe_weights_fp4_t* w,
                                  const uint16_t* a_rows, int32_t T, const int32_t* expert_offsets,
                                  uint16_t* out_rows, void* ws, size_t ws_bytes, uint32_t flags,
                                  void* stream);

/* The dense bf16 shared expert. Passage: "Kimi-K2.6" catalog page, GEOMETRY
 * (n_shared_experts 1, moe_intermediate_size 2048) and PARAMS (the BF16
 * share of the checkpoint, outside the INT4 bank).
 * out bf16 [T][H] = Wd (SiLU(Wg x) .* (Wu x)) for
 * x bf16 [T][H], fp32 accumulation. Needs w->shared_wgu, w->shared_wd, and
 * moe_workspace_size(d, T, w->shared_I, flags) bytes of workspace. With
 * MOE_FLAG_OUT_F32, out is fp32 [T][H]. */
MOE_API moe_status_t moe_shared_expert(moe_dims_t d, const moe_weights_t* w, const uint16_t* x, int32_t T,
                               uint16_t* out, void* ws, size_t ws_bytes, uint32_t flags, void* stream);

/* Step 5, combine. Passage: "Kimi-K2.6" catalog page, GEOMETRY (8 routed
 * experts plus one shared expert per token, summed into one output);
 * "feat(pytorch): support Kimi K2.6", Changes ("MoE routing": the routing
 * weights scale the experts' outputs).
 * out[t] = bf16( sum_j topk_w[t][j] * y[inv_perm[t*k+j]]
 * (+ addend[t]) ), fp32 accumulation in rank order j, one rounding at the end.
 * y_rows bf16 [T*k][H], addend bf16 [T][H] or NULL, out bf16 [T][H]. */
MOE_API moe_status_t moe_combine(const uint16_t* y_rows, const int32_t* inv_perm, const float* topk_w,
                         int32_t T, int32_t k, int32_t H, const uint16_t* addend,
                         uint16_t* out, void* stream);

/* moe_combine over fp32 rows: y_rows fp32 [T*k][H] (the down projection with
 * MOE_FLAG_OUT_F32), addend fp32 [T][H] or NULL; the same sum in rank order,
 * rounded to bf16 once. This is the combine moe_forward runs: with no bf16
 * rounding of the rows before the sum, the layer's largest outputs keep their
 * error within the stated bound. */
MOE_API moe_status_t moe_combine_f32(const float* y_rows, const int32_t* inv_perm, const float* topk_w,
                             int32_t T, int32_t k, int32_t H, const float* addend,
                             uint16_t* out, void* stream);

/* The whole layer. Passage: "feat(pytorch): support Kimi K2.6", Motivation
 * and Changes (the compressed-tensors W4A16 MoE with its routing) and
 * "Kimi-K2.6" catalog page, GEOMETRY/QUANT (384 INT4 routed experts, 8 per
 * token, one higher-precision shared expert).
 * Route, permute (with gather), gate/up GEMM, down GEMM,
 * the shared expert when w has one, combine.
 *   x bf16 [T][H], logits fp32 [T][E] -> out bf16 [T][H].
 * ws_bytes >= moe_workspace_size(d, T, w->shared_I, flags). */
MOE_API moe_status_t moe_forward(moe_dims_t d, const moe_weights_t* w, const uint16_t* x, const float* logits,
                         int32_t T, uint16_t* out, void* ws, size_t ws_bytes, uint32_t flags,
                         void* stream);

/* moe_forward with 4-bit float routed experts (and the optional bf16 shared
 * expert): workspace, flags and results as moe_forward (d.group == 16). */
MOE_API moe_status_t moe_forward_fp4(moe_dims_t d, const moe_weights_fp4_t* w, const uint16_t* x,
                             const float* logits, int32_t T, uint16_t* out, void* ws, size_t ws_bytes,
                             uint32_t flags, void* stream);

/* The routed-expert bank in host memory. Passage: "Kimi-K2.6" catalog page,
 * the paragraph on running with expert offload (8 of 384 experts per token:
 * a token's expert traffic is a small slice of the checkpoint, so the bank can
 * sit in system RAM).
 * moe_stage_experts copies, for every expert e with rows (expert_offsets[e+1]
 * > expert_offsets[e]), its W13, W13 scales, W2 and W2 scales from host_w to
 * the same places of dev_w; other experts' places in dev_w are left as they
 * are. host_w's four routed tensors must be page-locked host memory mapped
 * into the device's address space (cudaHostAlloc, or pinned memory on a
 * unified-addressing system): the GPU reads them over the host link
 * (NVLink-C2C on a Grace-Blackwell node). Otherwise MOE_ERR_INVALID_ARG is
 * returned before anything is launched. host_w's shared-expert pointers are
 * not read. dev_w: a device bank of the full bank's layout (a layer's worth
 * of device memory, reusable for every layer of a model).
 * moe_forward_offload is moe_forward with the bank in host memory: route,
 * permute, stage the touched experts into dev_w, then the GEMMs read dev_w
 * (dev_w's bf16 shared expert, if any, stays resident). */
MOE_API moe_status_t moe_stage_experts(moe_dims_t d, const moe_weights_t* host_w, const int32_t* expert_offsets,
                               const moe_weights_t* dev_w, void* stream);
MOE_API moe_status_t moe_forward_offload(moe_dims_t d, const moe_weights_t* host_w, const moe_weights_t* dev_w,
                                 const uint16_t* x, const float* logits, int32_t T, uint16_t* out, void* ws,
                                 size_t ws_bytes, uint32_t flags, void* stream);

/* The whole layer from the token activations alone: the router logits are
 * projected from x with w_gate (bf16 [E][H], as moe_router_logits) into the
 * workspace, then the layer runs as moe_forward on them.
 * ws_bytes >= moe_workspace_size(d, T, w->shared_I, MOE_FLAG_ROUTER_PROJECT). */
MOE_API moe_status_t moe_forward_project(moe_dims_t d, const moe_weights_t* w, const uint16_t* w_gate,
                                 const uint16_t* x, int32_t T, uint16_t* out, void* ws, size_t ws_bytes,
                                 uint32_t flags, void* stream);

/* moe_forward from and to HOST buffers: copies x_host and logits_host into the
 * workspace, runs the layer, copies the result to out_host, all enqueued on
 * `stream`; the call returns before the copies finish (synchronise the stream
 * before reading out_host). Host buffers should be page-locked for the copies
 * to be asynchronous. ws_bytes >= moe_workspace_size(...) plus
 * moe_host_staging_size(d, T). */
MOE_API size_t moe_host_staging_size(moe_dims_t d, int32_t T);
MOE_API moe_status_t moe_forward_host(moe_dims_t d, const moe_weights_t* w, const uint16_t* x_host,
                              const float* logits_host, int32_t T, uint16_t* out_host,
                              void* ws, size_t ws_bytes, uint32_t flags, void* stream);

/* Parameter-free RMSNorm of each row: out[t][i] = bf16(x[t][i] / r_t) with
 * r_t = sqrt(mean_i x[t][i]^2 + eps), in fp32 (squares summed, one IEEE
 * square root, one IEEE division per element). x, out bf16 [T][H], H a
 * multiple of 8; out may not overlap x. */
MOE_API moe_status_t moe_rmsnorm(const uint16_t* x, int32_t T, int32_t H, float eps, uint16_t* out, void* stream);

/* A stack of L routed-expert layers joined as pre-norm residual blocks,
 *   x_{l+1} = x_l + MoE_l(RMSNorm(x_l)),   l = 0 .. L-1,   out = x_L.
 * The catalog page gives 60 MoE layers of this shape ("Kimi-K2.6", GEOMETRY)
 * but not how they are joined; a bare x + MoE(x) grows without bound within
 * a few layers, and the usual pre-norm residual with a parameter-free norm is
 * the reading used here. Each layer's residual add happens inside its combine
 * (fp32, one bf16 rounding together with the layer's output).
 *   layers: HOST array of L weight sets (all with the same shared_I);
 *   logits: HOST array of L DEVICE pointers, fp32 [T][E] each (the router
 *           logits of each layer are inputs here);
 *   x, out: bf16 [T][H]; out may equal x.
 * ws_bytes >= moe_stack_workspace_size(d, T, shared_I, flags). The status word
 * is the workspace's, as for moe_forward. */
MOE_API size_t moe_stack_workspace_size(moe_dims_t d, int32_t T, int32_t shared_I, uint32_t flags);
MOE_API moe_status_t moe_stack_forward(moe_dims_t d, const moe_weights_t* layers, int32_t L,
                               const float* const* logits, const uint16_t* x, int32_t T, float eps,
                               uint16_t* out, void* ws, size_t ws_bytes, uint32_t flags, void* stream);

/* Synchronises `stream`, reads the workspace status word, resets it to 0 and
 * returns it (MOE_OK if no device error was recorded since the last check). */
MOE_API moe_status_t moe_check_status(void* ws, void* stream);

/* Number of kernels this library has launched in this process. */
MOE_API uint64_t moe_launch_count(void);

/* Self-test of the bounded device waits: launches one block that waits on a
 * barrier nothing will complete, for at most timeout_ns (clamped to 1 ms ..
 * 2 s), then records MOE_ERR_DEVICE_TIMEOUT in the status word and returns.
 * The GPU stays usable. */
MOE_API moe_status_t moe_debug_expire_wait(void* ws, int64_t timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_W4A16_H */
