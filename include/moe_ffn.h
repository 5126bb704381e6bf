/*
 * moe_ffn.h -- C ABI of the GB300 fused MoE expert feed-forward with top-k combine.
 *
 * What the library computes (Ascend "mega_moe" page, "Computation Process", A16W16 use
 * case, and its A8W8-INT / A8W8-FP use cases; DeepGEMM MegaMoE page §4 for the
 * FP8-activation x FP4-weight recipe):
 *
 *     y_i = sum_{k<K} G[i,k] * Y_{e_ik}[row(i,k), :]
 *     Y_e = SwiGLU(X_e . W1[e]) . W2[e],   SwiGLU(H) = SiLU(H[:, :I]) * H[:, I:]
 *
 * in five stages on one GPU: route metadata (count, prefix sum, scatter), dispatch (gather
 * of the routed x rows into a per-expert pool), L1 grouped GEMM with SwiGLU and
 * re-quantisation fused, L2 grouped GEMM with the gate weight applied, and the combine of
 * the K weighted rows of each token in fixed slot order.
 *
 * Conventions shared by every entry point
 *   - All tensors are row-major and contiguous. Pointers marked "device" must point to
 *     device memory of the current CUDA device; the library reads inputs, writes outputs
 *     and the caller's workspace, and keeps no pointer after the call returns.
 *   - The library allocates nothing. The caller owns every buffer, including the workspace
 *     of moe_workspace_bytes() bytes (256-byte aligned).
 *   - Every call is asynchronous on `stream` (NULL = legacy default stream) and never
 *     synchronises the host, except moe_check_device_error().
 *   - Argument errors are found on the host before anything is launched and returned as a
 *     status. Errors found on the device (an expert id outside [-1, E), a bounded wait
 *     that ran out) are recorded in the workspace's error word; read them with
 *     moe_check_device_error().
 *   - Limits: 0 <= T, 1 <= K <= 32, K <= E <= 1024, H and I multiples of 128, and
 *     T*K <= 2^24; with S shared experts, K + S <= 32, E + S <= 1024 and T*(K+S) <= 2^24.
 */
#ifndef MOE_FFN_H
#define MOE_FFN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* A CUDA stream (cudaStream_t / CUstream) without including CUDA headers. */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* a size, pointer or alignment the op does not accept  */
    MOE_ERR_UNSUPPORTED = 2,   /* a mode / shape combination this build does not run    */
    MOE_ERR_CUDA = 3,          /* a CUDA runtime call or kernel launch failed           */
    MOE_ERR_BAD_ROUTE = 4,     /* device: an expert id outside [-1, E); route skipped   */
    MOE_ERR_TIMEOUT = 5,       /* device: a bounded wait ran out; results are invalid   */
    MOE_ERR_WORKSPACE = 6,     /* workspace missing, misaligned or too small            */
    MOE_ERR_BAD_SCALE = 7,     /* device: an FP8 x FP4 x scale that is not a power of two
                                  2^e, -127 <= e <= 127; the outputs are not defined     */
    MOE_ERR_BOUNDS = 8         /* device, builds with MOE_DEBUG only: an index outside its
                                  buffer; the access was skipped, results are invalid   */
} moe_status;

/* Storage formats of the five use cases (Ascend mega_moe page, "Use Case / A / W" table;
 * DeepGEMM page §1 for FP8 x FP4). T tokens, H hidden, I intermediate, E experts.
 *
 * MOE_A16W16        x bf16 [T,H]; w1 bf16 [E,H,2I]; w2 bf16 [E,I,H] (the page's math
 *                   layout: hidden x 2*intermediate per expert). No scales.
 * MOE_A8W8_FP8      x e4m3 [T,H] + UE8M0 bytes [T,H/32]; w1 e4m3 [E,2I,H] + UE8M0
 *                   [E,2I,H/32]; w2 e4m3 [E,H,I] + UE8M0 [E,H,I/32] (the page's transposed
 *                   FP8 layout; its (N, K/64, 2) scale shape is this (N, K/32)).
 * MOE_A8W8_INT8     x int8 [T,H] in [-127,127] + fp32 [T] per-token scale; w1 int8
 *                   [E,2I,H] + fp32 [E,2I]; w2 int8 [E,H,I] + fp32 [E,H] per output channel.
 * MOE_A8W4_FP8_FP4  x e4m3 [T,H] + fp32 [T,H/128] power-of-two block scales (2^e with
 *                   -127 <= e <= 127: the tensor cores take the scale's exponent byte as a UE8M0
 *                   scale; the dispatch stage checks every scale and records
 *                   MOE_ERR_BAD_SCALE for any other value); w1 e2m1
 *                   [E,2I,H/2] + UE8M0 [E,2I,H/32]; w2 e2m1 [E,H,I/2] + UE8M0 [E,H,I/32];
 *                   two e2m1 codes per byte, element 2j in the low nibble.
 * MOE_A8W4_INT      x as MOE_A8W8_INT8; w1 signed int4 [E,2I,H/2] + fp32 [E,2I]; w2 signed
 *                   int4 [E,H,I/2] + fp32 [E,H] per output channel; two's-complement codes in
 *                   [-8,7], two per byte, element 2j in the low nibble. The page's INT4 x INT4
 *                   MSD split of the activations and its offline bias 8 * (1^T W) are one way
 *                   to reach the exact integer product Q . W; the library computes that product
 *                   directly, so no bias input exists (the page's A8W4-INT use case).
 * MOE_A8W8_FP8_E5M2 as MOE_A8W8_FP8 with FLOAT8_E5M2 codes for x, w1, w2 and the re-quantised
 *                   A (the page's A8W8-FP use case with the E5M2 target type).
 * In every mode the gate columns of w1 are the first I outputs and the up columns the
 * last I; y is bf16 [T,H]. */
typedef enum {
    MOE_A16W16 = 0,
    MOE_A8W8_FP8 = 1,
    MOE_A8W8_INT8 = 2,
    MOE_A8W4_FP8_FP4 = 3,
    MOE_A8W4_INT = 4,
    MOE_A8W8_FP8_E5M2 = 5
} moe_dtype_mode;

typedef struct {
    int32_t num_tokens;    /* T */
    int32_t hidden;        /* H */
    int32_t intermediate;  /* I: the width of A; w1 has 2*I outputs */
    int32_t num_experts;   /* E: routed experts */
    int32_t topk;          /* K: routed slots per token */
    int32_t num_shared_experts; /* S >= 0: shared experts (DeepGEMM page §6), see below */
} moe_dims;

/* Shared experts. Each of the S shared experts runs on every token, in the same mode as the
 * routed ones, and its output goes to a combine slot after the K routed slots with weight 1;
 * the combine sums it with them in slot order. The weights (w1, w2 and their scales) then
 * hold E + S experts: the E routed experts first, shared expert j at index E + j. topk_ids
 * and topk_weights stay [T,K]; a routed id in [E, E+S) is a bad route. Internally every token
 * has K + S slots (token i, slot k is row i*(K+S)+k), so the plan covers E + S experts and
 * T*(K+S) slots: the counts, offsets and row_src that moe_plan writes have E+S, E+S+1 and
 * T*(K+S) entries. S = 0 is the plain routed layer. */

/* A quantised tensor: its codes and, where the mode has them, its scales (device). */
typedef struct {
    const void* data;
    const void* scale;
} moe_operand;

/* Flags of the GEMM stages. */
enum {
    MOE_FLAG_NONE = 0u,
    MOE_FLAG_SIMT = 1u,         /* run the CUDA-core reference GEMMs instead of the tensor-core ones */
    MOE_FLAG_WEIGHT_MAJOR = 2u, /* FP8 modes at prefill sizes: one-CTA tiles of 128 weight rows x 128
                                   tokens (the decode-style tile) instead of 128 tokens x 256 weight
                                   rows; same results up to fp32 summation order, for comparison.
                                   A8W4-INT: weight-major tiles (128 weight rows x up to 256 tokens)
                                   whatever the tile count (see MOE_FLAG_TOKEN_MAJOR); same bits */
    MOE_FLAG_QUANTIZE_X = 4u,   /* moe_forward: x.data is bf16 [T,H] (x.scale unused) and the
                                   dispatch stage quantises it as moe_dispatch_quantize does */
    MOE_FLAG_FUSED = 8u,        /* moe_forward: S3-S6 through moe_expert_ffn (one launch with
                                   L1 -> L2 dependency counters; A16W16 also combines in it). Every
                                   mode, on the shapes moe_expert_ffn lists (else
                                   MOE_ERR_UNSUPPORTED); with MOE_FLAG_SIMT it is
                                   MOE_ERR_INVALID_ARG. Same results as the separate stages (FP8 and
                                   A8W4-INT: on weight-major tiles) bit for bit. */
    MOE_FLAG_SINGLE_CTA = 16u,  /* A16W16: the L2 GEMM on one-CTA 128-row tiles instead of CTA pairs
                                   (256-row tiles, tcgen05 cta_group::2); same results bit for bit,
                                   for comparison. The fused launch always uses one-CTA tiles. */
    MOE_FLAG_PAIR_L1 = 32u,     /* A16W16: the L1 GEMM on CTA pairs too (by default it runs on
                                   one-CTA tiles, measured faster at the power cap); same results
                                   bit for bit. Ignored with MOE_FLAG_SINGLE_CTA.
                                   FP8 modes at prefill sizes: both GEMMs on weight-major tiles on
                                   CTA pairs (256 weight rows x up to 192 tokens, tcgen05
                                   cta_group::2, where H and I allow) instead of the token-major
                                   tiles; same results up to fp32 summation order, for comparison
                                   (measured slower). */
    MOE_FLAG_TOKEN_MAJOR = 64u, /* A8W4-INT: token-major tiles (128 pool rows x 256 weight rows)
                                   where weight-major ones (128 weight rows x up to 256 tokens) would
                                   run: experts x weight slabs of at least four rounds of tiles on
                                   the GPU. Same results bit for bit, for comparison. */
    MOE_FLAG_PREPARED_WEIGHTS = 128u /* A8W8-INT: w1.data and w2.data hold the weights as
                                   moe_prepare_weights wrote them (every int8 code as the exact f16
                                   value, same [E,N,K] layout; the fp32 scales unchanged). The
                                   tensor-core GEMMs then load f16 tiles directly instead of
                                   expanding int8 tiles in shared memory; same results bit for bit.
                                   Other modes, or with MOE_FLAG_SIMT: MOE_ERR_UNSUPPORTED. */
};

/* Bytes of workspace that moe_plan / moe_forward and the stage calls need for `d` and `m`.
 * Returns 0 when `d` is outside the limits above. The caller allocates it (device memory,
 * 256-byte aligned); its contents need no initialisation. */
MOE_API size_t moe_workspace_bytes(const moe_dims* d, moe_dtype_mode m);

/* One-time weight preparation, outside the timed path (the DeepGEMM page, §3 host preparation,
 * transforms its weights offline the same way; the Ascend page's A8W8-INT use case fixes the
 * values: int8 codes with fp32 per-output-channel scales). For MOE_A8W8_INT8 it writes every int8
 * code of w1 (layer 1, [E,2I,H]) or w2 (layer 2, [E,H,I]) as the exact f16 value of the code, in
 * the same layout: the operand the INT8 tensor-core GEMMs take with MOE_FLAG_PREPARED_WEIGHTS, which
 * then need no conversion in shared memory. E counts the shared experts too.
 *   moe_prepared_weights_bytes  bytes of the prepared tensor (2 per weight); 0 when d is outside
 *             the limits, layer is not 1 or 2, or the mode has no prepared form (modes other than
 *             MOE_A8W8_INT8).
 *   w         device int8 weights of the layer (read-only); out: device buffer of at least that
 *             many bytes, 16-byte aligned, owned by the caller.
 * Errors: MOE_ERR_UNSUPPORTED for other modes; MOE_ERR_INVALID_ARG for a bad layer, d, pointer,
 * size or alignment (nothing launched). Asynchronous on `stream`. */
MOE_API size_t moe_prepared_weights_bytes(const moe_dims* d, moe_dtype_mode m, int layer);
MOE_API moe_status moe_prepare_weights(const void* w, const moe_dims* d, moe_dtype_mode m, int layer, void* out,
                                       size_t out_bytes, moe_stream_t stream);

/* Stage S1, route metadata (Ascend page, A16W16 "EP Dispatch": I_e, N_e = |I_e|, row(i,k);
 * metadata page §1 and §3: count -> prefix sum -> scatter).
 *   topk_ids  device int32 [T,K]: expert of each (token, slot); -1 = masked route (skipped);
 *             other ids outside [0,E) set MOE_ERR_BAD_ROUTE and are skipped.
 *   counts    device int32 [E]   or NULL: N_e, the routed rows of each expert (the page's
 *             expert_token_nums output).
 *   offsets   device int32 [E+1] or NULL: exclusive prefix sum of counts; offsets[E] = R.
 *   row_src   device int32 [T*K] or NULL: row_src[p] = i*K+k for p < R, the (token, slot)
 *             (with shared experts: E+S, E+S+1 and T*(K+S) entries, slots i*(K+S)+k)
 *             identity of routed row p; rows of expert e fill [offsets[e], offsets[e+1]),
 *             in an order the call does not fix (the page allows any fixed order).
 * The plan is also kept in the workspace for the stages that follow. */
MOE_API moe_status moe_plan(const int32_t* topk_ids, const moe_dims* d, int32_t* counts, int32_t* offsets,
                    int32_t* row_src, void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* Stage S2, dispatch: copies x row i (and its scales) into the workspace's pool row of every
 * routed (i, k), the single-GPU form of the page's EP Dispatch. Needs moe_plan first.
 *   x  device operand in the mode's x format. */
MOE_API moe_status moe_dispatch(moe_operand x, const moe_dims* d, moe_dtype_mode m, void* workspace,
                        size_t workspace_bytes, moe_stream_t stream);

/* Stage S2 from bf16 activations, with the operator's own quantisation before dispatch (Ascend
 * page: parameter dispatch_quant_mode; A8W8-INT and A8W4-INT use cases "EP Dispatch": per token
 * s_i = max|X[i,:]|/127, q_i = round(X[i,:]/s_i), scale floored at 1e-8; A8W8-FP use case, first
 * phase: Q_MX with groups of 32, e4m3 codes and E8M0 scales). For A8W4_FP8_FP4 the same
 * shared-exponent rule on groups of 128 gives e4m3 codes with fp32 power-of-two scales (the
 * mode's x format); A16W16 is the plain gather. Each token is quantised once and written to its
 * K pool rows. Every code is decided on fp32 values (IEEE division, round half to even).
 * Needs moe_plan first.
 *   x_bf16  device bf16 [T,H], row-major. */
MOE_API moe_status moe_dispatch_quantize(const void* x_bf16, const moe_dims* d, moe_dtype_mode m, void* workspace,
                                 size_t workspace_bytes, moe_stream_t stream);

/* Stages S3+S4, L1 grouped GEMM with SwiGLU and the L2-operand re-quantisation fused
 * (Ascend page: "Linear1 Projection", "SwiGLU Activation", and the A8W8 activation
 * quantisation of "Linear2"; DeepGEMM page §4 step 6). Needs moe_dispatch first.
 *   w1  device operand in the mode's w1 format. Writes the L2 operand A into the workspace:
 *       bf16 (A16W16), e4m3 + UE8M0 per 1x32 (A8W8_FP8, A8W4_FP8_FP4), e5m2 + UE8M0 per 1x32
 *       (A8W8_FP8_E5M2), int8 + fp32 per row (INT8, A8W4-INT). */
MOE_API moe_status moe_expert_l1(moe_operand w1, const moe_dims* d, moe_dtype_mode m, uint32_t flags,
                         void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* Stage S5, L2 grouped GEMM with the gate weight applied (Ascend page "Linear2 Projection"
 * and "Token Combine": w_k * Y_e[row(i,k)]). Needs moe_expert_l1 first.
 *   w2            device operand in the mode's w2 format.
 *   topk_weights  device fp32 [T,K] gate weights G.
 * Writes bf16(G[i,k] * Y[row(i,k)]) (product in fp32) into the workspace's combine row i*K+k. */
MOE_API moe_status moe_expert_l2(moe_operand w2, const float* topk_weights, const moe_dims* d, moe_dtype_mode m,
                         uint32_t flags, void* workspace, size_t workspace_bytes, moe_stream_t stream);


/* Stage S6, combine (Ascend page "Token Combine"): y[i,:] = bf16( sum_{k=0..K-1} c[i,k,:] )
 * summed in fp32 in slot order; masked slots contribute nothing. Needs moe_expert_l2 first.
 *   y  device bf16 [T,H]; every row is written. */
MOE_API moe_status moe_combine(void* y, const moe_dims* d, void* workspace, size_t workspace_bytes,
                       moe_stream_t stream);

/* The whole path: moe_plan, moe_dispatch, moe_expert_l1, moe_expert_l2, moe_combine in
 * stream order. Deterministic: the same inputs give bit-identical y. */
MOE_API moe_status moe_forward(moe_operand x, const int32_t* topk_ids, const float* topk_weights, moe_operand w1,
                       moe_operand w2, void* y, const moe_dims* d, moe_dtype_mode m, uint32_t flags,
                       void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* Options of the _ex entry points; zero-initialise, then set what is used (a null pointer means
 * all defaults).
 *   flags                 MOE_FLAG_* as for moe_forward
 *   has_activation_clamp  nonzero: clip both inputs of SwiGLU (the gate and the up halves of H)
 *                         to [-activation_clamp, activation_clamp] before SiLU and the product
 *                         (Ascend page, parameter activation_clamp); activation_clamp must be
 *                         >= 0 (else MOE_ERR_INVALID_ARG). */
typedef struct {
    uint32_t flags;
    uint32_t has_activation_clamp;
    float activation_clamp;
} moe_options;

/* moe_expert_l1 with options. */
MOE_API moe_status moe_expert_l1_ex(moe_operand w1, const moe_dims* d, moe_dtype_mode m, const moe_options* opt,
                            void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* moe_forward with options. */
MOE_API moe_status moe_forward_ex(moe_operand x, const int32_t* topk_ids, const float* topk_weights, moe_operand w1,
                          moe_operand w2, void* y, const moe_dims* d, moe_dtype_mode m, const moe_options* opt,
                          void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* Stages S3-S5, and S6 when y is given, in one persistent cooperative launch (the DeepGEMM
 * page's single kernel, §5): every L1 tile (GEMM + SwiGLU), then every L2 tile (GEMM + gate),
 * then the combine of every token. An L2 tile starts once all L1 tiles of its 128-row route
 * tile have published their A rows; a token's combine starts once every L2 tile holding one of
 * its rows has published them, so CTAs that finish their L2 tiles early combine while others
 * are still in L2. Every wait is bounded (on time-out MOE_ERR_TIMEOUT goes to the error word).
 * The results equal moe_expert_l1, moe_expert_l2 and moe_combine. Needs moe_dispatch first;
 * opt may be NULL (of its flags only MOE_FLAG_PREPARED_WEIGHTS is read; the activation clamp
 * applies).
 * A16W16 needs H a multiple of 256. The FP8 modes (A8W8-FP8 e4m3 or e5m2, FP8 x FP4) run S3 and
 * S4 on the weight-major block-scaled tiles in one launch (L2 tiles waiting on the same
 * per-route-tile counters; at decode sizes 16-token sub-tiles, else 128-token ones) and S6 as a
 * second launch when y is given; they need I a multiple of 64 and H and I multiples of 128. The
 * integer modes (A8W8-INT, A8W4-INT on weight-major tiles) run S3, the per-row re-quantisation
 * of A and S4 in one launch: the last L1 tile of each 128-row route tile to finish re-quantises
 * that route tile's rows, and its L2 tiles wait for that; S6 follows as a second launch. They
 * need I a multiple of 128, H a multiple of 256 and H, I <= 8704; A8W8-INT also takes weights
 * from moe_prepare_weights with MOE_FLAG_PREPARED_WEIGHTS in opt. Other shapes, and prepared
 * weights in another mode, return MOE_ERR_UNSUPPORTED before any launch.
 *   w1, w2, topk_weights  as for moe_expert_l1 and moe_expert_l2.
 *   y                     device bf16 [T,H] or NULL (then the combine rows stay in the
 *                         workspace for moe_combine). */
MOE_API moe_status moe_expert_ffn(moe_operand w1, moe_operand w2, const float* topk_weights, void* y,
                          const moe_dims* d, moe_dtype_mode m, const moe_options* opt, void* workspace,
                          size_t workspace_bytes, moe_stream_t stream);

/* Synchronises `stream`, returns the first device-side error recorded in the workspace
 * (MOE_OK if none) and clears it. */
MOE_API moe_status moe_check_device_error(void* workspace, moe_stream_t stream);

/* Static text for a status code. */
MOE_API const char* moe_status_string(moe_status s);

/* Byte offsets of the workspace regions, for inspection of the intermediate stages (E and K
 * below count the shared experts and their slots when S > 0: E + S and K + S). Rows of
 * expert e in the pools start at pad_offsets[e] (a multiple of the 128-row tile) and the
 * pool holds at most pool_rows rows. A region that a mode does not use has size 0. */
typedef struct {
    size_t header;        /* int32[16]: [0] error word, [1] R, [2] padded rows, [3] row tiles */
    size_t counts;        /* int32[E]   */
    size_t offsets;       /* int32[E+1] */
    size_t pad_offsets;   /* int32[E+1] padded row offsets of the pools */
    size_t tile_offsets;  /* int32[E+1] cumulative 128-row tiles */
    size_t row_src;       /* int32[T*K] unpadded pool row -> i*K+k */
    size_t pool_src;      /* int32[pool_rows] padded pool row -> i*K+k, -1 for padding */
    size_t slot_row;      /* int32[T*K] i*K+k -> padded pool row, -1 if masked */
    size_t gates;         /* shared experts: fp32 [T*(K+S)], the routed gates then 1 per shared
                             slot (written by moe_expert_l2; S = 0: size 0) */
    size_t x_pool;        /* gathered x codes [pool_rows, H] */
    size_t x_pool_scale;  /* gathered x scales [pool_rows, *] */
    size_t a_pool;        /* L2 operand codes [pool_rows, I] */
    size_t a_pool_scale;  /* L2 operand scales [pool_rows, *] */
    size_t a_f32;         /* fp32 A [pool_rows, I] (integer modes: before the per-row quantisation) */
    size_t x_pool_planes; /* INT8 mode: the gathered x codes as two f16 planes [2][pool_rows, H],
                             hi = floor(q/16) and lo = q mod 16; A8W4-INT: one plane, the codes
                             as f16 [pool_rows, H] (other modes: size 0) */
    size_t a_pool_planes; /* the re-quantised A likewise: [2][pool_rows, I] (INT8), [pool_rows, I]
                             (A8W4-INT). A8W4-INT stores each group of 8 consecutive codes
                             q0..q7 in the order q0 q4 q1 q5 q2 q6 q3 q7 (the order its weight
                             expansion produces) */
    size_t pool_sums;     /* A8W4-INT: int32 [2][pool_rows], the sum of each pool row's codes:
                             x rows, then A rows (other modes: size 0) */
    size_t comb;          /* bf16 [T*K, H] weighted rows */
    size_t ffn_counters;  /* int32 [5 * pool_rows/128 + 3 + T]: moe_expert_ffn's counters. Per
                             128-row route tile the finished L1 tiles; then A16W16: per token the
                             finished combine rows; FP8 modes: the launch's finished L1 tiles;
                             integer modes (each route tile also counts its finished
                             re-quantisation jobs): jobs finished, queue head, queue tail and
                             4 job slots per route tile */
    size_t total;         /* = moe_workspace_bytes() */
    int64_t pool_rows;    /* rows reserved in each pool */
} moe_workspace_layout_t;

MOE_API moe_status moe_workspace_layout(const moe_dims* d, moe_dtype_mode m, moe_workspace_layout_t* out);

/* moe_plan without a workspace, for callers that cannot allocate device memory where they
 * need the plan: a runtime that forbids cudaMalloc on its execution path, or a plugin host
 * that passes an operator its inputs and outputs but no scratch buffer. (The pages have no
 * counterpart of this call; it is an allocation-free variant of moe_plan.)
 *   topk_ids, counts, offsets, row_src  as for moe_plan (device memory, owned by the caller;
 *             counts and offsets are required, row_src is required when T*K > 0).
 *   d         checked exactly as moe_plan checks it (hidden and intermediate included), then:
 *   Limits: T*K <= 65536 and E <= 1024 (T*(K+S) and E+S with shared experts, whose slots the
 *   plan includes as moe_plan's does); larger sizes return MOE_ERR_INVALID_ARG and launch
 *   nothing. The call allocates nothing: its scratch is one fixed 1,590,272-byte device array
 *   inside the library that every GPU which loads the library holds until the process exits.
 *   The first call on a device looks up that array's device address (cudaGetSymbolAddress)
 *   with the device current; make that first call before any stream capture. The address
 *   belongs to the device's current CUDA context: after cudaDeviceReset (or any new context)
 *   the next call looks it up again, so make that call before a capture too.
 *   Every call shares the array and it keeps the last call's contents (the call clears what
 *   must start at zero itself); calls that overlap on the GPU race on it, so order them on
 *   one stream. Expert ids outside [-1, E) are skipped like masked routes; this call has no
 *   error word to report them (moe_plan does). */
MOE_API moe_status moe_plan_noalloc(const int32_t* topk_ids, const moe_dims* d, int32_t* counts, int32_t* offsets,
                                    int32_t* row_src, moe_stream_t stream);

/* Test hook for the failure path of a bounded device wait: launches one thread that waits
 * on a workspace flag that nothing sets, gives up after `timeout_ns` nanoseconds, records
 * MOE_ERR_TIMEOUT in the error word and returns. The device stays usable. */
MOE_API moe_status moe_debug_bounded_wait(void* workspace, size_t workspace_bytes, uint64_t timeout_ns,
                                  moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FFN_H */
