/*
 * gbmoe.h -- C ABI of the GB300 (sm_103a) fused Mixture-of-Experts layer.
 *
 * The layer (one sparse FFN of a MoE transformer) as the serving pages state
 * it (Xeon 6 / SGLang DeepSeek-R1 blog, section "MoE"; SGLang CPU backend
 * write-up, section "(3) FusedMoE"):
 *
 *   1. routing alignment: argsort the flat topk_ids so that the (token, slot)
 *      pairs of each expert are contiguous, pad every expert's group to a
 *      multiple of a block size and record the expert of every block;
 *   2. GEMM1 in the A x [B1, B2] = [C1, C2] form, W13 = [gate; up], with
 *      h = SiLU(C1) * C2 computed in the epilogue;
 *   3. GEMM2, the down projection y = h x W2^T;
 *   4. the weighted combine out[t] = sum_k topk_weights[t,k] * y[t,k].
 *
 * Weights are FP8 E4M3 with one fp32 scale per 128x128 block (DeepSeek-style
 * block quantisation), INT8 with one fp32 scale per output channel and
 * dynamic per-row INT8 activations (DA8W8), or INT4 with one fp32 scale per
 * row and 128 columns.  Weights stay in their stored format in HBM and are
 * expanded in registers or shared memory.
 *
 * Conventions shared by every entry point
 *  - All data pointers are DEVICE pointers owned by the caller.  The library
 *    allocates no memory and never synchronises the stream, except
 *    moe_read_status, which waits for the stream.
 *  - Every call is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and is ordered with the caller's other work on it.
 *  - Matrices are row-major and contiguous.
 *  - Host-checkable errors (bad sizes, NULL pointers, short workspace) are
 *    returned before anything is launched.  A failed launch returns
 *    MOE_ERR_CUDA.  Conditions only the GPU can see (expert ids outside
 *    [0, E)) are counted in a status word inside the workspace; read it with
 *    moe_read_status.
 *  - A flat slot index is i = t * topk + k for token t and top-k column k.
 *  - Calls that share a workspace must not overlap on the GPU.
 */
#ifndef GBMOE_H
#define GBMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* the same type as cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* a size or pointer argument is invalid            */
  MOE_ERR_UNSUPPORTED = 2, /* valid, but outside what the kernels implement    */
  MOE_ERR_WORKSPACE = 3,   /* workspace NULL, misaligned or smaller than asked */
  MOE_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed      */
  MOE_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up               */
  MOE_ERR_BAD_IDS = 6      /* the device saw expert ids outside [0, E)         */
} moe_status_t;

/* flags of fused_moe_fp8 / fused_moe_int8 / fused_moe_int4 / fused_moe_gated */
#define MOE_PATH_AUTO 0x0u    /* decode below MOE_AUTO_PREFILL_TOKENS tokens (INT4: up to
                                 MOE_MAX_DECODE_TOKENS), else prefill                 */
#define MOE_PATH_DECODE 0x1u  /* weight-streaming GEMV path (small token counts)    */
#define MOE_PATH_PREFILL 0x2u /* tcgen05 grouped-GEMM path (large token counts)     */
#define MOE_PATH_MASK 0x3u
/* fused_moe_fp8 only: FP8 x FP8 products.  x and the intermediate h are
 * quantised to E4M3 in groups of 1 x 128 (one fp32 scale per row and 128
 * columns, as moe_quant_act_fp8 does) before they enter the tensor cores.
 * Runs on the tcgen05 path at every M; MOE_PATH_DECODE with it is
 * MOE_ERR_UNSUPPORTED. */
#define MOE_ACT_FP8_1X128 0x10u

#define MOE_WEIGHT_FP8 0
#define MOE_WEIGHT_INT8 1
#define MOE_WEIGHT_INT4 2

/* Limits of this implementation (larger sizes return MOE_ERR_UNSUPPORTED). */
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_DECODE_TOKENS 128 /* MOE_PATH_DECODE handles M <= this */
#define MOE_AUTO_PREFILL_TOKENS 128 /* MOE_PATH_AUTO takes the tcgen05 path from this many tokens */

/*
 * Capacity (entries) of sorted_ids for the given routing problem:
 * M*topk + E*(block_size-1), rounded up to a multiple of block_size.  Every
 * expert may waste at most block_size-1 padding slots.  Returns 0 for
 * invalid arguments.
 */
size_t moe_align_max_padded(int M, int topk, int num_experts, int block_size);

/*
 * Routing alignment ("moe_align_index"): the argsort of topk_ids by expert,
 * blocked per expert (SGLang CPU backend write-up, section "(3) FusedMoE",
 * the moe_align_index and thread-offset paragraphs; Xeon 6 / SGLang blog,
 * section "MoE").
 *
 *   topk_ids        int32 [M, topk]   expert chosen by each (token, slot)
 *   sorted_ids      int32 [cap]       out: flat slot indices grouped by
 *                                     expert (ascending), ascending slot
 *                                     order inside an expert, each group
 *                                     padded to a multiple of block_size
 *                                     with the sentinel M*topk; the tail
 *                                     past the last group is sentinel too
 *   expert_ids      int32 [cap/block_size]  out: expert of each block, -1
 *                                     for blocks past the last group
 *   num_tokens_post_padded int32 [1]  out: sum of the padded group sizes
 *   expert_offsets  int32 [E+1]       out: start of each expert's group in
 *                                     sorted_ids (exclusive prefix sum)
 * cap = moe_align_max_padded(M, topk, E, block_size).  Slots whose id lies
 * outside [0, E) are left out (as a non-local expert would be).  Experts
 * with no slot get no block.  1 <= block_size <= 256, E <= MOE_MAX_EXPERTS.
 * The result is deterministic and equals a stable argsort bit for bit.
 */
moe_status_t moe_align_block_size(const int32_t* topk_ids, int M, int topk, int num_experts,
                                  int block_size, int32_t* sorted_ids, int32_t* expert_ids,
                                  int32_t* num_tokens_post_padded, int32_t* expert_offsets,
                                  moe_stream_t stream);

/*
 * Router gating: each token's experts and routing weights from its router
 * logits.  The pages take topk_ids / topk_weights as the router's given
 * output; the two gating functions here are those of the model
 * configurations the layer serves (softmax top-k as in Qwen3-MoE, and the
 * DeepSeek-V3/R1 sigmoid router with group-limited selection).  Equal scores
 * go to the lower expert index.
 *
 *  MOE_GATE_SOFTMAX: p = softmax(logits[t]); topk_ids[t] = the topk largest p
 *    in descending order; topk_weights[t,j] = p_j / (sum of the chosen p).
 *    Ranking p is ranking the logits, so only the chosen terms are formed:
 *    w_j = exp(l_j - l_max) / sum over chosen of exp(l_i - l_max).
 *  MOE_GATE_SIGMOID_GROUPED: s = sigmoid(logits[t]) and b = s + bias (the
 *    bias only ranks).  The E experts form n_group consecutive groups of
 *    E / n_group; a group's score is the sum of its two largest b (its only b
 *    in a group of one); the topk_group best groups are kept and
 *    topk_ids[t] = the topk largest b inside them, descending;
 *    topk_weights[t,j] = s_j / (sum of the chosen s) * routed_scaling.
 * Arithmetic is fp32 (expf, IEEE division); rankings compare fp32 scores, so
 * scores closer than a few fp32 ulps may rank either way.  Whatever the
 * logits (NaN included), every written id lies in [0, E).
 */
#define MOE_GATE_SOFTMAX 0
#define MOE_GATE_SIGMOID_GROUPED 1
typedef struct moe_gate_config {
  int scoring;          /* MOE_GATE_SOFTMAX or MOE_GATE_SIGMOID_GROUPED                      */
  int n_group;          /* SIGMOID_GROUPED: 1..32, divides E.  SOFTMAX: must be 1              */
  int topk_group;       /* SIGMOID_GROUPED: 1..n_group, topk <= topk_group * E / n_group.
                           SOFTMAX: must be 1                                                  */
  float routed_scaling; /* SIGMOID_GROUPED: > 0.  SOFTMAX: must be 1.0                         */
  const float* bias;    /* SIGMOID_GROUPED: fp32 [E] device pointer, or NULL for none.
                           SOFTMAX: must be NULL                                               */
  int shared_expert;    /* 0 or 1: also write column topk of every row as (id E, weight 1.0)   */
} moe_gate_config_t;

/*
 *   logits        fp32 [M, E]                     router logits
 *   topk_ids      int32 [M, topk + shared_expert] out
 *   topk_weights  fp32  [M, topk + shared_expert] out
 * 1 <= topk <= min(E, 32), E <= MOE_MAX_EXPERTS, M >= 0.  One warp ranks one
 * token.  Launched with programmatic dependent launch: the kernel waits for
 * the stream's previous kernel before it reads or writes anything, and the
 * next kernel of the library may be scheduled while it runs.
 */
moe_status_t moe_gate_topk(const float* logits, int M, int E, int topk, const moe_gate_config_t* gate,
                           int32_t* topk_ids, float* topk_weights, moe_stream_t stream);

/*
 * Dynamic per-row INT8 quantisation of bf16 activations (the DA8W8
 * activation side; SGLang CPU backend write-up, section "(3) FusedMoE", the
 * dynamic-quant fusion paragraph):
 *   scale[r] = max_c |x[r,c]| / 127 (fp32; 1 for an all-zero row)
 *   q[r,c]   = round-half-even(x[r,c] / scale[r]) (IEEE fp32 division),
 *              clamped to [-127, 127]
 *   x bf16 [M, H] -> q int8 [M, H], scale fp32 [M].  M >= 0, 1 <= H.
 * The fused INT8 layer applies exactly this function to its input rows.
 */
moe_status_t moe_quant_act_int8(const void* x_bf16, int M, int H, int8_t* q, float* scale,
                                moe_stream_t stream);

/*
 * Dynamic FP8 quantisation of bf16 activations in groups of 1 x 128 (the
 * activation side of MOE_ACT_FP8_1X128).  The pages keep FP8-weight
 * activations in BF16 (Xeon 6 / SGLang blog, section "FP8 inference"); this
 * is the FP8 x FP8 form of the grouped GEMMs named in the news rewrite of the
 * LMSYS large-scale-EP blog (section "DeepGEMM integration"), with the group
 * along H matching the weights' 128-wide scale blocks:
 *   scale[r,g] = max over c in [128g, 128g+128) of |x[r,c]| / 448 (fp32; 1 for
 *                an all-zero group)
 *   q[r,c]     = E4M3(x[r,c] / scale[r, c/128]), the division in IEEE fp32,
 *                rounded to nearest even, saturated to +-448
 *   x bf16 [M, H] -> q uint8 E4M3 codes [M, H], scale fp32 [M, H/128].
 * H must be a multiple of 128 (else MOE_ERR_UNSUPPORTED); M >= 0.  x 16-byte
 * aligned, q 4-byte aligned.  The fused layer applies exactly this function
 * to its input rows.
 */
moe_status_t moe_quant_act_fp8(const void* x_bf16, int M, int H, uint8_t* q, float* scale,
                               moe_stream_t stream);

/*
 * Bytes of scratch the fused layer needs for these sizes and flags
 * (weight_kind MOE_WEIGHT_FP8, MOE_WEIGHT_INT8 or MOE_WEIGHT_INT4).  The workspace must be
 * 256-byte aligned.  Returns 0 for invalid or unsupported arguments.
 */
size_t moe_workspace_size(int M, int H, int I, int E, int topk, int weight_kind,
                          unsigned flags);

/*
 * The whole MoE layer with FP8 E4M3 block-scaled weights; activations enter
 * the products at their bf16 values (weight-only FP8, as in the Xeon 6 /
 * SGLang blog, section "FP8 inference", and the SGLang CPU backend
 * write-up, section "(4) FP8 GEMM").
 *
 *   x_bf16        bf16 [M, H]
 *   topk_ids      int32 [M, topk]        ids outside [0, E) contribute 0
 *   topk_weights  fp32 [M, topk]
 *   w13_e4m3      uint8 [E, 2I, H]       rows 0..I-1 gate, I..2I-1 up
 *   w13_scale     fp32 [E, 2I/128, H/128]  W13 = decode(code) * scale of its block
 *   w2_e4m3       uint8 [E, H, I]
 *   w2_scale      fp32 [E, H/128, I/128]
 *   out_bf16      bf16 [M, H]            out[t] = sum_k w[t,k] * y[t,k]
 *   workspace     moe_workspace_size(M, H, I, E, topk, MOE_WEIGHT_FP8, flags)
 *                 bytes of device memory, 256-byte aligned
 * H and I must be multiples of 128; 1 <= topk <= 32; M >= 0 (M == 0 is a
 * no-op).  A shared expert is passed as one more expert with a top-k column
 * of weight 1.0.  The products run on tensor cores with fp16 operands and
 * fp32 accumulation; each 128x128 block scale is applied once per 128-deep
 * partial sum.  Operands keep the range of their source type: the E4M3 to
 * fp16 expansion is exact; each x row is stored as fp16 in a power-of-two
 * frame of its own (its max |x| scaled into [2^14, 2^15), so every bf16 value
 * within 2^-28 of the row's largest is exact); the intermediate h is stored
 * as fp16 in a power-of-two frame per row (values within 2^-21 of the row's
 * largest keep full fp16 precision); on the tcgen05 path the block scales
 * are folded into the fp16 weights relative to a power of two per 128-row
 * block.  The frames are taken back in fp32, so no finite input overflows an
 * fp16 operand.
 * With MOE_ACT_FP8_1X128 in flags, x is quantised as moe_quant_act_fp8 does,
 * and so is each intermediate row h (fp32, per 128 columns of I) of a
 * (token, expert) pair before the down projection; the products are E4M3 x
 * E4M3 on the tensor cores, and every 128-deep partial sum is scaled by its
 * weight block scale times its activation group scale in fp32.
 */
moe_status_t fused_moe_fp8(const void* x_bf16, const int32_t* topk_ids, const float* topk_weights,
                           const void* w13_e4m3, const float* w13_scale, const void* w2_e4m3,
                           const float* w2_scale, int M, int H, int I, int E, int topk,
                           unsigned flags, void* out_bf16, void* workspace,
                           size_t workspace_bytes, moe_stream_t stream);

/*
 * The whole MoE layer with INT8 per-output-channel weights and dynamic
 * per-row INT8 activations (DA8W8; SGLang CPU backend write-up, section
 * "(3) FusedMoE"): x rows are quantised as moe_quant_act_int8 does, and each
 * intermediate row h of a (token, expert) pair is quantised the same way
 * before the down projection.
 *
 *   w13        int8 [E, 2I, H],  w13_scale fp32 [E, 2I]
 *   w2         int8 [E, H, I],   w2_scale  fp32 [E, H]
 * other arguments as for fused_moe_fp8.  H and I must be multiples of 128.
 */
moe_status_t fused_moe_int8(const void* x_bf16, const int32_t* topk_ids, const float* topk_weights,
                            const int8_t* w13, const float* w13_scale, const int8_t* w2,
                            const float* w2_scale, int M, int H, int I, int E, int topk,
                            unsigned flags, void* out_bf16, void* workspace,
                            size_t workspace_bytes, moe_stream_t stream);

/*
 * The whole MoE layer with group-wise INT4 weights (W4A16).  The pages name
 * INT4 as the quantised alternative to native FP8 (SGLang CPU backend
 * write-up, closing section; OSDI'26 local-MoE summary, the INT4 decode
 * baseline of its evaluation) but fix no layout; this one is:
 *
 *   w13        uint8 [E, 2I, H/2]   two's-complement int4 codes in [-8, 7],
 *                                   column 2j in the low nibble of byte j,
 *                                   column 2j+1 in its high nibble
 *   w13_scale  fp32 [E, 2I, H/128]  W13[e,n,k] = q * w13_scale[e, n, k/128]
 *   w2         uint8 [E, H, I/2],   w2_scale fp32 [E, H, I/128]
 * other arguments as for fused_moe_fp8.  Activations enter the products at
 * their bf16 values (in fp16 power-of-two frames, as on the FP8 weight-only
 * path) and each 128-deep partial sum is scaled by its row's group scale in
 * fp32.
 * H and I must be multiples of 128.  Paths as for fused_moe_fp8 (the
 * weight-streaming kernels up to MOE_MAX_DECODE_TOKENS tokens, the tcgen05
 * grouped GEMMs above; MOE_PATH_DECODE is accepted at any M for INT4);
 * MOE_ACT_FP8_1X128 is MOE_ERR_INVALID_ARG.  Workspace:
 * moe_workspace_size(..., MOE_WEIGHT_INT4, flags).
 */
moe_status_t fused_moe_int4(const void* x_bf16, const int32_t* topk_ids, const float* topk_weights,
                            const uint8_t* w13, const float* w13_scale, const uint8_t* w2,
                            const float* w2_scale, int M, int H, int I, int E, int topk,
                            unsigned flags, void* out_bf16, void* workspace,
                            size_t workspace_bytes, moe_stream_t stream);

/*
 * The experts of the layer on the masked, fixed-capacity layout of
 * expert-parallel low-latency dispatch (the "masked" grouped GEMM of the
 * DeepGEMM integration in the news rewrite of the LMSYS large-scale-EP blog,
 * section "DeepGEMM集成"): tokens arrive already grouped by expert, each expert
 * holding up to `cap` rows, and only a device-side count says how many are real.
 * Nothing in the call depends on host knowledge of the counts, so it can be
 * captured in a CUDA graph and replayed with new counts.
 *
 *   x_bf16     bf16 [E, cap, H]   row (e, i) is the i-th token sent to expert e
 *   masked_m   int32 [E]          rows held by expert e (device memory, read by
 *                                 the kernels); values are clamped to [0, cap]
 *   w13, w2 (+ scales)            as for fused_moe_fp8 (weight_kind
 *                                 MOE_WEIGHT_FP8) or fused_moe_int4
 *                                 (MOE_WEIGHT_INT4); MOE_WEIGHT_INT8 is
 *                                 MOE_ERR_UNSUPPORTED
 *   out_bf16   bf16 [E, cap, H]   out[e, i] = W2_e (SiLU(W1_e x) * (W3_e x)) for
 *                                 i < masked_m[e]; rows past the count are left
 *                                 untouched.  No routing weight is applied (the
 *                                 combine of the dispatch applies it).
 *   workspace  moe_workspace_size_masked(E, cap, H, I, weight_kind) bytes,
 *              256-byte aligned
 * x, w13 and w2 16-byte aligned; out_bf16 2-byte aligned, 16-byte aligned
 * with MOE_PATH_PREFILL (else MOE_ERR_INVALID_ARG).  H and I multiples of 128, E <= MOE_MAX_EXPERTS, cap >= 1.  The products
 * use the arithmetic of the weight kind's layer entry point.  Since the counts
 * are on the device the caller picks the kernels: MOE_PATH_AUTO or
 * MOE_PATH_DECODE runs the weight-streaming kernels (best for a few rows per
 * expert); MOE_PATH_PREFILL runs the tcgen05 kernels (best for many rows per
 * expert).  Every kernel of the call is enqueued on `stream`.
 */
size_t moe_workspace_size_masked(int E, int cap, int H, int I, int weight_kind);
moe_status_t fused_moe_masked(int weight_kind, const void* x_bf16, const int32_t* masked_m, const void* w13,
                              const float* w13_scale, const void* w2, const float* w2_scale, int E, int cap,
                              int H, int I, unsigned flags, void* out_bf16, void* workspace,
                              size_t workspace_bytes, moe_stream_t stream);

/*
 * The whole layer from router logits: moe_gate_topk, then fused_moe_fp8
 * (weight_kind MOE_WEIGHT_FP8), fused_moe_int8 (MOE_WEIGHT_INT8) or
 * fused_moe_int4 (MOE_WEIGHT_INT4) on its result, with no host step between
 * them.
 *
 *   router_logits  fp32 [M, E]   E = routed experts
 *   gate           gating function and options, as for moe_gate_topk
 *   w13, w2 (+ scales)  hold E + gate->shared_expert experts; a shared
 *                  expert is the last one
 *   topk_ids, topk_weights  out, [M, topk + gate->shared_expert], as
 *                  moe_gate_topk writes them (the routing the layer used)
 *   workspace      moe_workspace_size(M, H, I, E + shared_expert,
 *                  topk + shared_expert, weight_kind, flags) bytes
 * other arguments as for fused_moe_fp8 / _int8 / _int4 (flags must suit the
 * weight kind).  When M <= MOE_GATE_INLINE_TOKENS and E <= 256 the ranking
 * runs inside the layer's first kernel, ahead of the routing alignment (one
 * launch fewer); otherwise it is one more launch, chained to the layer by
 * programmatic dependent launch.  Results are the same either way.
 */
#define MOE_GATE_INLINE_TOKENS 64
moe_status_t fused_moe_gated(int weight_kind, const void* x_bf16, const float* router_logits,
                             const moe_gate_config_t* gate, const void* w13, const float* w13_scale,
                             const void* w2, const float* w2_scale, int M, int H, int I, int E, int topk,
                             unsigned flags, int32_t* topk_ids, float* topk_weights, void* out_bf16,
                             void* workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * fused_moe_fp8 for callers that cannot allocate device memory.  The pages
 * have no counterpart of this entry point; it exists for callers that hold
 * only raw input and output pointers and may not call a device allocator (a
 * plugin whose host framework owns all device memory, a C caller without an
 * allocator, or a loop that must not pay for cudaMalloc / cudaFree).
 *
 * Same arguments, layouts and results as fused_moe_fp8, without the
 * workspace: the scratch is a static device buffer of
 * MOE_STATIC_SCRATCH_BYTES inside the library.  Each device on which it runs
 * holds that buffer from its first call until the process exits.
 *  - The first call on a device looks the buffer's address up
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.  After a device reset the next call on that
 *    device looks it up again (a new CUDA context), so it too must come
 *    before any capture.
 *  - Invalid arguments return what fused_moe_fp8 returns for them.  Valid
 *    sizes whose moe_workspace_size(..., MOE_WEIGHT_FP8, flags) exceeds
 *    MOE_STATIC_SCRATCH_BYTES return MOE_ERR_UNSUPPORTED with a message that
 *    names the limit; nothing is launched.
 *  - Nothing is allocated or freed.  All calls share the buffer, which keeps
 *    the last call's contents; the kernels clear what must start at zero.
 *    Calls that overlap on the GPU race on it: serialise them.
 *  - Its device status words (ids out of range, a bounded wait that gave up)
 *    are read with moe_read_static_scratch_status.
 */
#define MOE_STATIC_SCRATCH_BYTES (16u << 20)
moe_status_t fused_moe_fp8_static_scratch(const void* x_bf16, const int32_t* topk_ids,
                                          const float* topk_weights, const void* w13_e4m3,
                                          const float* w13_scale, const void* w2_e4m3,
                                          const float* w2_scale, int M, int H, int I, int E, int topk,
                                          unsigned flags, void* out_bf16, moe_stream_t stream);

/*
 * moe_read_status for the static buffer of fused_moe_fp8_static_scratch on
 * the current device: waits for `stream`, then copies the status words of
 * the last call that ran there (see moe_read_status).  The pages have no
 * counterpart of this function either.
 */
moe_status_t moe_read_static_scratch_status(int32_t status_out[2], moe_stream_t stream);

/*
 * Waits for `stream`, then copies the workspace's status words to the host:
 *   status_out[0] = number of topk_ids entries outside [0, E) seen by the
 *                   last fused call on this workspace
 *   status_out[1] = bit set of device conditions (1 = a bounded wait gave up)
 * Returns MOE_ERR_BAD_IDS / MOE_ERR_TIMEOUT when they are non-zero.
 */
moe_status_t moe_read_status(const void* workspace, int32_t status_out[2], moe_stream_t stream);

/*
 * The routing alignment (step 1) that the last routed fused call on
 * `workspace` computed -- fused_moe_fp8, fused_moe_int8, fused_moe_int4 or
 * fused_moe_gated, called with these same M, H, I, E (all stored experts),
 * topk (all columns) and flags.  Outputs are as moe_align_block_size defines
 * them, for the block size the layer chose for its path (8 on the
 * weight-streaming kernels, 16 on the tcgen05 ones):
 *   block_size      HOST int out (may be NULL)
 *   sorted_ids      device int32 [moe_align_max_padded(M, topk, E, *block_size)]
 *   expert_ids      device int32 [that / *block_size]
 *   num_tokens_post_padded  device int32 [1]
 *   expert_offsets  device int32 [E + 1]
 * Any output pointer may be NULL (block_size alone answers the sizing
 * question).  The copies are stream-ordered device-to-device copies after
 * the layer's kernels; nothing synchronises.  The masked layout has no
 * alignment and is not covered.  Bad sizes give MOE_ERR_INVALID_ARG.
 */
moe_status_t moe_read_routing(const void* workspace, int M, int H, int I, int E, int topk, int weight_kind,
                              unsigned flags, int* block_size, int32_t* sorted_ids, int32_t* expert_ids,
                              int32_t* num_tokens_post_padded, int32_t* expert_offsets, moe_stream_t stream);

/*
 * Self-test of the failure path of the bounded device waits.  Launches one
 * small kernel whose waits can never complete: one gives up after
 * limit_cycles SM clocks (1000 <= limit_cycles <= 2^31, about a second at
 * most), sets bit 0 of the workspace's status words and the shared abort
 * flag; the other leaves through that flag, as every role of a GEMM kernel
 * does when one of them times out.  *gave_up (device int32) receives the
 * number of waits that gave up (2).  moe_read_status(workspace) then returns
 * MOE_ERR_TIMEOUT.  Only the status words (the first 8 bytes of any
 * workspace, at least 256 bytes, 256-byte aligned) and *gave_up are written;
 * nothing faults and the context stays usable.
 */
moe_status_t moe_selftest_wait_timeout(void* workspace, long long limit_cycles, int32_t* gave_up,
                                       moe_stream_t stream);

/*
 * Per-kernel timing of fused calls on the calling host thread (a profiling
 * aid; it changes nothing the layer computes).
 *
 * moe_profile_enable(max_calls): with max_calls > 0, creates CUDA timing
 * events on the current device for up to max_calls later fused calls and
 * starts recording: every such call records one event before its first
 * kernel and one after each kernel, on its own stream.  max_calls == 0 stops
 * recording and releases the events.  Calls past the limit are not recorded.
 *
 * moe_profile_read(stage_ms, stage_names, max_stages, n_stages, n_calls):
 * waits for the recorded events, writes per kernel ("stage") the summed
 * milliseconds over all recorded calls (stage order = launch order; all
 * recorded calls must have taken the same path) and the stage's name, then
 * forgets the recorded calls (recording continues).
 */
moe_status_t moe_profile_enable(int max_calls);
moe_status_t moe_profile_read(float* stage_ms, const char** stage_names, int max_stages, int* n_stages,
                              int* n_calls);

/* Static English text for a status code. */
const char* moe_status_string(moe_status_t status);

/* Text of the last error raised on the calling host thread ("" if none). */
const char* moe_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* GBMOE_H */
