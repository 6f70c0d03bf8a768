/*
 * moe.h -- C ABI of the GB300 (sm_103a) MoE layer forward.
 *
 * The layer computes y = sum_{i in TopK(x)} g_i(x) * E_i(x) (+ an optional
 * shared expert), each E_i a SwiGLU FFN ("TensorRT-LLM 源码完全拆解(十三): MoE 层前向执行",
 * section "MoE 在推理侧到底特殊在哪里"), in five steps:
 *
 *   1. moe_route     router logits -> (token_selected_experts, token_final_scales)
 *   2. moe_permute   rows of x gathered into contiguous per-expert blocks
 *   3. moe_fc1       grouped GEMM x_perm . w13[e]^T with SwiGLU fused -> h
 *   4. moe_fc2       grouped GEMM h . w2[e]^T -> out_perm
 *      (moe_fc1_fc2  steps 3 and 4 in one persistent launch, as moe_forward runs them)
 *   5. moe_finalize  unpermute, apply the routing weights, add the shared expert -> y
 *
 * moe_forward runs steps 2-5. Conventions common to every call:
 *
 *  - Pointers named "device" are CUDA device memory owned by the caller. The
 *    library allocates no device memory; the forward uses the caller's
 *    workspace (size from moe_workspace_bytes).
 *  - `stream` is a cudaStream_t (passed as void*). Work is enqueued on it
 *    only; no call below synchronises except moe_read_device_status and
 *    moe_static_read_device_status.
 *  - bf16 tensors are passed as void* to 2-byte IEEE bfloat16 elements,
 *    row-major, innermost dimension contiguous. Every device pointer must be
 *    16-byte aligned.
 *  - Errors found on the host (bad sizes, NULL or misaligned pointers, a
 *    workspace that is too small) return synchronously and enqueue nothing.
 *    A CUDA launch error returns MOE_ERR_CUDA (text in moe_last_error()).
 *    Errors found on the device (an expert id outside [0, E), a bounded wait
 *    that ran out) set bits in the workspace status word; the offending rows
 *    are skipped. moe_read_device_status reports them.
 *  - T = 0 is a valid no-op.
 *
 * Thread safety: calls may come from several host threads; calls that share
 * a workspace must be ordered on one stream.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 1

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,        /* NULL/misaligned pointer, negative size          */
  MOE_ERR_UNSUPPORTED = 2,        /* shape outside the supported envelope (reason)    */
  MOE_ERR_WORKSPACE_TOO_SMALL = 3,
  MOE_ERR_CUDA = 4,               /* a CUDA runtime call failed                       */
  MOE_ERR_DEVICE_BAD_ID = 5,      /* device saw an expert id outside [0, E)           */
  MOE_ERR_DEVICE_TIMEOUT = 6,     /* a bounded device-side wait ran out               */
  MOE_ERR_NOT_IMPLEMENTED = 7
} moe_status;

/* Routing methods; the values are those of the RoutingMethodType enum on the
 * TensorRT-LLM MoE page (section "路由方法枚举"). */
typedef enum {
  MOE_ROUTE_DEFAULT = 0,           /* softmax over E -> top-k, weights = selected probabilities   */
  MOE_ROUTE_RENORMALIZE = 1,       /* top-k -> softmax over the k selected logits                 */
  MOE_ROUTE_DEEPSEEKV3 = 2,        /* sigmoid, +bias for selection, top-2 per group, top groups,
                                      top-k; weights = unbiased sigmoid / (sum + 1e-20) * rsf    */
  MOE_ROUTE_LLAMA4 = 3,            /* top-k by logit ("Top1"), weights = sigmoid of each selected
                                      logit, not renormalised                                     */
  MOE_ROUTE_RENORMALIZE_NAIVE = 4, /* softmax over E -> top-k -> divide by the selected sum       */
  MOE_ROUTE_MINIMAX2 = 5,          /* sigmoid, +bias for selection, top-k over all E; weights =
                                      unbiased sigmoid / their sum (bias optional, NULL = 0)     */
  MOE_ROUTE_SIGMOID_RENORM = 6,    /* sigmoid -> top-k -> divide by the selected sum              */
  /* vLLM's GroupedTopKRouter (vLLM MoE page, section "GroupedTopKRouter：分组的专家选择"); the
   * values lie outside RoutingMethodType's range (0-8). */
  MOE_ROUTE_GROUPED_TOPK = 16,     /* sigmoid scores; group score = sum of the group's scores;
                                      top topk_group groups; top_k / topk_group experts inside
                                      each; weights = scores / their sum * rsf (see moe_route) */
  MOE_ROUTE_GROUPED_TOPK_SOFTMAX = 17  /* the same with a softmax inside each group: its group
                                      scores are all 1, so the group choice would rest on
                                      tie-breaking alone; always rejected (MOE_REASON_DEGENERATE) */
} moe_route_method;

/* Why moe_can_implement rejected a problem. */
typedef enum {
  MOE_REASON_OK = 0,
  MOE_REASON_T_RANGE = 1,          /* T < 0 or T > 2^24                                   */
  MOE_REASON_E_RANGE = 2,          /* E < 1 or E > 256                                    */
  MOE_REASON_TOPK_RANGE = 3,       /* k < 1 or k > 8                                      */
  MOE_REASON_H_ALIGN = 4,          /* H < 64, H % 64 != 0 or H > 32768                    */
  MOE_REASON_I_ALIGN = 5,          /* I < 64, I % 64 != 0 or I > 65536                    */
  MOE_REASON_SHARED_I_ALIGN = 6,   /* shared_I < 0, shared_I % 64 != 0 or > 65536         */
  MOE_REASON_GROUPS = 7,           /* routing groups invalid (see moe_route)              */
  MOE_REASON_METHOD = 8,           /* unknown routing method                              */
  MOE_REASON_ROWS = 9,             /* T*k (+T shared) permuted rows reach 2^31             */
  MOE_REASON_DEGENERATE = 10       /* a routing whose choice rests on tie-breaking alone   */
} moe_reason;

typedef struct {
  int32_t num_experts;            /* E                                                   */
  int32_t top_k;                  /* k                                                   */
  int32_t method;                 /* moe_route_method                                    */
  int32_t n_group;                /* DeepSeekV3, GROUPED_TOPK: expert groups; else 1      */
  int32_t topk_group;             /* DeepSeekV3, GROUPED_TOPK: groups kept; else 1        */
  float routed_scaling_factor;    /* DeepSeekV3, GROUPED_TOPK: multiplies the weights     */
} moe_route_params;

typedef struct {
  int64_t T;                      /* tokens                                              */
  int32_t H;                      /* hidden size                                         */
  int32_t I;                      /* routed expert intermediate size                     */
  int32_t E;                      /* routed experts                                      */
  int32_t k;                      /* experts per token                                   */
  int32_t shared_I;               /* shared expert intermediate size; 0 = no shared      */
} moe_problem;

/* Byte offsets of the workspace regions (all 1024-byte aligned). */
typedef struct {
  size_t status;      /* int32[4]: device status bits (MOE_DEVICE_FLAG_*)                    */
  size_t counts;      /* int32[G]: rows per group; G = E (+1 with a shared expert)           */
  size_t starts;      /* int32[G]: first permuted row of each group (shared group: T*k)      */
  size_t offsets;     /* int32[E+1]: exclusive scan of the routed counts                     */
  size_t tile_off1;   /* int32[2][G+1]: FC1 offsets per group, CTA-pair list then single-SM  */
  size_t tile_off2;   /* int32[2][G+1]: FC2 offsets per group, CTA-pair list then single-SM  */
  size_t sched;       /* int32[8 + G]: GEMM work-claim/finish counters, then per-group FC1 done  */
  size_t block_hist;  /* int32[nb*E]: per-chunk expert histograms                            */
  size_t perm_src;    /* int32[T*k]: permuted row -> flat index f = t*k + j                  */
  size_t perm_inv;    /* int32[T*k]: flat index -> permuted row (-1 if the id was invalid)   */
  size_t x_perm;      /* bf16[R, H]: gathered rows, R = T*k (+T shared rows)                 */
  size_t h;           /* bf16[R, Ih]: SwiGLU output, Ih = max(I, shared_I)                   */
  size_t out_perm;    /* bf16[R, H]: FC2 output in permuted order                            */
  size_t total;       /* bytes = moe_workspace_bytes()                                       */
  int64_t rows;       /* R                                                                   */
  int32_t groups;     /* G                                                                   */
  int32_t n_chunks;   /* nb                                                                  */
  int32_t h_ld;       /* Ih                                                                  */
  int32_t reserved;
} moe_ws_layout;

#define MOE_DEVICE_FLAG_BAD_ID 1
#define MOE_DEVICE_FLAG_TIMEOUT 2

int32_t moe_abi_version(void);
const char* moe_status_string(moe_status s);
/* Text of the last error seen on the calling host thread ("" if none). */
const char* moe_last_error(void);

/*
 * moe_route -- routing (step 1).
 * Source: TensorRT-LLM MoE page, sections "路由方法枚举" and "DeepSeek-V3 的 noaux_tc:
 * 分组路由的算术" (apply() returns token_selected_experts int32 [T, k] and
 * token_final_scales fp32 [T, k]); vLLM MoE page, section "FusedTopKRouter".
 *   logits  device fp32 [T, E] row-major.
 *   bias    device fp32 [E] e_score_correction_bias (DeepSeekV3), or NULL (= zeros).
 *   ids     device int32 [T, k] out: selected experts, by descending selection key,
 *           ties to the lower expert index. The key is the fp32 logit for the softmax
 *           and sigmoid methods; for DeepSeekV3 it is fl32(fl32(sigmoid_fp64(l)) + b).
 *   scales  device fp32 [T, k] out: routing weights (computed in fp64, rounded once).
 * Envelope (the fused-routing limits of the TensorRT-LLM page, section "融合算子与回退
 * 阈值"): 1 <= k <= 8, k <= E <= 256; DeepSeekV3 also E % n_group == 0, n_group <= 32,
 * 2 <= E/n_group <= 32, 1 <= topk_group <= n_group, k <= topk_group*E/n_group <= 256.
 * Outside it: MOE_ERR_UNSUPPORTED, nothing enqueued (there is no fallback).
 * Non-finite logits count as -inf for selection and in the normalisers.
 * MOE_ROUTE_GROUPED_TOPK (vLLM MoE page, section "GroupedTopKRouter"): score
 * s = sigmoid_fp64(l), key fl32(s); a group's score is the sum of its keys added in fp32
 * in expert order; the topk_group best groups (ties to the lower group index), then the
 * k / topk_group best keys inside each (ties to the lower index); slots by descending key;
 * weights s / sum(s) * routed_scaling_factor. Needs E % n_group == 0, n_group <= 32,
 * 1 <= topk_group <= n_group, k % topk_group == 0, k / topk_group <= E / n_group; `bias`
 * must be NULL (MOE_ERR_INVALID_ARG otherwise).
 */
moe_status moe_route(const float* logits, int64_t T, const float* bias, const moe_route_params* p,
                     int32_t* ids, float* scales, void* stream);

/* Pure check of a problem against the supported envelope; never touches the device.
 * Returns MOE_OK or MOE_ERR_UNSUPPORTED / MOE_ERR_INVALID_ARG; *reason (may be NULL)
 * receives a moe_reason. */
moe_status moe_can_implement(const moe_problem* p, int32_t* reason);

/* Workspace bytes the forward needs for this problem (0 if it is unsupported). */
size_t moe_workspace_bytes(const moe_problem* p);
/* Fills *out with the workspace layout for this problem. */
moe_status moe_workspace_layout(const moe_problem* p, moe_ws_layout* out);

/*
 * moe_forward -- steps 2-5 on one stream.
 * Source: vLLM MoE page, section "Router 的子类选择逻辑"/"量化与 MoE Kernel 选择" (the
 * modular path forward_modular(x, topk_weights, topk_ids)) and section "专家权重如何存储"
 * (w13 = gate and up merged [E, 2I, H], w2 = down [E, H, I]); TensorRT-LLM MoE page,
 * layer-structure figure (routed path + shared expert summed).
 *   x        device bf16 [T, H]
 *   ids      device int32 [T, k] (any values; ids outside [0, E) are skipped and flagged;
 *            repeated ids in a row are independent rows)
 *   scales   device fp32 [T, k]
 *   w13      device bf16 [E, 2I, H]: rows [0, I) gate (w1), rows [I, 2I) up (w3)
 *   w2       device bf16 [E, H, I]
 *   w13_s    device bf16 [2*shared_I, H] or NULL when shared_I == 0
 *   w2_s     device bf16 [H, shared_I]  or NULL when shared_I == 0
 *   y        device bf16 [T, H] out: sum_j scales[t,j] * E_ids[t,j](x[t]) + shared(x[t])
 *   workspace device, >= moe_workspace_bytes(p) bytes, 1024-byte aligned.
 * Accumulation is fp32; h and out_perm are rounded to bf16; y is rounded once to bf16.
 */
moe_status moe_forward(const moe_problem* p, const void* x, const int32_t* ids, const float* scales,
                       const void* w13, const void* w2, const void* w13_s, const void* w2_s,
                       void* y, void* workspace, size_t ws_bytes, void* stream);

/*
 * moe_forward_static -- moe_forward without a caller workspace. The pages have no
 * counterpart; this entry point exists for callers that cannot allocate device memory:
 * plugins hosted by an inference engine that owns every device allocation, and
 * latency-critical loops that must not call cudaMalloc (it can synchronise the whole
 * device). The scratch the forward needs lives in a fixed array inside this library,
 * MOE_STATIC_SCRATCH_BYTES bytes on every GPU that loads it, held until the process
 * exits. Arguments are those of moe_forward minus the workspace.
 *  - Problems whose workspace (moe_workspace_bytes) exceeds MOE_STATIC_SCRATCH_BYTES are
 *    rejected with MOE_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
 *  - The first call on a device looks up the array's device address (once per device,
 *    with that device current); make that first call before any stream capture.
 *  - Every call on a device shares the one array and it keeps the previous call's
 *    contents (the call clears what must start at zero itself). Calls whose work
 *    overlaps on the GPU race: order them on one stream.
 *  - Device-detected errors (ids outside [0, E), a bounded wait that ran out) skip rows
 *    as in moe_forward and set the status word inside the array, which each call clears
 *    when it starts; moe_static_read_device_status reads it back.
 * It allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 */
#define MOE_STATIC_SCRATCH_BYTES ((size_t)32 << 20)
moe_status moe_forward_static(const moe_problem* p, const void* x, const int32_t* ids,
                              const float* scales, const void* w13, const void* w2,
                              const void* w13_s, const void* w2_s, void* y, void* stream);

/* The status word of moe_forward_static on the current device: synchronises `stream`
 * (the stream the forward ran on), reads and clears the word inside the library's
 * scratch array. *flags (may be NULL) receives the MOE_DEVICE_FLAG_* bits. Returns
 * MOE_ERR_DEVICE_BAD_ID or MOE_ERR_DEVICE_TIMEOUT when a bit is set, else MOE_OK;
 * MOE_ERR_CUDA if the copy or the device lookup fails. Like the forward, it allocates
 * nothing; the word is shared by every caller of moe_forward_static on the device. */
moe_status moe_static_read_device_status(void* stream, int32_t* flags);

/* Router gate (vLLM MoE page, section "Gate 计算与 FSE"): router logits = x . wg^T with
 * fp32 accumulation, one GEMM for the routed experts' gate and, with n_shared = 1, the
 * fused shared-expert gate (FSE: wg is [E + 1, H], its last row the shared expert's gate).
 *   x              device bf16 [T, H]
 *   wg             device bf16 [E + n_shared, H]
 *   routed_logits  device fp32 [T, E]: the logits moe_route takes
 *   shared_logits  device fp32 [T] when n_shared = 1 (moe_forward_partial's shared_gate),
 *                  else ignored (may be NULL)
 * Requires H % 64 == 0 (64..32768), 1 <= E <= 256, n_shared in {0, 1}; 16-byte aligned
 * pointers. Deterministic: partial sums over K are added in a fixed order. */
moe_status moe_gate(const void* x, const void* wg, int64_t T, int32_t H, int32_t E,
                    int32_t n_shared, float* routed_logits, float* shared_logits, void* stream);

/* Router gate and routing in one launch (vLLM MoE page, section "Gate 计算与 FSE": the gate
 * GEMM that produces router_logits; TensorRT-LLM MoE page, layer-structure figure: fc_gate
 * ahead of routing): moe_gate, then moe_route on its logits. After the gate's fixed-order
 * reduction, the CTA that holds a token's complete row of routed logits routes the token
 * itself, so the logits need not travel through HBM to a second launch.
 *   x, wg, T, H, n_shared  as for moe_gate, with E = p->num_experts
 *   bias, p                as for moe_route (every method and envelope of moe_route)
 *   ids, scales            device int32 / fp32 [T, k] out, as moe_route writes them
 *   routed_logits          device fp32 [T, E] out, or NULL (then not written)
 *   shared_logits          device fp32 [T] out when n_shared = 1, else ignored (may be NULL)
 * The logits equal moe_gate's and the ids and scales equal moe_route's on those logits, bit
 * for bit. Errors: those of moe_gate and of moe_route, checked on the host before anything
 * is enqueued. */
moe_status moe_gate_route(const void* x, const void* wg, int64_t T, int32_t H, int32_t n_shared,
                          const float* bias, const moe_route_params* p, int32_t* ids,
                          float* scales, float* routed_logits, float* shared_logits,
                          void* stream);

/* moe_forward restricted to the experts [e_lo, e_hi) of this call: the expert-parallel
 * seam of the TensorRT-LLM MoE page, section on supports_finalize_before_combine ("finalize
 * before combine": the top-k weighted sum taken on a rank's own rows, slots of other
 * ranks' experts contributing exactly 0, so that the combine is an unweighted row sum).
 *   y[t] = sum over j with ids[t,j] in [e_lo, e_hi) of scales[t,j] * E_{ids[t,j]}(x[t])
 *          (+ shared(x[t]) when p->shared_I > 0)
 * The y of calls over a partition of [0, E) (the shared expert in exactly one of them) add
 * up to moe_forward's y. w13 / w2 hold the local experts only: [e_hi - e_lo, 2I, H] and
 * [e_hi - e_lo, H, I], expert g at plane g - e_lo. Requires 0 <= e_lo < e_hi <= E; ids in
 * [0, E) outside the range are not errors. shared_gate: device fp32 [T] logits of the
 * shared expert's gate (vLLM MoE page, "Gate 计算与 FSE": the shared expert's activation,
 * a sigmoid), so that it enters with weight sigmoid(shared_gate[t]); NULL = weight 1.
 * moe_forward is this call with [0, E) and no shared gate. */
moe_status moe_forward_partial(const moe_problem* p, int32_t e_lo, int32_t e_hi, const void* x,
                               const int32_t* ids, const float* scales, const void* w13,
                               const void* w2, const void* w13_s, const void* w2_s,
                               const float* shared_gate, void* y, void* workspace,
                               size_t ws_bytes, void* stream);

/* Step entry points (the kernels moe_forward runs, one at a time). Each takes the
 * same workspace; later steps read what earlier ones wrote into it. */

/* Step 2 (Dense GEMM -> GroupedGEMM article, sections 2.1-2.2: per-expert contiguous
 * blocks and an offset array). Clears the status word, then writes counts, starts,
 * offsets, the FC1/FC2 tile lists, perm_src, perm_inv and x_perm. Rows of an expert
 * keep ascending flat index f = t*k + j. */
moe_status moe_permute(const moe_problem* p, const void* x, const int32_t* ids,
                       void* workspace, size_t ws_bytes, void* stream);
/* Step 3: h[r, :] = silu(x_perm[r] . w13[e][0:I]^T) * (x_perm[r] . w13[e][I:2I]^T). */
moe_status moe_fc1(const moe_problem* p, const void* w13, const void* w13_s, void* workspace,
                   size_t ws_bytes, void* stream);
/* Step 4: out_perm[r, :] = h[r] . w2[e]^T. */
moe_status moe_fc2(const moe_problem* p, const void* w2, const void* w2_s, void* workspace,
                   size_t ws_bytes, void* stream);
/* Steps 3 and 4 as moe_forward runs them: one persistent launch whose work list holds
 * FC1's tiles, then FC2's; an FC2 tile starts once every FC1 tile of its expert has
 * stored its h rows (a per-expert completion counter in the workspace, bounded wait).
 * Same results, bit for bit, as moe_fc1 followed by moe_fc2. Call it after moe_permute on
 * the same workspace: that step zeroes the counters it uses. */
moe_status moe_fc1_fc2(const moe_problem* p, const void* w13, const void* w13_s, const void* w2,
                       const void* w2_s, void* workspace, size_t ws_bytes, void* stream);
/* Step 5 (TensorRT-LLM MoE page: routing weights applied after FC2; finalize = top-k
 * weighted row sum): y[t] = sum_j scales[t,j] * out_perm[perm_inv[t*k+j]] (+ shared row). */
moe_status moe_finalize(const moe_problem* p, const float* scales, void* y, void* workspace,
                        size_t ws_bytes, void* stream);

/* Synchronises `stream`, reads and clears the workspace status word. *flags (may be
 * NULL) receives the MOE_DEVICE_FLAG_* bits. Returns MOE_ERR_DEVICE_BAD_ID or
 * MOE_ERR_DEVICE_TIMEOUT when a bit is set, else MOE_OK. */
moe_status moe_read_device_status(void* workspace, void* stream, int32_t* flags);

/* Self-test of the device failure path, with no fault and no hang: one kernel (one CTA)
 * whose two pipeline roles wait on mbarriers that nothing arrives on, with the same
 * bounded wait as every pipelined kernel here (2 s of wall clock). The producer's wait
 * runs out, sets MOE_DEVICE_FLAG_TIMEOUT in the workspace status word and raises the
 * abort flag; the consumer, which started waiting 1 s later, leaves through that flag
 * and sets status word 1 to 1 when it left before its own limit. `workspace`: any
 * workspace of this library (16-byte aligned; only its first 16 bytes are touched, and
 * words 0-1 are cleared first). Enqueued on `stream`; returns at once. The timeout then
 * reads back through moe_read_device_status, and the context stays usable. Errors:
 * MOE_ERR_INVALID_ARG (NULL or misaligned workspace), MOE_ERR_CUDA (launch). */
moe_status moe_selftest_wait(void* workspace, void* stream);

/* Round-to-nearest-even conversion of n fp32 values to bf16 (device in/out). */
moe_status moe_cast_f32_to_bf16(const float* in, void* out, int64_t n, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
