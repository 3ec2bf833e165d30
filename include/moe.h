/*
 * moe.h -- C ABI of a single-GPU Mixture-of-Experts SwiGLU FFN layer forward (sm_103a).
 *
 * The layer (source pages, by title and section):
 *   router   l = W_r x, W_r [E, d]            "DeepSeek-V4 MoE source analysis (SGLang)", sec. 二
 *                                             (MoEGate weight [n_routed_experts, hidden_size])
 *   scores   softmax | sigmoid | sqrt(softplus) "MoE compute and communication", sec. 二.2;
 *                                             "DeepSeek-V4 MoE", eq. dsv4-moe-softplus
 *   select   top-k of (score + bias); optional group-limited top-k (sum of each group's top
 *            group_topk keys, keep topk_groups groups)  "MoE compute and communication",
 *            sec. 五.3 and 七.3; "DeepSeek-V4 MoE", sec. "V3 的节点路由约束"
 *            or HashTopK ids = tid2eid[token_id]    SGLang analysis, sec. 二 (HashTopK)
 *   weights  g_i = s_i / sum_{TopK} s_j (unbiased s); softmax of the k logits for
 *            MOE_SCORE_SOFTMAX_TOPK               "Mixture of Experts: router, token dispatch,
 *                                                 grouped GEMM", sec. "Router 的选择过程"
 *   dispatch expert-major rows, tokens_per_expert  same page, sec. "Token Dispatch"
 *   experts  FFN_e(x) = W2_e (SiLU(W1_e x) * W3_e x), gate/up fused as w13
 *                                                 SGLang analysis, sec. 四
 *   combine  y_t = sum_j g_{t,j} FFN_{e_j}(x_t) + FFN_shared(x_t)
 *                                                 "MoE compute and communication", sec. 二.2;
 *                                                 router page, sec. "Token Combine"
 *
 * Conventions (every entry point):
 *   - Tensors are row-major and contiguous.  Unless stated, pointers are DEVICE pointers on
 *     the current CUDA device, owned by the caller, and must be 16-byte aligned.
 *       x, out     [T, d]           bf16 (moe_bf16 = raw bf16 bits)
 *       w_r        [E, d]           bf16
 *       w13        [E, 2*d_ff, d]   bf16; rows 0..d_ff-1 of an expert = gate (W1),
 *                                   rows d_ff..2*d_ff-1 = up (W3)
 *       w2         [E, d, d_ff]     bf16 (W2, down projection)
 *       w13_sh     [2*d_ff, d], w2_sh [d, d_ff]   bf16, shared expert (n_shared = 1)
 *       bias       [E]              fp32 selection bias (NULL = none)
 *       token_ids  [T]              int32 (hash routing only)
 *       topk_ids   [T, k] int32, topk_w [T, k] fp32
 *   - All work is enqueued on `stream` (NULL = legacy default stream); calls return without
 *     waiting for the GPU.  The library never allocates device memory: scratch lives in the
 *     caller's workspace `ws` of at least moe_workspace_bytes(plan, T) bytes (256-byte
 *     aligned).  A plan may be used from one host thread at a time, one stream at a time;
 *     two calls that share a workspace must not overlap on the GPU.
 *   - Argument and shape errors are returned synchronously before anything is enqueued.
 *     Launch failures return MOE_ERR_CUDA.  Bad device DATA (token id outside [0, vocab),
 *     tid2eid entry or topk id outside [0, E)) is clamped into range, computed, and flagged
 *     in the workspace error word; moe_check_status() reports it as MOE_ERR_DEVICE_INPUT.
 *     A kernel whose internal pipeline wait exceeds ~2 s stops, flags MOE_ERR_TIMEOUT in the
 *     same word and returns (no GPU trap).  A library built with MOE_DEBUG_BOUNDS=1 also checks
 *     the internal row indices of the dispatch, the grouped GEMMs' stores and the combine;
 *     a failed check skips that access and is reported as MOE_ERR_INTERNAL.
 *   - T = 0 is valid and enqueues nothing.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */
typedef struct CUevent_st* moe_event_t;   /* same type as cudaEvent_t  */
typedef uint16_t moe_bf16;                /* raw bfloat16 bits          */
typedef struct moe_plan moe_plan;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* NULL pointer, bad size, T > max_tokens, bad config        */
  MOE_ERR_UNSUPPORTED = 2,  /* valid but outside the library's limits (see moe_config) */
  MOE_ERR_ALIGNMENT = 3,    /* a pointer is not 16-byte aligned (workspace: 256-byte)    */
  MOE_ERR_WORKSPACE = 4,    /* ws_bytes < moe_workspace_bytes(plan, T)                    */
  MOE_ERR_CUDA = 5,         /* a CUDA runtime/driver call or a launch failed             */
  MOE_ERR_DEVICE_INPUT = 6, /* device data out of range (clamped); from moe_check_status */
  MOE_ERR_TIMEOUT = 7,      /* a kernel pipeline wait timed out; from moe_check_status   */
  MOE_ERR_INTERNAL = 8      /* an internal index check failed (library built with
                               MOE_DEBUG_BOUNDS=1 only); from moe_check_status           */
} moe_status;

typedef enum {
  MOE_SCORE_SOFTMAX_TOPK = 0, /* select top-k on logits (+bias); weights = softmax of the
                                 k selected logits (router page, "Router 的选择过程")        */
  MOE_SCORE_SOFTMAX = 1,      /* p = softmax over all E; select top-k of p (+bias);
                                 weights = p renormalised over the k (Mixtral)              */
  MOE_SCORE_SIGMOID = 2,      /* s = 1/(1+e^-l) (DeepSeek-V3)                               */
  MOE_SCORE_SQRT_SOFTPLUS = 3 /* s = sqrt(ln(1+e^l)) (DeepSeek-V4)                          */
} moe_score;

/* Layer configuration.  Limits of the library: d and d_ff multiples of 64, 1 <= E <= 512,
 * 1 <= top_k <= 8 and top_k <= E, n_shared in {0,1} (the shared expert has d_ff rows),
 * n_groups in {0} U [1, 32] with E % n_groups == 0, max_tokens <= 2^20. */
typedef struct {
  int32_t d;            /* hidden size                                                    */
  int32_t d_ff;         /* expert intermediate size                                       */
  int32_t n_experts;    /* E, routed experts                                              */
  int32_t top_k;        /* k                                                              */
  int32_t n_shared;     /* 0 or 1 always-on shared expert, added with weight 1            */
  int32_t max_tokens;   /* upper bound on T for every call with this plan                 */
  int32_t score;        /* moe_score                                                      */
  int32_t n_groups;     /* 0 = plain top-k; else group-limited over n_groups contiguous    */
  int32_t topk_groups;  /*   groups of E/n_groups experts: keep topk_groups groups ranked  */
  int32_t group_topk;   /*   by the fp32 sum of their group_topk largest selection keys    */
  const int32_t* tid2eid; /* device [vocab, top_k]; non-NULL selects HashTopK routing:
                             ids = tid2eid[token_id] in table order, bias ignored, weights
                             from the unbiased scores of those experts' logits.  Owned by
                             the caller; must stay valid while the plan is used.           */
  int32_t vocab;        /* rows of tid2eid (hash routing only)                            */
} moe_config;

/* Validate `cfg` and create a host-side plan (no device memory, no CUDA call).
 * Returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED for a bad config. */
moe_status moe_plan_create(const moe_config* cfg, moe_plan** out_plan);

/* Free a plan and, if moe_forward_host was called with it, the side stream and events that
 * call created (on the device it was created on; call after that work has finished).  NULL is
 * accepted. */
moe_status moe_plan_destroy(moe_plan* plan);

/* Bytes of workspace a call with T tokens needs (0 if plan is NULL or T is out of range).
 * Host-only.  The same workspace serves moe_route, moe_permute, moe_forward,
 * moe_forward_routed and moe_forward_host. */
size_t moe_workspace_bytes(const moe_plan* plan, int32_t T);

/* Router: logits = x W_r^T (bf16 inputs, fp32 accumulation), then scoring, optional bias /
 * groups / hash lookup, top-k and gate weights.  The logits run on the tensor cores and the
 * selection in a second kernel; batches of at most 64 tokens over at most 64 experts run both in
 * one kernel (the logits in K slices of 256 on the CUDA cores, summed in slice order before the
 * selection).
 *   topk_ids [T,k] int32 out: descending selection key, ties -> lower expert id (hash: table
 *   order); topk_w [T,k] fp32 out.  logits [T,E] fp32 out, optional (NULL = not exported).
 *   token_ids is required iff the plan uses hash routing; bias may be NULL. */
moe_status moe_route(moe_plan* plan, int32_t T, const moe_bf16* x, const int32_t* token_ids,
                     const moe_bf16* w_r, const float* bias, int32_t* topk_ids, float* topk_w,
                     float* logits, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Dispatch permutation of given topk_ids [T,k] (router page, "Token Dispatch"):
 *   counts [E] (tokens_per_expert), offsets [E+1] (exclusive prefix sum),
 *   perm_tok [T*k] (permuted_token_ids: token of each expert-major row),
 *   inv [T*k] (row of assignment t*k+j).  Rows are ordered by expert, then by t*k+j.
 * Any output pointer may be NULL (not written).  Integer-exact and deterministic. */
moe_status moe_permute(moe_plan* plan, int32_t T, const int32_t* topk_ids, int32_t* counts,
                       int32_t* offsets, int32_t* perm_tok, int32_t* inv, void* ws,
                       size_t ws_bytes, moe_stream_t stream);

/* moe_permute without a workspace, for callers that cannot allocate device memory: a plugin
 * inside a host framework that owns all device memory through its own allocator, or a
 * latency-critical loop where cudaMalloc (which can synchronise the device) is not allowed.
 * The source pages have no counterpart: this is an interface convenience of this library.
 * Same outputs as moe_permute (all four must be non-NULL).  Scratch lives in a fixed
 * ~0.33 MB array of device memory inside the library (held by every GPU that loads it until
 * exit); T * top_k above 131072 returns MOE_ERR_UNSUPPORTED.  Every call shares that array:
 * calls whose work overlaps on the GPU (unordered streams) race.  The first call on a device
 * looks up the array's address; make it before any stream capture.  Nothing is allocated.
 * An expert id outside [0, E) is clamped into range as in moe_permute and flagged in the
 * array's error word (cleared by every call); this call itself returns MOE_OK regardless,
 * and moe_permute_noalloc_status reports the flag. */
moe_status moe_permute_noalloc(moe_plan* plan, int32_t T, const int32_t* topk_ids, int32_t* counts,
                               int32_t* offsets, int32_t* perm_tok, int32_t* inv, moe_stream_t stream);

/* Device-data status of the most recent moe_permute_noalloc call on the current device (whatever
 * its stream): synchronises `stream` (which should be the one that call ran on), then returns
 * MOE_ERR_DEVICE_INPUT if that call met an expert id outside [0, E), else MOE_OK (also when no
 * call has run on this device).  Allocates nothing. */
moe_status moe_permute_noalloc_status(moe_stream_t stream);

/* FP8 (E4M3) weights with one power-of-two scale per 128 x 128 tile ("DeepSeek-V4 MoE",
 * section "FP4 QAT 怎么做到反量化无损": FP8 E4M3 weights, one scale per 128 x 128 tile).
 *   w [n_mats, rows, K] bf16 (device, 2-byte aligned) -> codes [n_mats, rows, K] uint8 E4M3 bit
 *   patterns and exps [n_mats, ceil(rows/128), ceil(K/128)] int8, tiles counted from each
 *   matrix's first row and column.  e = the smallest integer with max|w| <= 448 * 2^e over the
 *   tile (0 for an all-zero tile, at least -126); code = round-to-nearest-even of w * 2^-e,
 *   negative zero stored as 0x00.  q * 2^e is exact and is a bf16 value.  Run once per weight
 *   set (w13 as n_mats = E, rows = 2*d_ff, K = d; w2 as E, d, d_ff; shared with n_mats = 1)
 *   for moe_forward_fp8.  Enqueued on `stream`; no plan needed; outputs caller-owned. */
moe_status moe_quantize_fp8(const moe_bf16* w, int32_t n_mats, int32_t rows, int32_t K, uint8_t* codes,
                            int8_t* exps, moe_stream_t stream);

/* MXFP4 (E2M1) weights with one power-of-two scale per 1 x 32 sub-block ("DeepSeek-V4 MoE",
 * section "FP4 QAT 怎么做到反量化无损": FP4 E2M1 sub-blocks of 1 x 32, losslessly dequantised to
 * FP8 E4M3 tiles of 128 x 128 while the sub-block scales inside a tile stay within the FP8
 * exponent headroom).
 *   w [n_mats, rows, K] bf16 (device, 16-byte aligned, K a multiple of 32) -> codes
 *   [n_mats, rows, K/2] uint8 (16-byte aligned; two elements per byte, element 2i of a row in
 *   the low nibble of byte i, each nibble an E2M1 code: sign << 3 | the index of the magnitude
 *   in {0, 0.5, 1, 1.5, 2, 3, 4, 6}) and exps
 *   [n_mats, rows, K/32] int8.  s = the smallest integer with max|w| <= 6 * 2^s over the
 *   sub-block (at least -114), raised to (the largest s of its 128 x 128 tile) - 14 where lower;
 *   an all-zero sub-block takes the tile's largest s.  code = round-to-nearest-even of w * 2^-s
 *   on the E2M1 grid, zero stored as +0.  Enqueued on `stream`; no plan needed. */
moe_status moe_quantize_mxfp4(const moe_bf16* w, int32_t n_mats, int32_t rows, int32_t K, uint8_t* codes,
                              int8_t* exps, moe_stream_t stream);

/* The lossless conversion of MXFP4 weights (as moe_quantize_mxfp4 writes them) to the FP8 form
 * of moe_quantize_fp8: per 128 x 128 tile, E = (largest sub-block exponent) - 6 and each element
 * the E4M3 code of q * 2^(s - E), exact because s - E lies in [-8, 6].  codes [n_mats, rows,
 * K/2], exps [n_mats, rows, K/32] -> q8 [n_mats, rows, K] (16-byte aligned), e8 [n_mats,
 * ceil(rows/128), ceil(K/128)], ready for moe_forward_fp8.  q8 may be NULL: only e8 is
 * written.  Exponents from elsewhere that exceed
 * the headroom are rounded to nearest E4M3 (saturating).  Enqueued on `stream`. */
moe_status moe_mxfp4_to_fp8(const uint8_t* codes, const int8_t* exps, int32_t n_mats, int32_t rows, int32_t K,
                            uint8_t* q8, int8_t* e8, moe_stream_t stream);

/* moe_forward with FP8 expert weights (the router stays bf16): q13 [E, 2*d_ff, d] and q2
 * [E, d, d_ff] hold E4M3 codes, e13 [E, ceil(2*d_ff/128), ceil(d/128)] and e2 [E, ceil(d/128),
 * ceil(d_ff/128)] their tile exponents, as moe_quantize_fp8 writes them (shared expert: the
 * same with E = 1; NULL without one).  The layer is moe_forward on the dequantised weights
 * q * 2^e, with the activations kept at bf16-level precision.  With d and d_ff multiples of 128
 * the codes go straight to the tensor cores, with the activations as sums of E4M3 pieces (piece
 * p weighted 2^(-4p)) and one power-of-two scale per row: x in two pieces, exact for every value
 * above 2^-13.8 of its row's largest magnitude and within 2^-21 of that magnitude below it; h in
 * four pieces, within 2^-16 of each value plus 2^-29 of the row's largest magnitude.  Batches of
 * at most 64 tokens, or that route at most 48 rows to an expert on average (T k <= 48 E), stream
 * the weights through single-CTA kernels (the 8-bit MMA, the tile scales applied per K tile);
 * larger batches run the block-scaled 2-SM MMA (kind::mxf8f6f4), the tile scales applied by the
 * tensor cores.  Other shapes widen the codes to bf16 (in Tensor Memory on the single-CTA
 * kernels, in shared memory on CTA pairs) and run the bf16 MMA on moe_forward's activations
 * (bf16 x, the (hi, lo) pair for h).  moe_forward and moe_forward_mxfp4 choose between their
 * single-CTA and CTA-pair kernels by the same rule.
 * Code pointers 16-byte aligned; same workspace and outputs as moe_forward. */
moe_status moe_forward_fp8(moe_plan* plan, int32_t T, const moe_bf16* x, const int32_t* token_ids,
                           const moe_bf16* w_r, const float* bias, const uint8_t* q13, const int8_t* e13,
                           const uint8_t* q2, const int8_t* e2, const uint8_t* q13_sh, const int8_t* e13_sh,
                           const uint8_t* q2_sh, const int8_t* e2_sh, moe_bf16* out, void* ws, size_t ws_bytes,
                           moe_stream_t stream);

/* Aux-loss-free selection-bias step ("MoE compute and communication", sec. 七.3; "DeepSeek-V4
 * MoE", aux-loss-free balancing, update speed 0.001): for each expert e with load counts[e]
 * (tokens_per_expert of a T-token step, e.g. from moe_permute or moe_workspace_views),
 * bias[e] -= gamma if counts[e] > T*k/E, bias[e] += gamma if counts[e] < T*k/E, unchanged at
 * the mean (compared exactly in integers; one fp32 addition).  counts [E] int32 and bias [E]
 * fp32 (updated in place) are device pointers; gamma >= 0 (0.001 in the pages). */
moe_status moe_update_bias(moe_plan* plan, int32_t T, const int32_t* counts, float* bias, float gamma,
                           moe_stream_t stream);

/* Whole layer forward: route, dispatch, grouped SwiGLU GEMMs (routed + shared expert),
 * combine.  out [T,d] bf16.  Deterministic: no atomics in any floating-point reduction.
 * w13_sh / w2_sh are required iff n_shared = 1.  Intermediates (routing result, dispatch
 * rows, activations) stay in the workspace; see moe_workspace_views(). */
moe_status moe_forward(moe_plan* plan, int32_t T, const moe_bf16* x, const int32_t* token_ids,
                       const moe_bf16* w_r, const float* bias, const moe_bf16* w13,
                       const moe_bf16* w2, const moe_bf16* w13_sh, const moe_bf16* w2_sh,
                       moe_bf16* out, void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_forward with native MXFP4 expert weights (the router stays bf16): c13 [E, 2*d_ff, d/2]
 * and c2 [E, d, d_ff/2] packed E2M1 codes, s13 [E, 2*d_ff, d/32] and s2 [E, d, d_ff/32] their
 * sub-block exponents, as moe_quantize_mxfp4 writes them; shared expert the same with E = 1
 * (NULL without one).  The GEMMs feed the stored 4-bit codes to the block-scaled tensor-core MMA
 * with their 1 x 32 sub-block scales 2^s (as UE8M0 scales, s below -127 taken as -127) and the
 * activations as E4M3 pieces (see moe_forward_fp8), accumulating in fp32: the layer is the bf16
 * layer on the dequantised weights q * 2^s up to the pieces' precision and the order of the
 * fp32 sums.  Needs d and d_ff multiples of 128 (else MOE_ERR_UNSUPPORTED); 16-, 32- or 64-row
 * token tiles by batch size.  Code pointers 32-byte aligned, sub-block exponents 4-byte aligned
 * (else MOE_ERR_ALIGNMENT); same workspace and outputs as moe_forward. */
moe_status moe_forward_mxfp4(moe_plan* plan, int32_t T, const moe_bf16* x, const int32_t* token_ids,
                             const moe_bf16* w_r, const float* bias, const uint8_t* c13, const int8_t* s13,
                             const uint8_t* c2, const int8_t* s2, const uint8_t* c13_sh, const int8_t* s13_sh,
                             const uint8_t* c2_sh, const int8_t* s2_sh, moe_bf16* out, void* ws, size_t ws_bytes,
                             moe_stream_t stream);

/* Layer forward with the routing given by the caller (topk_ids [T,k] int32 in [0,E),
 * topk_w [T,k] fp32): dispatch, grouped GEMMs and combine only. */
moe_status moe_forward_routed(moe_plan* plan, int32_t T, const moe_bf16* x,
                              const int32_t* topk_ids, const float* topk_w,
                              const moe_bf16* w13, const moe_bf16* w2, const moe_bf16* w13_sh,
                              const moe_bf16* w2_sh, moe_bf16* out, void* ws, size_t ws_bytes,
                              moe_stream_t stream);

/* moe_forward with HOST activations: x_host [T,d] bf16 and token_ids_host [T] (hash only)
 * are copied to the workspace, the layer runs, and out_host [T,d] receives the result
 * (pinned host memory makes the copies asynchronous).  Weights stay device pointers.
 * The input copy runs on a side stream the plan creates on first use (on the current device):
 * it lands in one of two staging slots that alternate between calls, waits only for the layer
 * that last read that slot, and `stream` waits for it before the layer runs.  So consecutive
 * calls overlap one call's input copy with the previous call's layer, while synchronising
 * `stream` still covers the whole call; the caller must not change x_host / token_ids_host
 * until then.  When out_host is page-locked memory the device can address (cudaHostAlloc /
 * cudaMallocHost), the combine writes the result into it directly; otherwise the result is
 * staged in the workspace and copied.  A plan serves one host thread at a time. */
moe_status moe_forward_host(moe_plan* plan, int32_t T, const moe_bf16* x_host,
                            const int32_t* token_ids_host, const moe_bf16* w_r,
                            const float* bias, const moe_bf16* w13, const moe_bf16* w2,
                            const moe_bf16* w13_sh, const moe_bf16* w2_sh, moe_bf16* out_host,
                            void* ws, size_t ws_bytes, moe_stream_t stream);

/* Synchronise `stream` and read the workspace error word written by the last call that used
 * `ws`: MOE_OK, MOE_ERR_DEVICE_INPUT (clamped bad ids), MOE_ERR_TIMEOUT, or (debug-bounds
 * builds) MOE_ERR_INTERNAL; a timeout takes precedence, then an internal check. */
moe_status moe_check_status(moe_plan* plan, const void* ws, moe_stream_t stream);

/* Device addresses, inside `ws`, of the intermediates of the last forward with T tokens.
 * Valid until the next call that uses `ws`.  Any output may be NULL. */
typedef struct {
  int32_t* topk_ids;   /* [T, k]                                                      */
  float* topk_w;       /* [T, k]                                                      */
  float* logits;       /* [T, E] router logits                                        */
  int32_t* counts;     /* [E]                                                         */
  int32_t* offsets;    /* [E+1]                                                       */
  int32_t* perm_tok;   /* [T*k]                                                       */
  int32_t* inv;        /* [T*k]                                                       */
  moe_bf16* h;         /* [T*k + n_shared*T, 2*d_ff] SwiGLU activations h = hi + lo (bf16 pair;
                          per 64-feature block b, hi in columns 128b..128b+63, lo in the next
                          64); routed rows first,
                          expert-major; then the shared expert's T rows)               */
  float* o;            /* [T*k + n_shared*T, d] gate-weighted expert outputs          */
} moe_ws_views;
moe_status moe_workspace_views(const moe_plan* plan, int32_t T, void* ws, moe_ws_views* out);

/* Stage timing.  With events set, moe_forward / moe_forward_routed record events[0] before
 * the first launch and events[i] after stage i (stages: 1 router GEMM, 2 top-k (empty where the
 * router is one kernel, see moe_route),
 * 3 dispatch (histogram, scan, scatter, row gather), 4 gate/up grouped GEMM, 5 down grouped
 * GEMM, 6 combine; moe_forward_routed records the stages it runs).  n_events must be
 * >= moe_forward_stage_count() + 1; NULL / 0 disables.  Events are the caller's. */
int32_t moe_forward_stage_count(void);
moe_status moe_plan_set_events(moe_plan* plan, moe_event_t* events, int32_t n_events);

/* Kernel launches one moe_forward enqueues (memsets and event records not counted). */
int32_t moe_forward_launch_count(const moe_plan* plan, int32_t T);

/* Static text for a status code. */
const char* moe_status_string(moe_status status);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
