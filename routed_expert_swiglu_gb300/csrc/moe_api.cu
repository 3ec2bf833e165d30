// C ABI of the MoE layer (declared in include/moe.h): argument validation, workspace layout,
// and the launch sequence router GEMM -> top-k -> dispatch -> gate/up GEMM -> down GEMM ->
// combine on the caller's stream.  No device allocation, no host synchronisation (except
// moe_check_status).
#include <cuda_runtime.h>

#include <algorithm>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"

// Side stream of moe_forward_host: input copies run on it so that the copy of one call's input
// overlaps the previous call's layer (created on first use, on the device current then).
struct HostPipe {
  int dev;
  cudaStream_t copy;
  cudaEvent_t h2d_done;
  cudaEvent_t slot_free[2];  // the layer that last read input slot s has finished
  int slot;
};

struct moe_plan {
  moe_config cfg;
  moe_event_t* events;
  int n_events;
  HostPipe* pipe;
};

static void destroy_pipe(HostPipe* q) {
  if (q == nullptr) return;
  cudaEventDestroy(q->h2d_done);
  cudaEventDestroy(q->slot_free[0]);
  cudaEventDestroy(q->slot_free[1]);
  cudaStreamDestroy(q->copy);
  free(q);
}

namespace moe {

WsLayout ws_layout(const moe_config& c, int T) {
  WsLayout L;
  memset(&L, 0, sizeof(L));
  const int E = c.n_experts, k = c.top_k, d = c.d, f = c.d_ff, sh = c.n_shared;
  L.T = T;
  L.N = T * k;
  L.G = E + sh;
  L.TN = token_tile_for(T, k, E);
  L.nblk = ceil_div(L.N > 0 ? L.N : 1, PERMUTE_CHUNK);
  // row tiles of the narrowest schedule a forward may build
  const int tn_sched = 16;  // the narrowest: the MXFP4 kernels' 16-row tiles
  L.max_rt = E + ceil_div(L.N, tn_sched) + sh * ceil_div(T, tn_sched) + 1;
  const size_t rows_h = (size_t)L.N + (size_t)sh * T;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + (bytes ? bytes : 1), 256);
    return at;
  };
  L.err = take(ERR_BLOCK_BYTES);
  // Input staging of moe_forward_host: two slots (alternate calls) of max_tokens rows, at the
  // same offsets for every T, so that a side-stream copy into one never overlaps a buffer of
  // another call on the same workspace.
  L.x_stage = take((size_t)2 * c.max_tokens * d * 2);
  L.tok_stage = take((size_t)2 * c.max_tokens * 4);
  L.topk_ids = take((size_t)T * k * 4);
  L.topk_w = take((size_t)T * k * 4);
  // partial logits of the K slices (the tensor-core router's, or the fused small-batch router's)
  const int slabs = std::max(router_ksplit(c, T), router_fused(T, E) ? router_fused_slices(d) : 1);
  L.logits = take((size_t)slabs * T * E * 4);
  L.blockhist = take((size_t)L.nblk * E * 4);
  L.counts = take((size_t)E * 4);
  L.offsets = take((size_t)(E + 1) * 4);
  L.grp = take((size_t)(L.G + 1) * 16);
  L.rt2g = take((size_t)L.max_rt * 4);
  L.perm_tok = take((size_t)L.N * 4);
  L.inv = take((size_t)L.N * 4);
  L.row_w = take((size_t)L.N * 4);
  // dispatched rows (bf16), or with FP8 weights the routed and shared rows as two E4M3 pieces
  L.xd = take(rows_h * d * 2);
  L.xexp = take(rows_h * 4);
  L.h = take(rows_h * 2 * f * 2);  // hi/lo bf16 pair per activation (FP8 weights: fp32, then 4 pieces)
  L.hexp = take(rows_h * 4);
  L.o = take(rows_h * d * 4);
  L.out_stage = take((size_t)T * d * 2);
  L.total = off;
  return L;
}

const moe_config* plan_config(const moe_plan* p) { return &p->cfg; }

int router_ksplit(const moe_config& c, int T) {
  if (T <= 0) return 1;
  const int mblk = c.n_experts > 128 ? 2 : 1;
  const int base_tiles = ceil_div(T, router_tile_for(T)) * ceil_div(c.n_experts, gemm_features_per_tile(1, mblk));
  if (base_tiles >= 64) return 1;
  int want = 128 / base_tiles;
  if (want > 16) want = 16;
  const int KB = c.d / 64;
  int ks = 1;
  for (int q = 1; q <= want; ++q)
    if (KB % q == 0) ks = q;
  return ks;
}

}  // namespace moe

using namespace moe;

namespace {

enum Stage { ST_START = 0, ST_ROUTER_GEMM = 1, ST_TOPK = 2, ST_DISPATCH = 3, ST_GATE_UP = 4, ST_DOWN = 5,
             ST_COMBINE = 6, ST_COUNT = 6 };

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

moe_status validate_config(const moe_config* c) {
  if (c == nullptr) return MOE_ERR_INVALID_ARG;
  if (c->d <= 0 || c->d_ff <= 0 || c->n_experts <= 0 || c->top_k <= 0 || c->max_tokens <= 0)
    return MOE_ERR_INVALID_ARG;
  if (c->n_shared < 0 || c->n_shared > 1) return MOE_ERR_UNSUPPORTED;
  if (c->top_k > c->n_experts) return MOE_ERR_INVALID_ARG;
  if (c->score < MOE_SCORE_SOFTMAX_TOPK || c->score > MOE_SCORE_SQRT_SOFTPLUS) return MOE_ERR_INVALID_ARG;
  if (c->d % 64 != 0 || c->d_ff % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (c->n_experts > MAX_EXPERTS || c->top_k > MAX_TOPK || c->max_tokens > MAX_TOKENS) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)c->n_experts * 2 * c->d_ff >= (1ll << 31) || (int64_t)c->n_experts * c->d >= (1ll << 31))
    return MOE_ERR_UNSUPPORTED;
  if ((int64_t)c->max_tokens * c->top_k * (c->d > c->d_ff ? c->d : c->d_ff) >= (1ll << 40))
    return MOE_ERR_UNSUPPORTED;
  if (c->n_groups < 0 || c->topk_groups < 0 || c->group_topk < 0) return MOE_ERR_INVALID_ARG;
  if (c->n_groups > 0) {
    if (c->n_groups > MAX_GROUPS) return MOE_ERR_UNSUPPORTED;
    if (c->n_experts % c->n_groups != 0) return MOE_ERR_INVALID_ARG;
    const int gsz = c->n_experts / c->n_groups;
    if (c->topk_groups < 1 || c->topk_groups > c->n_groups) return MOE_ERR_INVALID_ARG;
    if (c->group_topk < 1 || c->group_topk > gsz) return MOE_ERR_INVALID_ARG;
    if (c->group_topk > 8) return MOE_ERR_UNSUPPORTED;
    if (c->top_k > c->topk_groups * gsz) return MOE_ERR_INVALID_ARG;
  }
  if (c->tid2eid != nullptr) {
    if (c->vocab <= 0) return MOE_ERR_INVALID_ARG;
    if (!aligned(c->tid2eid, 4)) return MOE_ERR_ALIGNMENT;
  }
  return MOE_OK;
}

moe_status check_common(const moe_plan* p, int32_t T, const void* ws, size_t ws_bytes) {
  if (p == nullptr) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > p->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return MOE_ERR_ALIGNMENT;
  if (ws_bytes < ws_layout(p->cfg, T).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

moe_status need16(const void* ptr) {
  if (ptr == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned(ptr, 16)) return MOE_ERR_ALIGNMENT;
  return MOE_OK;
}

#define MOE_TRY(expr)                    \
  do {                                   \
    const moe_status st_ = (expr);       \
    if (st_ != MOE_OK) return st_;       \
  } while (0)
#define MOE_CUDA(expr)                              \
  do {                                              \
    if ((expr) != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

moe_status num_sms(int* out) {
  int dev = 0;
  MOE_CUDA(cudaGetDevice(&dev));
  MOE_CUDA(cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev));
  return MOE_OK;
}

void record(const moe_plan* p, int stage, cudaStream_t s) {
  if (p->events != nullptr && stage < p->n_events) cudaEventRecord(reinterpret_cast<cudaEvent_t>(p->events[stage]), s);
}

// Host-side NVTX range around one launch ("moe.<kernel>"), closed on every return path.  NVTX is
// header-only here and costs nothing unless a profiler is attached.
struct LaunchRange {
  explicit LaunchRange(const char* name) { nvtxRangePushA(name); }
  ~LaunchRange() { nvtxRangePop(); }
};

// Router GEMM + top-k into the given outputs.
moe_status run_route(const moe_plan* p, int T, const moe_bf16* x, const int32_t* token_ids, const moe_bf16* w_r,
                     const float* bias, float* logits, int32_t* ids, float* w, void* ws, int sms, cudaStream_t s) {
  const moe_config& c = p->cfg;
  const WsLayout L = ws_layout(c, T);
  int* err = at<int>(ws, L.err);
  if (router_fused(T, c.n_experts)) {
    // one launch: logits in K slices, the last block of each token group sums them and selects
    RouterFusedLaunch rf;
    memset(&rf, 0, sizeof(rf));
    rf.x = x;
    rf.w_r = w_r;
    rf.T = T;
    rf.d = c.d;
    rf.E = c.n_experts;
    rf.partial = at<float>(ws, L.logits);
    rf.counters = reinterpret_cast<int*>(at<char>(ws, L.err) + ROUTER_COUNTERS_OFFSET);
    TopkLaunch& tk = rf.tk;
    tk.logits = rf.partial;
    tk.nsplit = router_fused_slices(c.d);
    tk.split_stride = (long long)T * c.n_experts;
    tk.logits_out = logits;  // the summed logits (over slab 0 of the token's row when it is the workspace's)
    tk.bias = bias;
    tk.T = T;
    tk.E = c.n_experts;
    tk.k = c.top_k;
    tk.score = c.score;
    tk.n_groups = c.n_groups;
    tk.topk_groups = c.topk_groups;
    tk.group_topk = c.group_topk;
    tk.token_ids = token_ids;
    tk.tid2eid = c.tid2eid;
    tk.vocab = c.vocab;
    tk.topk_ids = ids;
    tk.topk_w = w;
    tk.err = err;
    {
      LaunchRange r("moe.router_fused");
      MOE_CUDA(launch_router_fused(rf, s));
    }
    record(p, ST_ROUTER_GEMM, s);
    record(p, ST_TOPK, s);
    return MOE_OK;
  }
  GemmLaunch g;
  memset(&g, 0, sizeof(g));
  g.epi = 1;
  g.TN = router_tile_for(T);
  g.a_ptr = w_r;
  g.a_rows = c.n_experts;
  g.b_ptr = x;
  g.b_rows = T;
  g.K = c.d;
  g.mblk = c.n_experts > 128 ? 2 : 1;
  g.num_mblocks = ceil_div(c.n_experts, gemm_features_per_tile(1, g.mblk));
  g.out_features = c.n_experts;
  g.out_ld = c.n_experts;
  g.out_rows = T;
  g.out = logits;
  g.n_routed = 1;
  g.dense_rows = T;
  g.ksplit = router_ksplit(c, T);
  g.split_stride = (long long)T * c.n_experts;
  if (g.ksplit > 1) g.out = at<float>(ws, L.logits);  // partial slabs; top-k sums them
  g.max_tiles = ceil_div(T, g.TN) * g.num_mblocks;
  g.err = err;
  g.num_sms = sms;
  {
    LaunchRange r("moe.router_gemm");
    MOE_CUDA(launch_grouped_gemm(g, s));
  }
  record(p, ST_ROUTER_GEMM, s);
  TopkLaunch tk;
  tk.nsplit = g.ksplit;
  tk.split_stride = g.split_stride;
  tk.logits = g.ksplit > 1 ? at<float>(ws, L.logits) : logits;
  // summed logits go to the caller's buffer, or in place into slab 0 of the workspace
  tk.logits_out = g.ksplit > 1 ? logits : nullptr;
  tk.bias = bias;
  tk.T = T;
  tk.E = c.n_experts;
  tk.k = c.top_k;
  tk.score = c.score;
  tk.n_groups = c.n_groups;
  tk.topk_groups = c.topk_groups;
  tk.group_topk = c.group_topk;
  tk.token_ids = token_ids;
  tk.tid2eid = c.tid2eid;
  tk.vocab = c.vocab;
  tk.topk_ids = ids;
  tk.topk_w = w;
  tk.err = err;
  {
    LaunchRange r("moe.topk");
    MOE_CUDA(launch_topk(tk, s));
  }
  record(p, ST_TOPK, s);
  return MOE_OK;
}

// Shapes for which FP8 weights feed the MMA directly: every 128-row weight slab and 128-wide K
// tile lies on one scale tile, and activation rows fit the split kernel.
bool fp8_mma_shapes(const moe_config& c) {
  return MOE_FP8_MMA && c.d % 128 == 0 && c.d_ff % 128 == 0 && (size_t)c.d * 4 <= SPLIT_SMEM_MAX &&
         (size_t)c.d_ff * 4 <= SPLIT_SMEM_MAX;
}

// Dispatch + grouped GEMMs + combine, from routing in the workspace or the caller's buffers.
// FP8 (E4M3) expert weights: codes and 128 x 128 tile exponents (see moe_quantize_fp8).  With
// the sub-block exponents s* set, MXFP4 weights instead: packed E2M1 codes and their 1 x 32
// sub-block exponents (see moe_quantize_mxfp4); the tile exponents are then unused.
struct Fp8Weights {
  const uint8_t* q13; const int8_t* e13; const uint8_t* q2; const int8_t* e2;
  const uint8_t* q13_sh; const int8_t* e13_sh; const uint8_t* q2_sh; const int8_t* e2_sh;
  const int8_t* s13; const int8_t* s2; const int8_t* s13_sh; const int8_t* s2_sh;
};

moe_status run_experts(const moe_plan* p, int T, const moe_bf16* x, const int32_t* ids, const float* w,
                       const moe_bf16* w13, const moe_bf16* w2, const moe_bf16* w13_sh, const moe_bf16* w2_sh,
                       moe_bf16* out, void* ws, int sms, cudaStream_t s, const Fp8Weights* q8 = nullptr) {
  const moe_config& c = p->cfg;
  const WsLayout L = ws_layout(c, T);
  int* err = at<int>(ws, L.err);
  const int E = c.n_experts, d = c.d, f = c.d_ff, sh = c.n_shared;
  PermuteLaunch pm;
  pm.topk_ids = ids;
  pm.topk_w = w;
  pm.T = T;
  pm.k = c.top_k;
  pm.E = E;
  pm.n_shared = sh;
  // FP8 weights: a schedule of the FP8 kernels' own row tiles (the widening kernels: 64 rows)
  const bool f4 = q8 != nullptr && q8->s13 != nullptr;  // native MXFP4 (block-scaled MMA)
  if (f4 && !fp8_mma_shapes(c)) return MOE_ERR_UNSUPPORTED;
  // FP8 / MXFP4 weights at prefill: the block-scaled CTA-pair kernels (codes and scales into the
  // 2-SM MMA, E4M3-piece activations, 224-row token tiles); FP8 shapes they do not take (d or
  // d_ff not a multiple of 128): codes widened to bf16 in shared memory on the CTA-pair kernels,
  // bf16 activations (the dispatched rows and the (hi, lo) pair), the bf16 path's schedule
  const bool stream = streams_weights(T, c.top_k, E);
  const bool bs_pair = q8 != nullptr && !stream && fp8_mma_shapes(c);
  const bool f8pair = q8 != nullptr && !f4 && !stream && !fp8_mma_shapes(c);
  const bool f8mma = q8 != nullptr && !f8pair && fp8_mma_shapes(c);
  const int sched_tn = (q8 == nullptr || f8pair) ? L.TN
                       : bs_pair                 ? BS_PAIR_TN
                       : f8mma                   ? fp8_token_tile(T, c.top_k, E)
                                                 : 64;
  pm.TN = sched_tn;
  pm.nblk = L.nblk;
  pm.blockhist = at<int32_t>(ws, L.blockhist);
  pm.counts = at<int32_t>(ws, L.counts);
  pm.offsets = at<int32_t>(ws, L.offsets);
  pm.grp = at<int4>(ws, L.grp);
  pm.rt2g = at<int32_t>(ws, L.rt2g);
  pm.perm_tok = at<int32_t>(ws, L.perm_tok);
  pm.inv = at<int32_t>(ws, L.inv);
  pm.row_w = at<float>(ws, L.row_w);
  pm.err = err;
  // FP8 weights straight into the MMA: the activation rows go in as E4M3 pieces (the gather
  // from x builds them, so the dispatch copies no rows)
  pm.x = x;
  pm.xd = f8mma ? nullptr : at<void>(ws, L.xd);
  pm.d = d;
  pm.num_sms = sms;
  {
    LaunchRange r("moe.dispatch");
    MOE_CUDA(launch_permute(pm, s));
  }
  const int64_t rows_h = (int64_t)L.N + (int64_t)sh * T;
  if (f8mma) {
    LaunchRange r("moe.split_rows_e4m3");
    if (T >= SPLIT_TOKEN_MAJOR_MIN_T)  // each x row split once, written to its k (+1) rows
      MOE_CUDA(launch_split_tokens_e4m3(x, pm.inv, T, c.top_k, L.N, sh, d, at<uint8_t>(ws, L.xd),
                                        at<int32_t>(ws, L.xexp), err, s));
    else
      MOE_CUDA(launch_split_rows_e4m3(x, true, pm.perm_tok, L.N, (int)rows_h, d, 2, at<uint8_t>(ws, L.xd),
                                      at<int32_t>(ws, L.xexp), s));
  }
  record(p, ST_DISPATCH, s);

  GemmLaunch g1;
  memset(&g1, 0, sizeof(g1));
  g1.epi = 0;
  g1.TN = L.TN;
  g1.a_ptr = w13;
  g1.a_rows = (int64_t)E * 2 * f;
  g1.a_sh_ptr = sh ? w13_sh : nullptr;
  g1.a_sh_rows = 2 * f;
  g1.b_ptr = pm.xd;
  g1.b_rows = L.N;
  g1.b_sh_ptr = sh ? x : nullptr;
  g1.b_sh_rows = T;
  g1.K = d;
  g1.mblk = 1;
  g1.pair = !stream;
  g1.num_mblocks = ceil_div(f, gemm_features_per_tile(0, 1));
  g1.a_rows_per_group = 2 * f;
  g1.a_up_offset = f;
  g1.out_features = f;
  g1.out_ld = 2 * f;
  g1.out_rows = (int)rows_h;
  g1.out = at<void>(ws, L.h);
  g1.n_routed = E;
  g1.shared_b_shift = -L.N;
  g1.grp = pm.grp;
  g1.rt2g = pm.rt2g;
  g1.max_tiles = L.max_rt * g1.num_mblocks;
  if (q8 != nullptr) {
    g1.q8 = 1;
    g1.a_ptr = q8->q13;
    g1.a_exp = q8->e13;
    g1.a_sh_ptr = sh ? q8->q13_sh : nullptr;
    g1.a_sh_exp = sh ? q8->e13_sh : nullptr;
    g1.pair = f8pair || bs_pair;
    g1.TN = sched_tn;
    g1.kernel_tn = sched_tn;
    if (f8mma) {
      g1.q8 = f4 ? 3 : 2;
      g1.a_sub = f4 ? q8->s13 : nullptr;
      g1.a_sh_sub = (f4 && sh) ? q8->s13_sh : nullptr;
      g1.b_ptr = at<void>(ws, L.xd);
      g1.b_rows = rows_h;  // routed rows, then the shared expert's
      g1.b_sh_ptr = nullptr;
      g1.shared_b_shift = 0;
      g1.b_exp = at<int32_t>(ws, L.xexp);
      g1.out_ld = f;       // fp32 h
    }
  }
  g1.err = err;
  g1.num_sms = sms;
  {
    LaunchRange r("moe.gate_up_gemm");
    MOE_CUDA(launch_grouped_gemm(g1, s));
  }
  if (f8mma) {  // h (fp32) -> four E4M3 pieces per row, in place
    LaunchRange r("moe.split_rows_e4m3");
    MOE_CUDA(launch_split_rows_e4m3(at<void>(ws, L.h), false, nullptr, 0, (int)rows_h, f, 4, at<uint8_t>(ws, L.h),
                                    at<int32_t>(ws, L.hexp), s));
  }
  record(p, ST_GATE_UP, s);

  GemmLaunch g2;
  memset(&g2, 0, sizeof(g2));
  g2.epi = 1;
  g2.TN = L.TN;
  g2.a_ptr = w2;
  g2.a_rows = (int64_t)E * d;
  g2.a_sh_ptr = sh ? w2_sh : nullptr;
  g2.a_sh_rows = d;
  g2.b_ptr = at<void>(ws, L.h);
  g2.b_rows = rows_h;
  g2.K = f;
  g2.hilo = 1;         // B rows hold the (hi, lo) pair: 2*f values, each pair against one W2 block
  g2.mblk = 2;         // decode: two 128-feature blocks per CTA; prefill: a pair tile covers 256
  g2.kernel_tn = L.TN;
  g2.pair = !stream;
  g2.num_mblocks = ceil_div(d, gemm_features_per_tile(1, g2.mblk));
  g2.a_rows_per_group = d;
  g2.out_features = d;
  g2.out_ld = d;
  g2.out_rows = (int)rows_h;
  g2.out = at<void>(ws, L.o);
  g2.row_scale = pm.row_w;
  g2.n_routed = E;
  g2.shared_b_shift = 0;
  g2.grp = pm.grp;
  g2.rt2g = pm.rt2g;
  g2.max_tiles = L.max_rt * g2.num_mblocks;
  if (q8 != nullptr) {
    g2.q8 = 1;
    g2.a_ptr = q8->q2;
    g2.a_exp = q8->e2;
    g2.a_sh_ptr = sh ? q8->q2_sh : nullptr;
    g2.a_sh_exp = sh ? q8->e2_sh : nullptr;
    g2.pair = f8pair || bs_pair;
    g2.TN = sched_tn;
    g2.kernel_tn = sched_tn;
    // four 64-row pieces already fill N = 256 (MXFP4: 32-row tiles too, whose four pieces then sit
    // side by side in N); a pair 256
    g2.mblk = (f8mma && !bs_pair && (sched_tn == 64 || (f4 && sched_tn == 32))) ? 1 : 2;
    g2.num_mblocks = ceil_div(d, gemm_features_per_tile(1, g2.mblk));
    g2.max_tiles = L.max_rt * g2.num_mblocks;
    if (f8mma) {
      g2.q8 = f4 ? 3 : 2;
      g2.a_sub = f4 ? q8->s2 : nullptr;
      g2.a_sh_sub = (f4 && sh) ? q8->s2_sh : nullptr;
      g2.hilo = 0;
      g2.b_exp = at<int32_t>(ws, L.hexp);
    }
  }
  g2.err = err;
  g2.num_sms = sms;
  {
    LaunchRange r("moe.down_gemm");
    MOE_CUDA(launch_grouped_gemm(g2, s));
  }
  record(p, ST_DOWN, s);

  CombineLaunch cb;
  cb.o = at<float>(ws, L.o);
  cb.inv = pm.inv;
  cb.T = T;
  cb.k = c.top_k;
  cb.d = d;
  cb.N = L.N;
  cb.n_shared = sh;
  cb.out = out;
  cb.err = err;
  {
    LaunchRange r("moe.combine");
    MOE_CUDA(launch_combine(cb, s));
  }
  record(p, ST_COMBINE, s);
  return MOE_OK;
}

moe_status check_forward_ptrs(const moe_plan* p, const moe_bf16* w13, const moe_bf16* w2, const moe_bf16* w13_sh,
                              const moe_bf16* w2_sh) {
  MOE_TRY(need16(w13));
  MOE_TRY(need16(w2));
  if (p->cfg.n_shared) {
    MOE_TRY(need16(w13_sh));
    MOE_TRY(need16(w2_sh));
  }
  return MOE_OK;
}

moe_status check_route_ptrs(const moe_plan* p, const moe_bf16* x, const int32_t* token_ids, const moe_bf16* w_r,
                            const float* bias) {
  MOE_TRY(need16(x));
  MOE_TRY(need16(w_r));
  if (bias != nullptr && !aligned(bias, 4)) return MOE_ERR_ALIGNMENT;
  if (p->cfg.tid2eid != nullptr) {
    if (token_ids == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned(token_ids, 4)) return MOE_ERR_ALIGNMENT;
  }
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_plan_create(const moe_config* cfg, moe_plan** out_plan) {
  if (out_plan == nullptr) return MOE_ERR_INVALID_ARG;
  *out_plan = nullptr;
  MOE_TRY(validate_config(cfg));
  moe_plan* p = static_cast<moe_plan*>(calloc(1, sizeof(moe_plan)));
  if (p == nullptr) return MOE_ERR_INVALID_ARG;
  p->cfg = *cfg;
  *out_plan = p;
  return MOE_OK;
}

moe_status moe_plan_destroy(moe_plan* plan) {
  if (plan != nullptr) destroy_pipe(plan->pipe);
  free(plan);
  return MOE_OK;
}

size_t moe_workspace_bytes(const moe_plan* plan, int32_t T) {
  if (plan == nullptr || T < 0 || T > plan->cfg.max_tokens) return 0;
  return ws_layout(plan->cfg, T).total;
}

moe_status moe_route(moe_plan* plan, int32_t T, const moe_bf16* x, const int32_t* token_ids, const moe_bf16* w_r,
                     const float* bias, int32_t* topk_ids, float* topk_w, float* logits, void* ws, size_t ws_bytes,
                     moe_stream_t stream) {
  MOE_TRY(check_common(plan, T, ws, ws_bytes));
  if (T == 0) return MOE_OK;
  MOE_TRY(check_route_ptrs(plan, x, token_ids, w_r, bias));
  if (topk_ids == nullptr || topk_w == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned(topk_ids, 4) || !aligned(topk_w, 4) || (logits != nullptr && !aligned(logits, 16)))
    return MOE_ERR_ALIGNMENT;
  int sms = 0;
  MOE_TRY(num_sms(&sms));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const WsLayout L = ws_layout(plan->cfg, T);
  MOE_CUDA(cudaMemsetAsync(at<int>(ws, L.err), 0, ERR_BLOCK_BYTES, s));
  float* lg = logits != nullptr ? logits : at<float>(ws, L.logits);
  return run_route(plan, T, x, token_ids, w_r, bias, lg, topk_ids, topk_w, ws, sms, s);
}

moe_status moe_permute(moe_plan* plan, int32_t T, const int32_t* topk_ids, int32_t* counts, int32_t* offsets,
                       int32_t* perm_tok, int32_t* inv, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_common(plan, T, ws, ws_bytes));
  if (T == 0) return MOE_OK;
  if (topk_ids == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned(topk_ids, 4) || !aligned(counts, 4) || !aligned(offsets, 4) || !aligned(perm_tok, 4) ||
      !aligned(inv, 4))
    return MOE_ERR_ALIGNMENT;
  int sms = 0;
  MOE_TRY(num_sms(&sms));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const moe_config& c = plan->cfg;
  const WsLayout L = ws_layout(c, T);
  int* err = at<int>(ws, L.err);
  MOE_CUDA(cudaMemsetAsync(err, 0, sizeof(int), s));
  PermuteLaunch pm;
  memset(&pm, 0, sizeof(pm));
  pm.topk_ids = topk_ids;
  pm.T = T;
  pm.k = c.top_k;
  pm.E = c.n_experts;
  pm.n_shared = c.n_shared;
  pm.TN = L.TN;
  pm.nblk = L.nblk;
  pm.blockhist = at<int32_t>(ws, L.blockhist);
  pm.counts = counts != nullptr ? counts : at<int32_t>(ws, L.counts);
  pm.offsets = offsets != nullptr ? offsets : at<int32_t>(ws, L.offsets);
  pm.grp = at<int4>(ws, L.grp);
  pm.rt2g = at<int32_t>(ws, L.rt2g);
  pm.perm_tok = perm_tok != nullptr ? perm_tok : at<int32_t>(ws, L.perm_tok);
  pm.inv = inv != nullptr ? inv : at<int32_t>(ws, L.inv);
  pm.err = err;
  pm.num_sms = sms;
  MOE_CUDA(launch_permute(pm, s));
  return MOE_OK;
}

moe_status moe_forward(moe_plan* plan, int32_t T, const moe_bf16* x, const int32_t* token_ids, const moe_bf16* w_r,
                       const float* bias, const moe_bf16* w13, const moe_bf16* w2, const moe_bf16* w13_sh,
                       const moe_bf16* w2_sh, moe_bf16* out, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_common(plan, T, ws, ws_bytes));
  if (T == 0) return MOE_OK;
  MOE_TRY(check_route_ptrs(plan, x, token_ids, w_r, bias));
  MOE_TRY(check_forward_ptrs(plan, w13, w2, w13_sh, w2_sh));
  MOE_TRY(need16(out));
  int sms = 0;
  MOE_TRY(num_sms(&sms));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const WsLayout L = ws_layout(plan->cfg, T);
  record(plan, ST_START, s);
  MOE_CUDA(cudaMemsetAsync(at<int>(ws, L.err), 0, ERR_BLOCK_BYTES, s));
  int32_t* ids = at<int32_t>(ws, L.topk_ids);
  float* w = at<float>(ws, L.topk_w);
  MOE_TRY(run_route(plan, T, x, token_ids, w_r, bias, at<float>(ws, L.logits), ids, w, ws, sms, s));
  return run_experts(plan, T, x, ids, w, w13, w2, w13_sh, w2_sh, out, ws, sms, s);
}

moe_status moe_forward_fp8(moe_plan* plan, int32_t T, const moe_bf16* x, const int32_t* token_ids,
                           const moe_bf16* w_r, const float* bias, const uint8_t* q13, const int8_t* e13,
                           const uint8_t* q2, const int8_t* e2, const uint8_t* q13_sh, const int8_t* e13_sh,
                           const uint8_t* q2_sh, const int8_t* e2_sh, moe_bf16* out, void* ws, size_t ws_bytes,
                           moe_stream_t stream) {
  MOE_TRY(check_common(plan, T, ws, ws_bytes));
  if (T == 0) return MOE_OK;
  MOE_TRY(check_route_ptrs(plan, x, token_ids, w_r, bias));
  MOE_TRY(need16(q13));
  MOE_TRY(need16(q2));
  if (e13 == nullptr || e2 == nullptr) return MOE_ERR_INVALID_ARG;
  if (plan->cfg.n_shared) {
    MOE_TRY(need16(q13_sh));
    MOE_TRY(need16(q2_sh));
    if (e13_sh == nullptr || e2_sh == nullptr) return MOE_ERR_INVALID_ARG;
  }
  MOE_TRY(need16(out));
  int sms = 0;
  MOE_TRY(num_sms(&sms));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const WsLayout L = ws_layout(plan->cfg, T);
  record(plan, ST_START, s);
  MOE_CUDA(cudaMemsetAsync(at<int>(ws, L.err), 0, ERR_BLOCK_BYTES, s));
  int32_t* ids = at<int32_t>(ws, L.topk_ids);
  float* w = at<float>(ws, L.topk_w);
  MOE_TRY(run_route(plan, T, x, token_ids, w_r, bias, at<float>(ws, L.logits), ids, w, ws, sms, s));
  const Fp8Weights qw = {q13, e13, q2, e2, q13_sh, e13_sh, q2_sh, e2_sh, nullptr, nullptr, nullptr, nullptr};
  return run_experts(plan, T, x, ids, w, nullptr, nullptr, nullptr, nullptr, out, ws, sms, s, &qw);
}

moe_status moe_forward_mxfp4(moe_plan* plan, int32_t T, const moe_bf16* x, const int32_t* token_ids,
                             const moe_bf16* w_r, const float* bias, const uint8_t* c13, const int8_t* s13,
                             const uint8_t* c2, const int8_t* s2, const uint8_t* c13_sh, const int8_t* s13_sh,
                             const uint8_t* c2_sh, const int8_t* s2_sh, moe_bf16* out, void* ws, size_t ws_bytes,
                             moe_stream_t stream) {
  MOE_TRY(check_common(plan, T, ws, ws_bytes));
  if (T == 0) return MOE_OK;
  if (!fp8_mma_shapes(plan->cfg)) return MOE_ERR_UNSUPPORTED;
  MOE_TRY(check_route_ptrs(plan, x, token_ids, w_r, bias));
  if (c13 == nullptr || c2 == nullptr || s13 == nullptr || s2 == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned(c13, 32) || !aligned(c2, 32) || !aligned(s13, 4) || !aligned(s2, 4)) return MOE_ERR_ALIGNMENT;
  if (plan->cfg.n_shared) {
    if (c13_sh == nullptr || c2_sh == nullptr || s13_sh == nullptr || s2_sh == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned(c13_sh, 32) || !aligned(c2_sh, 32) || !aligned(s13_sh, 4) || !aligned(s2_sh, 4))
      return MOE_ERR_ALIGNMENT;
  }
  MOE_TRY(need16(out));
  int sms = 0;
  MOE_TRY(num_sms(&sms));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const WsLayout L = ws_layout(plan->cfg, T);
  record(plan, ST_START, s);
  MOE_CUDA(cudaMemsetAsync(at<int>(ws, L.err), 0, ERR_BLOCK_BYTES, s));
  int32_t* ids = at<int32_t>(ws, L.topk_ids);
  float* w = at<float>(ws, L.topk_w);
  MOE_TRY(run_route(plan, T, x, token_ids, w_r, bias, at<float>(ws, L.logits), ids, w, ws, sms, s));
  const Fp8Weights qw = {c13, nullptr, c2, nullptr, c13_sh, nullptr, c2_sh, nullptr, s13, s2, s13_sh, s2_sh};
  return run_experts(plan, T, x, ids, w, nullptr, nullptr, nullptr, nullptr, out, ws, sms, s, &qw);
}

moe_status moe_forward_routed(moe_plan* plan, int32_t T, const moe_bf16* x, const int32_t* topk_ids,
                              const float* topk_w, const moe_bf16* w13, const moe_bf16* w2, const moe_bf16* w13_sh,
                              const moe_bf16* w2_sh, moe_bf16* out, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_common(plan, T, ws, ws_bytes));
  if (T == 0) return MOE_OK;
  MOE_TRY(need16(x));
  if (topk_ids == nullptr || topk_w == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned(topk_ids, 4) || !aligned(topk_w, 4)) return MOE_ERR_ALIGNMENT;
  MOE_TRY(check_forward_ptrs(plan, w13, w2, w13_sh, w2_sh));
  MOE_TRY(need16(out));
  int sms = 0;
  MOE_TRY(num_sms(&sms));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const WsLayout L = ws_layout(plan->cfg, T);
  record(plan, ST_START, s);
  MOE_CUDA(cudaMemsetAsync(at<int>(ws, L.err), 0, ERR_BLOCK_BYTES, s));
  record(plan, ST_ROUTER_GEMM, s);
  record(plan, ST_TOPK, s);
  return run_experts(plan, T, x, topk_ids, topk_w, w13, w2, w13_sh, w2_sh, out, ws, sms, s);
}

moe_status moe_forward_host(moe_plan* plan, int32_t T, const moe_bf16* x_host, const int32_t* token_ids_host,
                            const moe_bf16* w_r, const float* bias, const moe_bf16* w13, const moe_bf16* w2,
                            const moe_bf16* w13_sh, const moe_bf16* w2_sh, moe_bf16* out_host, void* ws,
                            size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_common(plan, T, ws, ws_bytes));
  if (T == 0) return MOE_OK;
  if (x_host == nullptr || out_host == nullptr) return MOE_ERR_INVALID_ARG;
  if (plan->cfg.tid2eid != nullptr && token_ids_host == nullptr) return MOE_ERR_INVALID_ARG;
  MOE_TRY(need16(w_r));
  MOE_TRY(check_forward_ptrs(plan, w13, w2, w13_sh, w2_sh));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0;
  MOE_CUDA(cudaGetDevice(&dev));
  if (plan->pipe == nullptr || plan->pipe->dev != dev) {
    destroy_pipe(plan->pipe);
    plan->pipe = nullptr;
    HostPipe* q = static_cast<HostPipe*>(calloc(1, sizeof(HostPipe)));
    if (q == nullptr) return MOE_ERR_INVALID_ARG;
    q->dev = dev;
    if (cudaStreamCreateWithFlags(&q->copy, cudaStreamNonBlocking) != cudaSuccess) {
      free(q);
      return MOE_ERR_CUDA;
    }
    cudaError_t e = cudaEventCreateWithFlags(&q->h2d_done, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&q->slot_free[0], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&q->slot_free[1], cudaEventDisableTiming);
    if (e != cudaSuccess) {
      destroy_pipe(q);
      return MOE_ERR_CUDA;
    }
    plan->pipe = q;
  }
  HostPipe* q = plan->pipe;
  const int slot = q->slot;
  const moe_config& c = plan->cfg;
  const WsLayout L = ws_layout(c, T);
  const size_t xbytes = (size_t)T * c.d * 2;
  moe_bf16* xd = at<moe_bf16>(ws, L.x_stage + (size_t)slot * c.max_tokens * c.d * 2);
  moe_bf16* od = at<moe_bf16>(ws, L.out_stage);
  int32_t* td = nullptr;
  // input copy on the side stream, once the layer that last read this slot (two calls back)
  // is done; the caller's stream waits for it, so every step still carries its own copies
  MOE_CUDA(cudaStreamWaitEvent(q->copy, q->slot_free[slot], 0));
  MOE_CUDA(cudaMemcpyAsync(xd, x_host, xbytes, cudaMemcpyHostToDevice, q->copy));
  if (c.tid2eid != nullptr) {
    td = at<int32_t>(ws, L.tok_stage + (size_t)slot * c.max_tokens * 4);
    MOE_CUDA(cudaMemcpyAsync(td, token_ids_host, (size_t)T * 4, cudaMemcpyHostToDevice, q->copy));
  }
  MOE_CUDA(cudaEventRecord(q->h2d_done, q->copy));
  MOE_CUDA(cudaStreamWaitEvent(s, q->h2d_done, 0));
  // Page-locked, device-mapped host output: the combine writes the result straight into it
  // (one pass over the host link during the combine); any other host buffer gets a copy.
  cudaPointerAttributes pa;
  moe_bf16* out_dev = nullptr;
  if (cudaPointerGetAttributes(&pa, out_host) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
      pa.devicePointer != nullptr && aligned(pa.devicePointer, 16)) {
    out_dev = static_cast<moe_bf16*>(pa.devicePointer);
  } else {
    cudaGetLastError();  // a pageable pointer is not an error
  }
  MOE_TRY(moe_forward(plan, T, xd, td, w_r, bias, w13, w2, w13_sh, w2_sh, out_dev != nullptr ? out_dev : od, ws,
                      ws_bytes, stream));
  MOE_CUDA(cudaEventRecord(q->slot_free[slot], s));
  q->slot = slot ^ 1;
  if (out_dev == nullptr) MOE_CUDA(cudaMemcpyAsync(out_host, od, xbytes, cudaMemcpyDeviceToHost, s));
  return MOE_OK;
}

moe_status moe_check_status(moe_plan* plan, const void* ws, moe_stream_t stream) {
  if (plan == nullptr || ws == nullptr) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  MOE_CUDA(cudaStreamSynchronize(s));
  int v = 0;
  MOE_CUDA(cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost));  // the error word is at offset 0
  if (v & DEVERR_TIMEOUT) return MOE_ERR_TIMEOUT;
  if (v & DEVERR_BOUNDS) return MOE_ERR_INTERNAL;
  if (v != 0) return MOE_ERR_DEVICE_INPUT;
  return MOE_OK;
}

moe_status moe_workspace_views(const moe_plan* plan, int32_t T, void* ws, moe_ws_views* out) {
  if (plan == nullptr || ws == nullptr || out == nullptr || T < 0 || T > plan->cfg.max_tokens)
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(plan->cfg, T);
  out->topk_ids = at<int32_t>(ws, L.topk_ids);
  out->topk_w = at<float>(ws, L.topk_w);
  out->logits = at<float>(ws, L.logits);
  out->counts = at<int32_t>(ws, L.counts);
  out->offsets = at<int32_t>(ws, L.offsets);
  out->perm_tok = at<int32_t>(ws, L.perm_tok);
  out->inv = at<int32_t>(ws, L.inv);
  out->h = at<moe_bf16>(ws, L.h);
  out->o = at<float>(ws, L.o);
  return MOE_OK;
}

int32_t moe_forward_stage_count(void) { return ST_COUNT; }

moe_status moe_plan_set_events(moe_plan* plan, moe_event_t* events, int32_t n_events) {
  if (plan == nullptr) return MOE_ERR_INVALID_ARG;
  if (events == nullptr || n_events <= 0) {
    plan->events = nullptr;
    plan->n_events = 0;
    return MOE_OK;
  }
  if (n_events < ST_COUNT + 1) return MOE_ERR_INVALID_ARG;
  plan->events = events;
  plan->n_events = n_events;
  return MOE_OK;
}

int32_t moe_forward_launch_count(const moe_plan* plan, int32_t T) {
  if (plan == nullptr || T <= 0) return 0;
  return (router_fused(T, plan->cfg.n_experts) ? 1 : 2) /* router GEMM and top-k (fused for small ones) */ +
         permute_launch_count(true, (long long)T * plan->cfg.top_k) +
         2 /* grouped GEMMs */ +
         1 /* combine */;
}

const char* moe_status_string(moe_status status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_ALIGNMENT: return "misaligned pointer";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_INPUT: return "device input out of range (clamped)";
    case MOE_ERR_TIMEOUT: return "kernel pipeline wait timed out";
    case MOE_ERR_INTERNAL: return "internal index check failed";
  }
  return "unknown status";
}

}  // extern "C"
