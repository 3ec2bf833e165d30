// Host-side declarations shared by the translation units of the library: workspace layout,
// kernel launchers and the configuration they need.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int MAX_EXPERTS = 512;
constexpr int MAX_TOPK = 8;
constexpr int MAX_GROUPS = 32;
constexpr int MAX_TOKENS = 1 << 20;
constexpr int PERMUTE_CHUNK = 1024;  // assignments per block in the dispatch kernels

// Token-tile width of the grouped GEMMs for large batches (compile-time, so that it can be swept),
// and TMEM columns per CTA of the CTA-pair (2-SM MMA) prefill kernels.
#ifndef MOE_TN_PREFILL
#define MOE_TN_PREFILL 256
#endif
#ifndef MOE_PAIR_TMEM
#define MOE_PAIR_TMEM 512
#endif
// 1 (test builds only, with a short MOE_WAIT_LIMIT_NS): the epilogue warps of the grouped GEMMs
// (bf16, FP8 and MXFP4) first wait on a barrier phase nothing completes, so that every such
// launch runs out of time and reports MOE_ERR_TIMEOUT through its abort path.
#ifndef MOE_TEST_UNSET_WAIT
#define MOE_TEST_UNSET_WAIT 0
#endif
// 1: FP8 expert weights run the kernels that feed the E4M3 codes straight to the tensor cores
// (tcgen05 kind::f8f6f4, activations split into E4M3 pieces) where the shapes allow it
// (d and d_ff multiples of 128); 0: always the kernels that widen the codes to bf16 first.
#ifndef MOE_FP8_MMA
#define MOE_FP8_MMA 1
#endif
// Largest activation row (bytes, staged as fp32) the E4M3 split kernel takes.
constexpr size_t SPLIT_SMEM_MAX = 200 * 1024;

// Which kernels run the expert GEMMs.  A batch that routes at most 48 rows to an expert on
// average (T k <= 48 E), or has at most 64 tokens, runs the weight-streaming single-CTA kernels
// (64-row token tiles; 16- and 32-row tiles, which leave more of each stage to the weight slab,
// measured slower in bf16); larger ones run the CTA-pair kernels (2-SM MMA, 256 weight rows
// against up to 256 token rows per tile).  Measured with the V4-Flash and V3 layer shapes: up to
// 48 rows per expert the streaming kernels were faster (bf16 layer 3 to 11 %, FP8 and MXFP4
// weights 1.3 to 2.8x), at 64 and more slower.
constexpr long long STREAM_MAX_ROWS_PER_EXPERT = 48;
inline bool streams_weights(int T, int k, int E) {
  return T <= 64 || (long long)T * k <= STREAM_MAX_ROWS_PER_EXPERT * E;
}

// Token-tile width (B-operand rows per tile) of the expert GEMMs and their schedule.
inline int token_tile_for(int T, int k, int E) { return streams_weights(T, k, E) ? 64 : MOE_TN_PREFILL; }

// Token-tile width of the router GEMM: 64-row tiles up to 3072 tokens (measured faster there),
// 256-row tiles above.
inline int router_tile_for(int T) { return T <= 3072 ? 64 : MOE_TN_PREFILL; }

// Token rows per tile of the block-scaled CTA-pair kernels (FP8 / MXFP4 weights at prefill):
// the most that leaves Tensor Memory room for the scales beside two accumulator buffers.
constexpr int BS_PAIR_TN = 224;

// From this batch size the E4M3 pieces of x are made token-major (one split per x row, written
// to all its dispatched rows); below it one CTA per dispatched row gives more parallelism.
constexpr int SPLIT_TOKEN_MAJOR_MIN_T = 1024;

// Row-tile width of the FP8-weight GEMMs' schedule, from the mean rows per routed expert
// T k / E: 16 up to 8 rows, 32 up to 24, else 64.  Narrow tiles leave more of each pipeline
// stage to the weight codes; a tile narrower than an expert's rows streams its weights again.
// The kernels run this schedule without sub-tiles (sub-tiles of a wider schedule alias with the
// grid stride, leaving the CTAs that only ever draw the mostly empty later sub-tiles idle).
inline int fp8_token_tile(int T, int k, int E) {
  const long long rows = (long long)T * k;
  return rows <= 8LL * E ? 16 : rows <= 24LL * E ? 32 : 64;
}

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Byte offsets of every scratch buffer inside the caller's workspace (256-byte aligned).
struct WsLayout {
  int T, N, G, TN, nblk, max_rt;
  size_t err, topk_ids, topk_w, logits, blockhist, counts, offsets, grp, rt2g, perm_tok, inv,
      row_w, xd, xexp, h, hexp, o, x_stage, out_stage, tok_stage, total;
};

WsLayout ws_layout(const moe_config& c, int T);

// K slices of the router GEMM for a batch of T tokens: few token tiles -> split K so that
// enough SMs stream the router weight; partial logits are summed in slice order by top-k.
int router_ksplit(const moe_config& c, int T);

// The configuration a plan was created with.
const moe_config* plan_config(const moe_plan* p);

// Launchers.  Each returns cudaSuccess or the launch error; none synchronises.
struct GemmLaunch {
  int epi;                 // 0 = SwiGLU dual accumulator -> bf16, 1 = fp32 (x optional row scale)
  int TN;                  // rows per row tile of the schedule (and of the kernel unless kernel_tn)
  int kernel_tn;           // 0, or a divisor of TN: the kernel splits each row tile
  // A (weights) routed / shared, B (activations) routed / shared: 2-D bf16, K innermost.
  const void* a_ptr; int64_t a_rows;
  const void* a_sh_ptr; int64_t a_sh_rows;
  const void* b_ptr; int64_t b_rows;
  const void* b_sh_ptr; int64_t b_sh_rows;
  // FP8 weights (q8 = 1): a_ptr / a_sh_ptr hold E4M3 codes and a_exp / a_sh_exp the int8
  // exponents of their 128 x 128 tiles ([mats, ceil(rows/128), ceil(K/128)])
  int q8; const int8_t* a_exp; const int8_t* a_sh_exp;
  // q8 = 2: the codes feed the MMA directly; B rows are E4M3 pieces ([rows, pieces, K] codes,
  // 2 pieces for SwiGLU, 4 for fp32) with one power-of-two exponent per row (b_exp), shared rows
  // after the routed ones in the same buffers
  const int32_t* b_exp;
  // q8 = 3: a_ptr / a_sh_ptr hold packed MXFP4 (E2M1) codes [rows, K/2], a_sub / a_sh_sub their
  // 1 x 32 sub-block exponents [rows, K/32] and a_exp / a_sh_exp the 128 x 128 tile exponents
  // (largest sub-block exponent - 6); B as for q8 = 2
  const int8_t* a_sub; const int8_t* a_sh_sub;
  int K;
  int hilo;                // activation operand is the (hi, lo) pair: B rows hold 2*K values
  int pair;                // run on CTA pairs (2-SM MMA, 256 weight rows per tile)
  int mblk;                // fp32 variant: 128-feature m-blocks per tile (1 or 2)
  int num_mblocks, a_rows_per_group, a_up_offset, out_features, out_ld;
  int out_rows;            // rows of `out` (per K slice): checked in MOE_DEBUG_BOUNDS builds, 0 = unchecked
  void* out;
  const float* row_scale;
  int n_routed, shared_b_shift;
  const int4* grp; const int* rt2g;
  int dense_rows;
  int ksplit;              // dense schedule: split K into this many slices (0 or 1: none)
  long long split_stride;  // elements between the partial outputs of consecutive slices
  int max_tiles;           // upper bound on the tile count (grid sizing)
  int* err;
  int num_sms;
};
cudaError_t launch_grouped_gemm(const GemmLaunch& L, cudaStream_t s);
int gemm_features_per_tile(int epi, int mblk);

struct TopkLaunch {
  const float* logits;     // nsplit partial [T, E] slabs, split_stride elements apart
  int nsplit; long long split_stride;
  float* logits_out;       // optional: the summed logits (only written when nsplit > 1)
  const float* bias; int T, E, k, score;
  int n_groups, topk_groups, group_topk;
  const int32_t* token_ids; const int32_t* tid2eid; int vocab;
  int32_t* topk_ids; float* topk_w; int* err;
};
cudaError_t launch_topk(const TopkLaunch& L, cudaStream_t s);

// Batches of at most ROUTER_FUSED_MAX_T tokens over at most ROUTER_FUSED_MAX_E experts run the
// router (logits and selection) as one kernel: K slices of ROUTER_FUSED_KS values on the CUDA
// cores, the last block of each group of 8 tokens summing the slices in order and selecting.
// Measured: Mixtral's 8 experts at 16 tokens 0.014 ms against 0.020 ms for the tensor-core router
// GEMM and top-k; V4-Flash's 256 at 64 tokens 0.037 against 0.028 ms (each warp's experts
// are computed in turn), hence the expert limit.  tk.logits: the partial buffer
// (router_fused_slices(d) slabs of T x E fp32, tk.split_stride apart), tk.nsplit the slice count;
// partial: that buffer, writable (tk.logits points to it too); counters: one int per group of 8
// tokens, zero before the launch (words of the workspace's error block after the error word,
// which every entry point clears).
constexpr int ROUTER_FUSED_MAX_T = 64;
constexpr int ROUTER_FUSED_MAX_E = 64;
constexpr int ROUTER_FUSED_KS = 256;
constexpr int ERR_BLOCK_BYTES = 256;       // the workspace's error block, cleared by every entry point
constexpr int ROUTER_COUNTERS_OFFSET = 64;  // bytes into the error block
static_assert(ROUTER_COUNTERS_OFFSET + (ROUTER_FUSED_MAX_T / 8) * 4 <= ERR_BLOCK_BYTES, "router counters");
inline int router_fused_slices(int d) { return (d + ROUTER_FUSED_KS - 1) / ROUTER_FUSED_KS; }
inline bool router_fused(int T, int E) { return T <= ROUTER_FUSED_MAX_T && E <= ROUTER_FUSED_MAX_E; }
struct RouterFusedLaunch {
  const void* x;    // [T, d] bf16
  const void* w_r;  // [E, d] bf16
  int T, d, E;
  float* partial;
  int* counters;
  TopkLaunch tk;
};
cudaError_t launch_router_fused(const RouterFusedLaunch& L, cudaStream_t s);

struct PermuteLaunch {
  const int32_t* topk_ids; const float* topk_w; int T, k, E, n_shared, TN, nblk;
  int32_t* blockhist; int32_t* counts; int32_t* offsets; int4* grp; int32_t* rt2g;
  int32_t* perm_tok; int32_t* inv; float* row_w; int* err;
  // optional row gather x -> xd ([N, d] bf16); skipped when xd is null
  const void* x; void* xd; int d; int num_sms;
};
cudaError_t launch_permute(const PermuteLaunch& L, cudaStream_t s);
int permute_launch_count(bool gather, long long N);  // N = T * k assignments

// Activation rows -> E4M3 pieces and one exponent per row (the B operand of the q8 = 2 GEMMs):
// bf16 rows (2 pieces; row r < n_gather is row gather[r] of src, later rows row r - n_gather)
// or fp32 rows (4 pieces, in place allowed).  K * 4 <= SPLIT_SMEM_MAX.
cudaError_t launch_split_rows_e4m3(const void* src, bool bf16_src, const int32_t* gather, int n_gather, int rows,
                                   int K, int pieces, uint8_t* dst, int32_t* exps, cudaStream_t s);
// The two-piece split of x for the dispatch, token-major: token t's pieces and exponent go to
// rows inv[t*k + j] and, with a shared expert, row N + t.
cudaError_t launch_split_tokens_e4m3(const void* x, const int32_t* inv, int T, int k, int N, int n_shared, int K,
                                     uint8_t* dst, int32_t* exps, int* err, cudaStream_t s);

struct CombineLaunch {
  const float* o; const int32_t* inv; int T, k, d, N, n_shared; void* out;
  int* err;  // MOE_DEBUG_BOUNDS builds: row checks
};
cudaError_t launch_combine(const CombineLaunch& L, cudaStream_t s);

// cuTensorMapEncodeTiled resolved through the runtime (no link-time libcuda dependency).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);
EncodeTiledFn get_encode_fn();

}  // namespace moe
