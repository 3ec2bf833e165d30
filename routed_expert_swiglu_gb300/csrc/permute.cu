// Token dispatch: token-major assignments -> expert-major rows, with the inverse map kept
// ("Mixture of Experts: router, token dispatch, grouped GEMM", section "Token Dispatch":
// permuted_token_ids, tokens_per_expert; SGLang analysis page, sec. 三/四: the mapping back to
// each token's output row must be kept).
//
// Assignment i = t*k + j.  Rows are ordered by expert and, inside an expert, by i.  Integer
// only, so the result is exact and independent of scheduling:
//   1. hist     per-chunk expert histograms (chunk = 1024 consecutive assignments)
//               (a batch of one chunk runs steps 1 to 3 in one block: permute_small_kernel)
//   2. scan     per-expert prefix over chunks, exclusive scan over experts (offsets), and the
//               grouped-GEMM schedule: row tiles per group and the row-tile -> group map
//   3. scatter  rank inside the chunk from warp match masks + per-warp prefix, so row =
//               offset of the expert + its rows in earlier chunks + warp prefix + rank among
//               equal ids in the warp
//   4. rows     X_dispatch rows, 16-byte vectors: token-major X_dispatch[inv[t*k + j]] = x[t]
//               (each x row read once) for large batches, row-major by perm_tok for small ones
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {

// Batches of at least this many tokens copy the dispatched rows token-major (one warp per token
// keeps every SM busy from here on).
constexpr int DISPATCH_TOKEN_MAJOR_MIN_T = 1024;

__device__ __forceinline__ int clamp_expert(int e, int E, int* err) {
  if (e < 0 || e >= E) {
    atomicOr(err, DEVERR_TOPK_ID);
    e = min(max(e, 0), E - 1);
  }
  return e;
}

__global__ void __launch_bounds__(256) hist_kernel(const int32_t* __restrict__ ids, int N, int E,
                                                   int32_t* __restrict__ blockhist, int* err) {
  __shared__ int h[MAX_EXPERTS];
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
  const int base = blockIdx.x * PERMUTE_CHUNK;
  const int end = min(base + PERMUTE_CHUNK, N);
  for (int i = base + threadIdx.x; i < end; i += blockDim.x) atomicAdd(&h[clamp_expert(__ldg(ids + i), E, err)], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) blockhist[(size_t)blockIdx.x * E + e] = h[e];
}

// Exclusive scan of one int per thread over a block of exactly 1024 threads.
__device__ __forceinline__ int block_excl_scan(int v, int* s_warp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  const int prefix = (warp > 0) ? s_warp[warp - 1] : 0;
  total = s_warp[31];
  __syncthreads();
  return prefix + x - v;
}

__global__ void __launch_bounds__(1024) scan_kernel(int32_t* __restrict__ blockhist, int nblk, int E, int n_shared,
                                                    int T, int N, int TN, int32_t* __restrict__ counts,
                                                    int32_t* __restrict__ offsets, int4* __restrict__ grp,
                                                    int32_t* __restrict__ rt2g) {
  __shared__ int s_warp[32];
  const int e = threadIdx.x;
  int cnt = 0;
  if (e < E) {
    // blockhist[b][e] <- rows of expert e in chunks before b (eight loads in flight per step)
    for (int b0 = 0; b0 < nblk; b0 += 8) {
      int c[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) c[u] = (b0 + u < nblk) ? blockhist[(size_t)(b0 + u) * E + e] : 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (b0 + u < nblk) blockhist[(size_t)(b0 + u) * E + e] = cnt;
        cnt += c[u];
      }
    }
  }
  int total_rows;
  const int off = block_excl_scan(cnt, s_warp, total_rows);
  if (e < E) {
    counts[e] = cnt;
    offsets[e] = off;
  }
  if (e == 0) offsets[E] = total_rows;
  // grouped-GEMM schedule: groups 0..E-1 routed, group E shared (rows N .. N+T-1)
  const int G = E + n_shared;
  int rows = 0, row_base = 0;
  if (e < E) {
    rows = cnt;
    row_base = off;
  } else if (e < G) {
    rows = T;
    row_base = N;
  }
  const int R = (rows + TN - 1) / TN;
  int total_rt;
  const int rt_start = block_excl_scan(R, s_warp, total_rt);
  if (e < G) {
    grp[e] = make_int4(row_base, rows, rt_start, 0);
    for (int j = 0; j < R; ++j) rt2g[rt_start + j] = e;
  }
  if (e == 0) grp[G] = make_int4(0, 0, total_rt, 0);
}

__global__ void __launch_bounds__(PERMUTE_CHUNK) scatter_kernel(const int32_t* __restrict__ ids,
                                                                const float* __restrict__ w, int N, int k, int E,
                                                                const int32_t* __restrict__ blockbase,
                                                                const int32_t* __restrict__ offsets,
                                                                int32_t* __restrict__ perm_tok,
                                                                int32_t* __restrict__ inv, float* __restrict__ row_w,
                                                                int* err) {
  extern __shared__ int wcnt[];  // [32 warps][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int x = threadIdx.x; x < 32 * E; x += blockDim.x) wcnt[x] = 0;
  __syncthreads();
  const int i = blockIdx.x * PERMUTE_CHUNK + threadIdx.x;
  const bool valid = i < N;
  const int e = valid ? clamp_expert(__ldg(ids + i), E, err) : -1;
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  if (valid && rank == 0) wcnt[warp * E + e] = __popc(peers);
  __syncthreads();
  for (int x = threadIdx.x; x < E; x += blockDim.x) {
    int run = 0;
    for (int v = 0; v < 32; ++v) {
      const int c = wcnt[v * E + x];
      wcnt[v * E + x] = run;
      run += c;
    }
  }
  __syncthreads();
  if (valid) {
    const int row = __ldg(offsets + e) + blockbase[(size_t)blockIdx.x * E + e] + wcnt[warp * E + e] + rank;
    if (bad_index(row, N, err)) return;
    if (perm_tok) perm_tok[row] = i / k;
    if (inv) inv[i] = row;
    if (row_w) row_w[row] = __ldg(w + i);
  }
}

// Steps 1 to 3 in one block for a batch of at most one chunk of assignments (decode sizes): the
// same integer arithmetic as hist + scan + scatter with a single chunk (no earlier chunks), in one
// launch instead of three.  Expert counts come from the per-warp match counts, the offsets and the
// schedule from the block scan over experts.
__global__ void __launch_bounds__(PERMUTE_CHUNK) permute_small_kernel(
    const int32_t* __restrict__ ids, const float* __restrict__ w, int N, int k, int E, int n_shared, int T, int TN,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int4* __restrict__ grp, int32_t* __restrict__ rt2g,
    int32_t* __restrict__ perm_tok, int32_t* __restrict__ inv, float* __restrict__ row_w, int* err) {
  extern __shared__ int wcnt[];  // [32 warps][E], then the per-expert totals / offsets [E]
  __shared__ int s_warp[32];
  int* tot = wcnt + 32 * E;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int x = threadIdx.x; x < 32 * E; x += blockDim.x) wcnt[x] = 0;
  __syncthreads();
  const int i = threadIdx.x;
  const bool valid = i < N;
  const int e = valid ? clamp_expert(__ldg(ids + i), E, err) : -1;
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  if (valid && rank == 0) wcnt[warp * E + e] = __popc(peers);
  __syncthreads();
  for (int x = threadIdx.x; x < E; x += blockDim.x) {
    int run = 0;
    for (int v = 0; v < 32; ++v) {
      const int c = wcnt[v * E + x];
      wcnt[v * E + x] = run;
      run += c;
    }
    tot[x] = run;
  }
  __syncthreads();
  // expert-level scan and the grouped-GEMM schedule, thread g = group g (as in scan_kernel)
  const int g = threadIdx.x;
  const int cnt = g < E ? tot[g] : 0;
  int total_rows;
  const int off = block_excl_scan(cnt, s_warp, total_rows);
  if (g < E) {
    counts[g] = cnt;
    offsets[g] = off;
  }
  if (g == 0) offsets[E] = total_rows;
  const int G = E + n_shared;
  int rows = 0, row_base = 0;
  if (g < E) {
    rows = cnt;
    row_base = off;
  } else if (g < G) {
    rows = T;
    row_base = N;
  }
  const int R = (rows + TN - 1) / TN;
  int total_rt;
  const int rt_start = block_excl_scan(R, s_warp, total_rt);
  if (g < G) {
    grp[g] = make_int4(row_base, rows, rt_start, 0);
    for (int j = 0; j < R; ++j) rt2g[rt_start + j] = g;
  }
  if (g == 0) grp[G] = make_int4(0, 0, total_rt, 0);
  if (g < E) tot[g] = off;  // only thread g read tot[g] as a count, above
  __syncthreads();
  if (valid) {
    const int row = tot[e] + wcnt[warp * E + e] + rank;
    if (bad_index(row, N, err)) return;
    if (perm_tok) perm_tok[row] = i / k;
    if (inv) inv[i] = row;
    if (row_w) row_w[row] = __ldg(w + i);
  }
}

// X_dispatch[row] = x[perm_tok[row]]: row-major, one warp per row, 8 x 16 bytes per lane in
// flight.  Used for small batches, where one warp per token would leave most SMs idle.
__global__ void __launch_bounds__(256) gather_rows_kernel(const int4* __restrict__ x, int4* __restrict__ xd,
                                                          const int32_t* __restrict__ perm_tok, int N,
                                                          int vec_per_row, int T, int* err) {
  constexpr int U = 8;
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < N; r += nwarps) {
    const int tok = __ldg(perm_tok + r);
    if (bad_index(tok, T, lane == 0 ? err : nullptr)) continue;
    const int4* src = x + (size_t)tok * vec_per_row;
    int4* dst = xd + (size_t)r * vec_per_row;
    for (int v0 = 0; v0 < vec_per_row; v0 += 32 * U) {
      int4 buf[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < vec_per_row) buf[u] = __ldg(src + v);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < vec_per_row) __stcs(dst + v, buf[u]);
      }
    }
  }
}

// X_dispatch[inv[t*k + j]] = x[t] for every slot j of token t: token-major, so each row of x is
// read once (it would be re-read k times by a row-major gather, from DRAM once x outgrows L2)
// and written to its k rows with evict-first stores.  One warp per token, 8 x 16 bytes per lane
// in flight.
__global__ void __launch_bounds__(256) dispatch_rows_kernel(const int4* __restrict__ x, int4* __restrict__ xd,
                                                            const int32_t* __restrict__ inv, int T, int k,
                                                            int vec_per_row, int* err) {
  constexpr int U = 8;
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += nwarps) {
    const int my_row = lane < k ? __ldg(inv + (size_t)t * k + lane) : 0;
    const int4* src = x + (size_t)t * vec_per_row;
    for (int v0 = 0; v0 < vec_per_row; v0 += 32 * U) {
      int4 buf[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < vec_per_row) buf[u] = __ldcs(src + v);
      }
#pragma unroll
      for (int j = 0; j < MAX_TOPK; ++j) {
        if (j < k) {
          const int row = __shfl_sync(0xffffffffu, my_row, j);
          if (bad_index(row, (long long)T * k, lane == 0 ? err : nullptr)) continue;
          int4* dst = xd + (size_t)row * vec_per_row;
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int v = v0 + u * 32 + lane;
            if (v < vec_per_row) __stcs(dst + v, buf[u]);
          }
        }
      }
    }
  }
}

int permute_launch_count(bool gather, long long N) { return (N <= PERMUTE_CHUNK ? 1 : 3) + (gather ? 1 : 0); }

cudaError_t launch_permute(const PermuteLaunch& L, cudaStream_t s) {
  const int N = L.T * L.k;
  cudaError_t e;
  if (N <= PERMUTE_CHUNK) {
    const int smem = 33 * L.E * (int)sizeof(int);
    if (smem > 48 * 1024) {
      e = cudaFuncSetAttribute(permute_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
    }
    permute_small_kernel<<<1, PERMUTE_CHUNK, smem, s>>>(L.topk_ids, L.topk_w, N, L.k, L.E, L.n_shared, L.T, L.TN,
                                                         L.counts, L.offsets, L.grp, L.rt2g, L.perm_tok, L.inv,
                                                         L.row_w, L.err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  } else {
    hist_kernel<<<L.nblk, 256, 0, s>>>(L.topk_ids, N, L.E, L.blockhist, L.err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    scan_kernel<<<1, 1024, 0, s>>>(L.blockhist, L.nblk, L.E, L.n_shared, L.T, N, L.TN, L.counts, L.offsets, L.grp,
                                   L.rt2g);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int smem = 32 * L.E * (int)sizeof(int);
    if (smem > 48 * 1024) {
      e = cudaFuncSetAttribute(scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
    }
    scatter_kernel<<<L.nblk, PERMUTE_CHUNK, smem, s>>>(L.topk_ids, L.topk_w, N, L.k, L.E, L.blockhist, L.offsets,
                                                        L.perm_tok, L.inv, L.row_w, L.err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (L.xd != nullptr) {
    const int vec = L.d / 8;
    const int cap = L.num_sms * 8;
    if (L.T >= DISPATCH_TOKEN_MAJOR_MIN_T) {
      if (L.inv == nullptr) return cudaErrorInvalidValue;  // the token-major copy goes by the inverse map
      const int blocks = std::min((L.T + 7) / 8, cap);
      dispatch_rows_kernel<<<blocks, 256, 0, s>>>(static_cast<const int4*>(L.x), static_cast<int4*>(L.xd), L.inv,
                                                  L.T, L.k, vec, L.err);
    } else {
      const int blocks = std::min((N + 7) / 8, cap);
      gather_rows_kernel<<<blocks, 256, 0, s>>>(static_cast<const int4*>(L.x), static_cast<int4*>(L.xd),
                                                L.perm_tok, N, vec, L.T, L.err);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace moe
