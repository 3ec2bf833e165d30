// Router epilogue: per-token scoring, optional selection bias, group-limited or hash
// selection, top-k and gate weights, from the fp32 logits the router GEMM produced.
//
//   scores   softmax | sigmoid | sqrt(softplus)     ("MoE compute and communication", sec. 二.2;
//                                                  "DeepSeek-V4 MoE", eq. dsv4-moe-softplus)
//   bias     selection key = score + b_e, weights from the unbiased score (same page, sec. 七.3)
//   groups   group score = sum of its group_topk largest keys; keep topk_groups groups
//            ("DeepSeek-V4 MoE", sec. "V3 的节点路由约束")
//   hash     ids = tid2eid[token_id]               (SGLang analysis page, sec. 二, HashTopK)
//   top-k then softmax over the selected logits  (router page, sec. "Router 的选择过程")
//
// One warp per token; expert e lives in lane e % 32, register slot e / 32 (the kernel is compiled
// for PL = 1, 2, 4, 8 or 16 slots per lane, the smallest that holds E).  Top-k is k rounds
// of a warp arg-max (larger key wins, equal keys -> lower expert id), so ids come out in
// descending key order.  All reductions use a fixed shuffle tree: results are deterministic.
#include <float.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int TOPK_WARPS = 8;
constexpr int MAX_GROUP_TOPK = 8;

__device__ __forceinline__ float score_fn(float l, int mode) {
  if (mode == MOE_SCORE_SIGMOID) return 1.0f / (1.0f + expf(-l));
  if (mode == MOE_SCORE_SQRT_SOFTPLUS) {
    const float sp = (l > 0.0f) ? l + log1pf(expf(-l)) : log1pf(expf(l));
    return sqrtf(sp);
  }
  return l;  // softmax modes are handled by the caller
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Value of register slot `i` without dynamic register indexing.
template <int PL>
__device__ __forceinline__ float pick(const float (&a)[PL], int i) {
  float v = 0.0f;
#pragma unroll
  for (int s = 0; s < PL; ++s)
    if (s == i) v = a[s];
  return v;
}

// Selection for token t by one warp: the logits (summed over the K slices), scores, bias, group
// limits or hash lookup, top-k and the gate weights, written to topk_ids / topk_w (and the summed
// logits to logits_out when given).  s_keys: PL * 32 floats of shared memory for this warp.
template <int PL>
__device__ __forceinline__ void route_token(const TopkLaunch& a, int t, float* s_keys) {
  constexpr int MAX_PER_LANE = PL;
  const int lane = threadIdx.x & 31;
  const int E = a.E, k = a.k, mode = a.score;
  const float* lrow = a.logits + (size_t)t * E;  // slab 0; slab s at + s * split_stride

  float l[MAX_PER_LANE], sc[MAX_PER_LANE], key[MAX_PER_LANE];
  // Router logits; with split-K the partial slabs are summed in slice order (slice-outer loop:
  // the loads of one slice are independent).  Plain loads: the sum may be written back over
  // slab 0 of this row.
#pragma unroll
  for (int i = 0; i < MAX_PER_LANE; ++i) {
    const int e = lane + 32 * i;
    l[i] = (e < E) ? __ldcg(lrow + e) : -INFINITY;
  }
  // G slices' loads are issued together (one memory latency per group instead of per slice);
  // the additions stay in slice order.
  constexpr int G = MAX_PER_LANE >= 16 ? 2 : MAX_PER_LANE >= 8 ? 4 : 8;
  for (int sp0 = 1; sp0 < a.nsplit; sp0 += G) {
    float pv[G][MAX_PER_LANE];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float* q = lrow + (size_t)(sp0 + g) * a.split_stride;
#pragma unroll
      for (int i = 0; i < MAX_PER_LANE; ++i) {
        const int e = lane + 32 * i;
        pv[g][i] = (sp0 + g < a.nsplit && e < E) ? __ldcg(q + e) : 0.0f;
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (sp0 + g >= a.nsplit) break;
#pragma unroll
      for (int i = 0; i < MAX_PER_LANE; ++i) l[i] += pv[g][i];
    }
  }
  if (a.logits_out != nullptr) {
#pragma unroll
    for (int i = 0; i < MAX_PER_LANE; ++i) {
      const int e = lane + 32 * i;
      if (e < E) a.logits_out[(size_t)t * E + e] = l[i];
    }
  }
  // unbiased scores (softmax_topk: the logits themselves)
  if (mode == MOE_SCORE_SOFTMAX) {
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < MAX_PER_LANE; ++i) m = fmaxf(m, l[i]);
    m = warp_max(m);
    float ex[MAX_PER_LANE], s = 0.0f;
#pragma unroll
    for (int i = 0; i < MAX_PER_LANE; ++i) {
      ex[i] = (lane + 32 * i < E) ? expf(l[i] - m) : 0.0f;
      s += ex[i];
    }
    s = warp_sum(s);
#pragma unroll
    for (int i = 0; i < MAX_PER_LANE; ++i) sc[i] = ex[i] / s;
  } else {
#pragma unroll
    for (int i = 0; i < MAX_PER_LANE; ++i) sc[i] = score_fn(l[i], mode);
  }

  int ids[MAX_TOPK];
  float sel[MAX_TOPK];   // unbiased score (or logit) of each selected expert
  if (a.tid2eid != nullptr) {
    // ---------------------------------------------------------------- HashTopK
    int tok = __ldg(a.token_ids + t);
    if (tok < 0 || tok >= a.vocab) {
      if (lane == 0) atomicOr(a.err, DEVERR_TOKEN_ID);
      tok = min(max(tok, 0), a.vocab - 1);
    }
#pragma unroll
    for (int j = 0; j < MAX_TOPK; ++j) {
      if (j < k) {
        int e = __ldg(a.tid2eid + (size_t)tok * k + j);
        if (e < 0 || e >= E) {
          if (lane == 0) atomicOr(a.err, DEVERR_TID2EID);
          e = min(max(e, 0), E - 1);
        }
        ids[j] = e;
        sel[j] = __shfl_sync(0xffffffffu, pick(sc, e >> 5), e & 31);
      }
    }
  } else {
    // ---------------------------------------------------------------- learned top-k
#pragma unroll
    for (int i = 0; i < MAX_PER_LANE; ++i) {
      const int e = lane + 32 * i;
      key[i] = (e < E) ? sc[i] + (a.bias != nullptr ? __ldg(a.bias + e) : 0.0f) : -INFINITY;
    }
    if (a.n_groups > 0) {
      const int gsz = E / a.n_groups;
#pragma unroll
      for (int i = 0; i < MAX_PER_LANE; ++i) {
        const int e = lane + 32 * i;
        if (e < E) s_keys[e] = key[i];
      }
      __syncwarp();
      float gscore = -INFINITY;
      if (lane < a.n_groups) {
        float top[MAX_GROUP_TOPK];
#pragma unroll
        for (int j = 0; j < MAX_GROUP_TOPK; ++j) top[j] = -INFINITY;
        const float* gk = &s_keys[lane * gsz];
        for (int x = 0; x < gsz; ++x) {
          float v = gk[x];
          // insert v into the descending list top[0..group_topk) (strictly larger moves up)
#pragma unroll
          for (int j = 0; j < MAX_GROUP_TOPK; ++j) {
            if (j < a.group_topk && v > top[j]) {
              const float tmp = top[j];
              top[j] = v;
              v = tmp;
            }
          }
        }
        float acc = top[0];
#pragma unroll
        for (int j = 1; j < MAX_GROUP_TOPK; ++j)
          if (j < a.group_topk) acc = acc + top[j];
        gscore = acc;
      }
      int rank = 0;
      for (int h = 0; h < a.n_groups; ++h) {
        const float o = __shfl_sync(0xffffffffu, gscore, h);
        if (o > gscore || (o == gscore && h < lane)) ++rank;
      }
      const unsigned keep = __ballot_sync(0xffffffffu, lane < a.n_groups && rank < a.topk_groups);
#pragma unroll
      for (int i = 0; i < MAX_PER_LANE; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((keep >> (e / gsz)) & 1u)) key[i] = -INFINITY;
      }
    }
    unsigned taken = 0;
#pragma unroll
    for (int j = 0; j < MAX_TOPK; ++j) {
      if (j < k) {
        float bk = -INFINITY;
        int bi = -1;
#pragma unroll
        for (int i = 0; i < MAX_PER_LANE; ++i) {
          const bool avail = (lane + 32 * i < E) && !((taken >> i) & 1u);
          if (avail && (key[i] > bk || bi < 0)) {
            bk = key[i];
            bi = i;
          }
        }
        int be = (bi >= 0) ? lane + 32 * bi : 0x7fffffff;
        if (bi < 0) bk = -INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
          const int oe = __shfl_xor_sync(0xffffffffu, be, o);
          if (ok > bk || (ok == bk && oe < be)) {
            bk = ok;
            be = oe;
          }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        ids[j] = be;
        sel[j] = __shfl_sync(0xffffffffu, pick(sc, be >> 5), be & 31);
      }
    }
  }

  // gate weights
  float w[MAX_TOPK];
  if (mode == MOE_SCORE_SOFTMAX_TOPK) {
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < MAX_TOPK; ++j)
      if (j < k) m = fmaxf(m, sel[j]);
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < MAX_TOPK; ++j)
      if (j < k) {
        w[j] = expf(sel[j] - m);
        s += w[j];
      }
#pragma unroll
    for (int j = 0; j < MAX_TOPK; ++j)
      if (j < k) w[j] = w[j] / s;
  } else {
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < MAX_TOPK; ++j)
      if (j < k) s += sel[j];
    s = fmaxf(s, 1e-30f);
#pragma unroll
    for (int j = 0; j < MAX_TOPK; ++j)
      if (j < k) w[j] = sel[j] / s;
  }
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < MAX_TOPK; ++j)
      if (j < k) {
        a.topk_ids[(size_t)t * k + j] = ids[j];
        a.topk_w[(size_t)t * k + j] = w[j];
      }
  }
}

template <int PL>
__global__ void __launch_bounds__(TOPK_WARPS * 32) topk_kernel(TopkLaunch a) {
  __shared__ float s_keys[TOPK_WARPS][PL * 32];
  const int warp = threadIdx.x >> 5;
  const int t = blockIdx.x * TOPK_WARPS + warp;
  if (t >= a.T) return;  // whole warp leaves together
  route_token<PL>(a, t, s_keys[warp]);
}

cudaError_t launch_topk(const TopkLaunch& L, cudaStream_t s) {
  static_assert(MAX_EXPERTS <= 16 * 32, "slots per lane");
  const int blocks = (L.T + TOPK_WARPS - 1) / TOPK_WARPS;
  if (L.E <= 32)
    topk_kernel<1><<<blocks, TOPK_WARPS * 32, 0, s>>>(L);
  else if (L.E <= 64)
    topk_kernel<2><<<blocks, TOPK_WARPS * 32, 0, s>>>(L);
  else if (L.E <= 128)
    topk_kernel<4><<<blocks, TOPK_WARPS * 32, 0, s>>>(L);
  else if (L.E <= 256)
    topk_kernel<8><<<blocks, TOPK_WARPS * 32, 0, s>>>(L);
  else
    topk_kernel<16><<<blocks, TOPK_WARPS * 32, 0, s>>>(L);
  return cudaGetLastError();
}

// ============================================================================ fused router (small T)
// Logits and selection in one launch for batches of at most ROUTER_FUSED_MAX_T tokens over at most
// ROUTER_FUSED_MAX_E experts, where the router GEMM is latency-bound and the tensor-core kernel's
// fixed costs and a second launch dominate.  Block (g, s) takes tokens [8 g, 8 g + 8) and the K slice
// [256 s, 256 s + 256): lane l holds K values 8 l .. 8 l + 7 of the slice of every token row,
// warp w computes the partial logits of experts w, w + 8, ... (the weight slices of eight experts
// loaded together; fp32 FMAs of the exact bf16 products, then a fixed butterfly over the lanes)
// and stores them in slab s of the partial buffer.  The block that raises the group's counter to the slice count last (release: the
// stores of every block are fenced before its increment) sums the slabs in slice order and runs
// the selection, one warp per token.  No block waits for another; the result is independent of
// which block comes last.
template <int PL>
__global__ void __launch_bounds__(256) router_fused_kernel(RouterFusedLaunch L) {
  constexpr int TOK = 8, U = 8;  // tokens per block; experts whose weight slices a warp loads at once
  static_assert(ROUTER_FUSED_KS == 32 * 8, "one 16-byte vector per lane covers a slice row");
  __shared__ float s_keys[TOK][PL * 32];
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x, slice = blockIdx.y, nslice = gridDim.y;
  const int t0 = g * TOK;
  const int ntok = min(TOK, L.T - t0);
  const int k0 = slice * ROUTER_FUSED_KS + lane * 8;       // this lane's 8 K values
  const bool act = k0 < L.d;                               // d is a multiple of 64
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(L.x);
  const __nv_bfloat16* w_r = static_cast<const __nv_bfloat16*>(L.w_r);
  float xf[TOK][8];  // the block's token rows at this lane's K values (0 past the batch)
#pragma unroll
  for (int r = 0; r < TOK; ++r) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (act && r < ntok) v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + r) * L.d + k0));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(h[j]);
      xf[r][2 * j] = f.x;
      xf[r][2 * j + 1] = f.y;
    }
  }
  float* slab = L.partial + (size_t)slice * L.tk.split_stride;
  for (int e0 = warp; e0 < L.E; e0 += TOK * U) {
    uint4 wv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int e = e0 + TOK * u;
      wv[u] = (act && e < L.E) ? __ldg(reinterpret_cast<const uint4*>(w_r + (size_t)e * L.d + k0))
                               : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int e = e0 + TOK * u;
      if (e >= L.E) break;  // the same for the whole warp
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&wv[u]);
      float wf[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(h[j]);
        wf[2 * j] = f.x;
        wf[2 * j + 1] = f.y;
      }
      float acc[TOK];
#pragma unroll
      for (int r = 0; r < TOK; ++r) {
        float a = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) a = fmaf(wf[j], xf[r][j], a);
        acc[r] = warp_sum(a);
      }
      float mine = 0.0f;
#pragma unroll
      for (int r = 0; r < TOK; ++r)
        if (lane == r) mine = acc[r];
      if (lane < ntok) slab[(size_t)(t0 + lane) * L.E + e] = mine;
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(L.counters + g, 1) == nslice - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (warp < ntok) route_token<PL>(L.tk, t0 + warp, s_keys[warp]);
}

cudaError_t launch_router_fused(const RouterFusedLaunch& L, cudaStream_t s) {
  if (L.T < 1 || L.T > ROUTER_FUSED_MAX_T || L.E > ROUTER_FUSED_MAX_E || L.d % 64 != 0) return cudaErrorInvalidValue;
  const dim3 grid((L.T + 7) / 8, router_fused_slices(L.d));
  if (L.E <= 32)
    router_fused_kernel<1><<<grid, 256, 0, s>>>(L);
  else if (L.E <= 64)
    router_fused_kernel<2><<<grid, 256, 0, s>>>(L);
  else if (L.E <= 128)
    router_fused_kernel<4><<<grid, 256, 0, s>>>(L);
  else if (L.E <= 256)
    router_fused_kernel<8><<<grid, 256, 0, s>>>(L);
  else
    router_fused_kernel<16><<<grid, 256, 0, s>>>(L);
  return cudaGetLastError();
}

}  // namespace moe
