// Combine: y_t = sum_{j<k} O[inv[t*k+j]] + O_shared[t], accumulated in fp32 in slot order and
// rounded once to bf16 ("Mixture of Experts: router, token dispatch, grouped GEMM", section
// "Token Combine": every position's weighted output is added into its token's row; "MoE compute
// and communication", sec. 二.2: the shared expert is added with weight 1).  The gate weight is
// already applied by the down-projection epilogue, so this is a pure gather-sum: a token's row is
// one block's (small batches: split over up to four blocks by columns), no atomics, fixed order
// -> bitwise deterministic.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {

__global__ void __launch_bounds__(256) combine_kernel(const float4* __restrict__ o, const int32_t* __restrict__ inv,
                                                      int k, int d4, int N, int n_shared, uint2* __restrict__ out,
                                                      int T, int* err) {
  __shared__ int rows[MAX_TOPK + 1];
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    const int r = __ldg(inv + (size_t)t * k + threadIdx.x);
    // debug-bounds builds: a routed row outside [0, N) is reported and left out of the sum
    rows[threadIdx.x] = bad_index(r, N, err) ? -1 : r;
  }
  if (threadIdx.x == 0 && n_shared) rows[k] = N + t;
  __syncthreads();
  const int nr = k + n_shared;
  for (int c = blockIdx.y * blockDim.x + threadIdx.x; c < d4; c += gridDim.y * blockDim.x) {
    // every slot's load issued before the additions, which stay in slot order
    float4 v[MAX_TOPK + 1];
#pragma unroll
    for (int j = 0; j < MAX_TOPK + 1; ++j)
      if (j < nr && !(MOE_DEBUG_BOUNDS && rows[j] < 0)) v[j] = __ldg(o + (size_t)rows[j] * d4 + c);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < MAX_TOPK + 1; ++j) {
      if (j >= nr) break;
      if (MOE_DEBUG_BOUNDS && rows[j] < 0) continue;
      acc.x += v[j].x;
      acc.y += v[j].y;
      acc.z += v[j].z;
      acc.w += v[j].w;
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&lo);
    packed.y = *reinterpret_cast<uint32_t*>(&hi);
    out[(size_t)t * d4 + c] = packed;
  }
}

cudaError_t launch_combine(const CombineLaunch& L, cudaStream_t s) {
  const int d4 = L.d / 4;
  // small batches: a token's columns over up to four blocks, so that more SMs take part
  const int split = std::max(1, std::min(std::min(4, d4 / 256), 512 / std::max(L.T, 1)));
  combine_kernel<<<dim3(L.T, split), 256, 0, s>>>(static_cast<const float4*>(static_cast<const void*>(L.o)), L.inv, L.k, d4, L.N,
                                     L.n_shared, static_cast<uint2*>(L.out), L.T, L.err);
  return cudaGetLastError();
}

}  // namespace moe
