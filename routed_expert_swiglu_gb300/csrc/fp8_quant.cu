// FP8 (E4M3) expert weights with one power-of-two scale per 128 x 128 tile ("DeepSeek-V4 MoE",
// section "FP4 QAT 怎么做到反量化无损": FP8 E4M3 weights share one scale per 128 x 128 tile).
//
// For each tile of each weight matrix: amax = max |w| (exact), e = the smallest integer with
// amax <= 448 * 2^e (from frexp: amax = m * 2^x, m in [0.5, 1); e = x - 9 if m <= 0.875, else
// x - 8; 0 for an all-zero tile; at least -126), code = E4M3 round-to-nearest-even of w * 2^-e
// (exact fp32 scaling), negative zero stored as 0x00.  Dequantisation q * 2^e is exact and
// every such value is a bf16 value.  One CTA per tile; deterministic.
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int QTILE = 128;

__global__ void __launch_bounds__(256) quantize_fp8_kernel(const __nv_bfloat16* __restrict__ w, int rows, int K,
                                                           uint8_t* __restrict__ codes, int8_t* __restrict__ exps) {
  __shared__ float s_max[8];
  __shared__ int s_e;
  const int nr = (rows + QTILE - 1) / QTILE, nk = (K + QTILE - 1) / QTILE;
  const int mat = blockIdx.z, ti = blockIdx.y, tj = blockIdx.x;
  const int r0 = ti * QTILE, c0 = tj * QTILE;
  const int nrows = min(QTILE, rows - r0), ncols = min(QTILE, K - c0);
  const size_t base = (size_t)mat * rows * K;
  // pass 1: amax of the tile (each thread: one column pair per row step)
  float m = 0.0f;
  for (int i = threadIdx.x; i < nrows * QTILE; i += blockDim.x) {
    const int r = i / QTILE, c = i % QTILE;
    if (c < ncols) m = fmaxf(m, fabsf(__bfloat162float(w[base + (size_t)(r0 + r) * K + c0 + c])));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float amax = 0.0f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) amax = fmaxf(amax, s_max[i]);
    int e = 0;
    if (amax > 0.0f) {
      int x;
      const float mant = frexpf(amax, &x);
      e = (mant <= 0.875f) ? x - 9 : x - 8;
      e = max(e, -126);
    }
    s_e = e;
    exps[((size_t)mat * nr + ti) * nk + tj] = (int8_t)e;
  }
  __syncthreads();
  const int e = s_e;
  // pass 2: codes
  for (int i = threadIdx.x; i < nrows * QTILE; i += blockDim.x) {
    const int r = i / QTILE, c = i % QTILE;
    if (c < ncols) {
      const size_t idx = base + (size_t)(r0 + r) * K + c0 + c;
      const float v = ldexpf(__bfloat162float(w[idx]), -e);
      uint8_t q = (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
      if ((q & 0x7F) == 0) q = 0;
      codes[idx] = q;
    }
  }
}

cudaError_t launch_quantize_fp8(const void* w, int n_mats, int rows, int K, uint8_t* codes, int8_t* exps,
                                cudaStream_t s) {
  const dim3 grid((K + QTILE - 1) / QTILE, (rows + QTILE - 1) / QTILE, n_mats);
  quantize_fp8_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(w), rows, K, codes, exps);
  return cudaGetLastError();
}

}  // namespace moe

extern "C" moe_status moe_quantize_fp8(const moe_bf16* w, int32_t n_mats, int32_t rows, int32_t K, uint8_t* codes,
                                       int8_t* exps, moe_stream_t stream) {
  if (n_mats <= 0 || rows <= 0 || K <= 0 || n_mats > 65535) return MOE_ERR_INVALID_ARG;
  if (w == nullptr || codes == nullptr || exps == nullptr) return MOE_ERR_INVALID_ARG;
  if ((int64_t)n_mats * rows * K >= (1ll << 40)) return MOE_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(w) & 1u) != 0) return MOE_ERR_ALIGNMENT;
  if (moe::launch_quantize_fp8(w, n_mats, rows, K, codes, exps, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
