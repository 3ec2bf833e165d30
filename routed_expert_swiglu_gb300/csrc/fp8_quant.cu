// FP8 (E4M3) expert weights with one power-of-two scale per 128 x 128 tile ("DeepSeek-V4 MoE",
// section "FP4 QAT 怎么做到反量化无损": FP8 E4M3 weights share one scale per 128 x 128 tile).
//
// For each tile of each weight matrix: amax = max |w| (exact), e = the smallest integer with
// amax <= 448 * 2^e (from frexp: amax = m * 2^x, m in [0.5, 1); e = x - 9 if m <= 0.875, else
// x - 8; 0 for an all-zero tile; at least -126), code = E4M3 round-to-nearest-even of w * 2^-e
// (exact fp32 scaling), negative zero stored as 0x00.  Dequantisation q * 2^e is exact and
// every such value is a bf16 value.  One CTA per tile; deterministic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <limits.h>

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

// ---------------------------------------------------------------------------------------------
// Activation rows as sums of E4M3 pieces, the B operand of the FP8-weight MMA kernels.
//
// Row r becomes P pieces of K codes (piece p at dst + (r * P + p) * K) and one exponent
// exps[r] = e such that row = 2^e * sum_p piece_p * 2^(-4p).  The scale 2^-e brings the row's
// largest magnitude into (224, 448] (e as for the weight tiles: the smallest integer with
// amax <= 448 * 2^e, 0 for a zero row, at least -126).  With v = value * 2^-e (exact), piece 0
// is the E4M3 rounding (nearest, ties to even) of v, and piece p the rounding of 16 times what
// the pieces before it leave: a normal E4M3 rounding leaves at most 2^-4 of its input, so each
// piece stays within the E4M3 range while the subnormal step (2^-9) of piece p sits at
// 2^(-9-4p) of v's scale.  Two pieces reproduce a bf16 value (8 significant bits) exactly when
// |v| >= 2^-6, i.e. above 2^-13.8 of the row's largest magnitude, and within 2^-14 of the scale
// (2^-21.8 of the largest magnitude) below that; four pieces keep 2^-16 of every value above the
// floor of 2^-22 of the scale (2^-29.8 of the largest magnitude).
//
// One CTA per row; the row is staged in shared memory as fp32 before any piece is written, so
// the fp32 source may be the destination itself (P = 4: a row's pieces fill exactly its fp32
// bytes).  Bf16 sources may be gathered: row r < n_gather reads row gather[r] of src, later
// rows read row r - n_gather.
constexpr int SPLIT_THREADS = 256;

template <bool BF16_SRC, int P>
__global__ void __launch_bounds__(SPLIT_THREADS) split_rows_e4m3_kernel(const void* src, const int32_t* __restrict__ gather,
                                                                        int n_gather, int K, uint8_t* dst,
                                                                        int32_t* __restrict__ exps) {
  extern __shared__ float srow[];
  __shared__ float s_max[SPLIT_THREADS / 32];
  __shared__ int s_e;
  const int r = blockIdx.x;
  float m = 0.0f;
  if (BF16_SRC) {
    const int sr = gather == nullptr ? r : (r < n_gather ? __ldg(gather + r) : r - n_gather);
    const uint4* s = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(src) + (size_t)sr * K);
    for (int i = threadIdx.x; i < K / 8; i += SPLIT_THREADS) {
      const uint4 v = __ldg(s + i);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
        srow[8 * i + 2 * j] = lo;
        srow[8 * i + 2 * j + 1] = hi;
        m = fmaxf(m, fmaxf(fabsf(lo), fabsf(hi)));
      }
    }
  } else {
    // plain loads: with an in-place split this CTA later overwrites the row
    const float4* s = reinterpret_cast<const float4*>(static_cast<const float*>(src) + (size_t)r * K);
    for (int i = threadIdx.x; i < K / 4; i += SPLIT_THREADS) {
      const float4 v = s[i];
      srow[4 * i] = v.x;
      srow[4 * i + 1] = v.y;
      srow[4 * i + 2] = v.z;
      srow[4 * i + 3] = v.w;
      m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float amax = 0.0f;
    for (int i = 0; i < SPLIT_THREADS / 32; ++i) amax = fmaxf(amax, s_max[i]);
    int e = 0;
    if (amax > 0.0f) {
      int x;
      const float mant = frexpf(amax, &x);
      e = max((mant <= 0.875f) ? x - 9 : x - 8, -126);
    }
    s_e = e;
    exps[r] = e;
  }
  __syncthreads();
  const float sc = __int_as_float((127 - s_e) << 23);  // 2^-e (e in [-126, 120])
  uint32_t* out = reinterpret_cast<uint32_t*>(dst + (size_t)r * P * K);
  for (int i = threadIdx.x; i < K / 4; i += SPLIT_THREADS) {
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = srow[4 * i + j] * sc;
#pragma unroll
    for (int pc = 0; pc < P; ++pc) {
      const __nv_fp8x2_storage_t c01 = __nv_cvt_float2_to_fp8x2(make_float2(v[0], v[1]), __NV_SATFINITE, __NV_E4M3);
      const __nv_fp8x2_storage_t c23 = __nv_cvt_float2_to_fp8x2(make_float2(v[2], v[3]), __NV_SATFINITE, __NV_E4M3);
      out[(size_t)pc * (K / 4) + i] = (uint32_t)c01 | ((uint32_t)c23 << 16);
      if (pc + 1 < P) {
        const __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2(c01, __NV_E4M3);
        const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2(c23, __NV_E4M3);
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
        const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
        // what the piece leaves, times 16 (exact: a rounding and its source lie within a factor
        // of two of each other, and the remainder is at most 2^-4 of the source or below 2^-10)
        v[0] = (v[0] - f01.x) * 16.0f;
        v[1] = (v[1] - f01.y) * 16.0f;
        v[2] = (v[2] - f23.x) * 16.0f;
        v[3] = (v[3] - f23.y) * 16.0f;
      }
    }
  }
}

// The same two-piece split of bf16 rows, token-major for the dispatch: CTA t splits x row t once
// and writes its pieces and exponent to every dispatched row that holds it -- the k routed rows
// inv[t*k + j] and, with a shared expert, row N + t -- so each x row is read and split once
// instead of once per slot.
__global__ void __launch_bounds__(SPLIT_THREADS) split_tokens_e4m3_kernel(const __nv_bfloat16* __restrict__ x,
                                                                          const int32_t* __restrict__ inv, int k,
                                                                          int N, int n_shared, int K,
                                                                          uint8_t* __restrict__ dst,
                                                                          int32_t* __restrict__ exps, int* err) {
  extern __shared__ float srow[];
  __shared__ float s_max[SPLIT_THREADS / 32];
  __shared__ int s_e;
  __shared__ int s_rows[MAX_TOPK + 1];
  const int t = blockIdx.x;
  const int nrows = k + n_shared;
  if (threadIdx.x < nrows) {
    int r = threadIdx.x < k ? __ldg(inv + (size_t)t * k + threadIdx.x) : N + t;
    if (bad_index(r, (long long)N + (long long)n_shared * gridDim.x, err)) r = -1;
    s_rows[threadIdx.x] = r;
  }
  float m = 0.0f;
  const uint4* s = reinterpret_cast<const uint4*>(x + (size_t)t * K);
  for (int i = threadIdx.x; i < K / 8; i += SPLIT_THREADS) {
    const uint4 v = __ldcs(s + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
      srow[8 * i + 2 * j] = lo;
      srow[8 * i + 2 * j + 1] = hi;
      m = fmaxf(m, fmaxf(fabsf(lo), fabsf(hi)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float amax = 0.0f;
    for (int i = 0; i < SPLIT_THREADS / 32; ++i) amax = fmaxf(amax, s_max[i]);
    int e = 0;
    if (amax > 0.0f) {
      int xe;
      const float mant = frexpf(amax, &xe);
      e = max((mant <= 0.875f) ? xe - 9 : xe - 8, -126);
    }
    s_e = e;
  }
  __syncthreads();
  if (threadIdx.x < nrows && s_rows[threadIdx.x] >= 0) exps[s_rows[threadIdx.x]] = s_e;
  const float sc = __int_as_float((127 - s_e) << 23);  // 2^-e (e in [-126, 120])
  for (int i = threadIdx.x; i < K / 4; i += SPLIT_THREADS) {
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = srow[4 * i + j] * sc;
    uint32_t code[2];
#pragma unroll
    for (int pc = 0; pc < 2; ++pc) {
      const __nv_fp8x2_storage_t c01 = __nv_cvt_float2_to_fp8x2(make_float2(v[0], v[1]), __NV_SATFINITE, __NV_E4M3);
      const __nv_fp8x2_storage_t c23 = __nv_cvt_float2_to_fp8x2(make_float2(v[2], v[3]), __NV_SATFINITE, __NV_E4M3);
      code[pc] = (uint32_t)c01 | ((uint32_t)c23 << 16);
      if (pc == 0) {
        const __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2(c01, __NV_E4M3);
        const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2(c23, __NV_E4M3);
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
        const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
        v[0] = (v[0] - f01.x) * 16.0f;  // what piece 0 leaves, times 16 (exact, as above)
        v[1] = (v[1] - f01.y) * 16.0f;
        v[2] = (v[2] - f23.x) * 16.0f;
        v[3] = (v[3] - f23.y) * 16.0f;
      }
    }
    for (int j = 0; j < nrows; ++j) {
      const int r = s_rows[j];
      if (r < 0) continue;
      uint32_t* out = reinterpret_cast<uint32_t*>(dst + (size_t)r * 2 * K);
      __stcs(out + i, code[0]);
      __stcs(out + K / 4 + i, code[1]);
    }
  }
}

cudaError_t launch_split_tokens_e4m3(const void* x, const int32_t* inv, int T, int k, int N, int n_shared, int K,
                                     uint8_t* dst, int32_t* exps, int* err, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (K % 8 != 0 || (size_t)K * 4 > SPLIT_SMEM_MAX || k > MAX_TOPK || inv == nullptr) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(split_tokens_e4m3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SPLIT_SMEM_MAX);
  if (e != cudaSuccess) return e;
  split_tokens_e4m3_kernel<<<T, SPLIT_THREADS, (size_t)K * 4, s>>>(static_cast<const __nv_bfloat16*>(x), inv, k, N,
                                                                   n_shared, K, dst, exps, err);
  return cudaGetLastError();
}

cudaError_t launch_split_rows_e4m3(const void* src, bool bf16_src, const int32_t* gather, int n_gather, int rows,
                                   int K, int pieces, uint8_t* dst, int32_t* exps, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (K % 8 != 0 || (size_t)K * 4 > SPLIT_SMEM_MAX) return cudaErrorInvalidValue;
  const size_t smem = (size_t)K * 4;
  if (bf16_src && pieces == 2) {
    auto kern = split_rows_e4m3_kernel<true, 2>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SPLIT_SMEM_MAX);
    if (e != cudaSuccess) return e;
    kern<<<rows, SPLIT_THREADS, smem, s>>>(src, gather, n_gather, K, dst, exps);
  } else if (!bf16_src && pieces == 4) {
    auto kern = split_rows_e4m3_kernel<false, 4>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SPLIT_SMEM_MAX);
    if (e != cudaSuccess) return e;
    kern<<<rows, SPLIT_THREADS, smem, s>>>(src, nullptr, 0, K, dst, exps);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------------
// MXFP4 (E2M1) weights with one power-of-two scale per 1 x 32 sub-block, and their lossless
// conversion to the FP8 tiles above ("DeepSeek-V4 MoE", section "FP4 QAT 怎么做到反量化无损":
// FP4 sub-blocks of 1 x 32, FP8 tiles of 128 x 128, the FP4 -> FP8 dequantisation lossless while
// the sub-block scales inside a tile stay within the FP8 exponent headroom).
//
// E2M1 code = sign << 3 | magnitude index, magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.  Storage:
// two consecutive codes per byte, code 2i in the low nibble of byte i of the row (the order in
// which the block-scaled MMA reads packed E2M1).  Sub-block exponent: the smallest s with
// amax <= 6 * 2^s (frexp: amax = m * 2^x, s = x - 3 if m <= 0.75 else x - 2), at least -114,
// then raised to (the largest s of its 128 x 128 tile) - 14; an all-zero sub-block takes the
// tile's largest s (-114 in an all-zero tile), so that E below is at least -120.  q * 2^t is an E4M3 value for every magnitude q iff -8 <= t <= 6, so with the
// FP8 tile exponent E = (largest s) - 6 the conversion is exact.  One CTA per 128 x 128 tile,
// two sub-blocks per thread; deterministic.
constexpr int MX_BLOCK = 32;
constexpr int MX_HEADROOM = 14;
constexpr int MX_MIN_EXP = -114;

// Round-to-nearest-even magnitude index of a (0 <= a <= 6) on the E2M1 grid: the count of grid
// midpoints below a, a midpoint counting when a passes it towards the neighbour with the even
// index (0.25 -> 0, 0.75 -> 2, 1.25 -> 2, 1.75 -> 4, 2.5 -> 4, 3.5 -> 6, 5 -> 6).
__device__ __forceinline__ uint32_t e2m1_index(float a) {
  return (uint32_t)(a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
}

__device__ __forceinline__ float e2m1_magnitude(uint32_t idx) {
  // 0, 0.5, 1, 1.5, 2, 3, 4, 6
  const float lo = (idx & 1u) ? 1.5f : 1.0f;
  const int e = (int)(idx >> 1) - 1;
  return idx < 2 ? 0.5f * (float)idx : ldexpf(lo, e);
}

__global__ void __launch_bounds__(256) quantize_mxfp4_kernel(const __nv_bfloat16* __restrict__ w, int rows, int K,
                                                             uint8_t* __restrict__ codes, int8_t* __restrict__ exps) {
  __shared__ int s_top[8];
  __shared__ int s_tile_top;
  const int kb = K / MX_BLOCK;                       // sub-blocks per row
  const int mat = blockIdx.z, r0 = blockIdx.y * QTILE, b0 = blockIdx.x * (QTILE / MX_BLOCK);
  const size_t base = (size_t)mat * rows * K;
  int fit[2];
  bool nz[2], valid[2];
  int top = INT_MIN;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int i = threadIdx.x * 2 + u;               // 512 sub-blocks: 128 rows x 4
    const int r = r0 + (i >> 2), b = b0 + (i & 3);
    valid[u] = r < rows && b < kb;
    float m = 0.0f;
    if (valid[u]) {
      const uint4* src = reinterpret_cast<const uint4*>(w + base + (size_t)r * K + (size_t)b * MX_BLOCK);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = __ldg(src + q);
        const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          m = fmaxf(m, fmaxf(fabsf(__uint_as_float(ww[j] << 16)), fabsf(__uint_as_float(ww[j] & 0xFFFF0000u))));
      }
    }
    nz[u] = m > 0.0f;
    int x = 0;
    const float mant = frexpf(nz[u] ? m : 1.0f, &x);
    fit[u] = max((mant <= 0.75f) ? x - 3 : x - 2, MX_MIN_EXP);
    if (valid[u] && nz[u]) top = max(top, fit[u]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) top = max(top, __shfl_xor_sync(0xffffffffu, top, o));
  if ((threadIdx.x & 31) == 0) s_top[threadIdx.x >> 5] = top;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = MX_MIN_EXP;  // an all-zero tile: as if its largest exponent were the minimum
    for (int i = 0; i < 8; ++i) t = max(t, s_top[i]);
    s_tile_top = t;
  }
  __syncthreads();
  const int floor_e = s_tile_top - MX_HEADROOM;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    if (!valid[u]) continue;
    const int i = threadIdx.x * 2 + u;
    const int r = r0 + (i >> 2), b = b0 + (i & 3);
    const int e = nz[u] ? max(fit[u], floor_e) : s_tile_top;
    exps[((size_t)mat * rows + r) * kb + b] = (int8_t)e;
    const uint4* src = reinterpret_cast<const uint4*>(w + base + (size_t)r * K + (size_t)b * MX_BLOCK);
    uint32_t out[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {            // 8 bf16 -> 8 codes -> one 32-bit word
      const uint4 v = __ldg(src + q);
      const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
      uint32_t word = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t bits = (j & 1) ? (ww[j >> 1] & 0xFFFF0000u) : (ww[j >> 1] << 16);
        const float val = ldexpf(__uint_as_float(bits), -e);  // exact power-of-two scaling
        const uint32_t idx = e2m1_index(fabsf(val));
        const uint32_t neg = (val < 0.0f && idx > 0) ? 1u : 0u;
        word |= (idx | (neg << 3)) << (4 * j);
      }
      out[q] = word;
    }
    *reinterpret_cast<uint4*>(codes + (base + (size_t)r * K + (size_t)b * MX_BLOCK) / 2) =
        make_uint4(out[0], out[1], out[2], out[3]);
  }
}

__global__ void __launch_bounds__(256) mxfp4_to_fp8_kernel(const uint8_t* __restrict__ codes, const int8_t* __restrict__ exps,
                                                           int rows, int K, uint8_t* __restrict__ q8,
                                                           int8_t* __restrict__ e8) {
  __shared__ int s_top[8];
  __shared__ int s_E;
  const int kb = K / MX_BLOCK;
  const int nr = (rows + QTILE - 1) / QTILE, nk = (K + QTILE - 1) / QTILE;
  const int mat = blockIdx.z, r0 = blockIdx.y * QTILE, b0 = blockIdx.x * (QTILE / MX_BLOCK);
  const size_t base = (size_t)mat * rows * K;
  int se[2];
  bool valid[2];
  int top = INT_MIN;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int i = threadIdx.x * 2 + u;
    const int r = r0 + (i >> 2), b = b0 + (i & 3);
    valid[u] = r < rows && b < kb;
    se[u] = valid[u] ? (int)exps[((size_t)mat * rows + r) * kb + b] : INT_MIN;
    top = max(top, se[u]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) top = max(top, __shfl_xor_sync(0xffffffffu, top, o));
  if ((threadIdx.x & 31) == 0) s_top[threadIdx.x >> 5] = top;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = INT_MIN;
    for (int i = 0; i < 8; ++i) t = max(t, s_top[i]);
    s_E = t - 6;
    e8[((size_t)mat * nr + blockIdx.y) * nk + blockIdx.x] = (int8_t)(t - 6);
  }
  __syncthreads();
  if (q8 == nullptr) return;  // tile exponents only
  const int E = s_E;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    if (!valid[u]) continue;
    const int i = threadIdx.x * 2 + u;
    const int r = r0 + (i >> 2), b = b0 + (i & 3);
    const size_t off = base + (size_t)r * K + (size_t)b * MX_BLOCK;
    const uint4 c = *reinterpret_cast<const uint4*>(codes + off / 2);
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
    const int t = se[u] - E;  // in [-8, 6] for exponents from moe_quantize_mxfp4
    uint32_t out[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int k = 4 * h + j;  // code k of the word
          const uint32_t idx = (cw[q] >> (4 * k)) & 7u;
          const uint32_t neg = (cw[q] >> (4 * k + 3)) & 1u;
          const float mag = ldexpf(e2m1_magnitude(idx), t);
          uint32_t b8 = (uint32_t)__nv_cvt_float_to_fp8(neg ? -mag : mag, __NV_SATFINITE, __NV_E4M3);
          if ((b8 & 0x7Fu) == 0) b8 = 0;
          word |= b8 << (8 * j);
        }
        out[2 * q + h] = word;
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(q8 + off);
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
  }
}

cudaError_t launch_quantize_mxfp4(const void* w, int n_mats, int rows, int K, uint8_t* codes, int8_t* exps,
                                  cudaStream_t s) {
  const dim3 grid((K + QTILE - 1) / QTILE, (rows + QTILE - 1) / QTILE, n_mats);
  quantize_mxfp4_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(w), rows, K, codes, exps);
  return cudaGetLastError();
}

cudaError_t launch_mxfp4_to_fp8(const uint8_t* codes, const int8_t* exps, int n_mats, int rows, int K, uint8_t* q8,
                                int8_t* e8, cudaStream_t s) {
  const dim3 grid((K + QTILE - 1) / QTILE, (rows + QTILE - 1) / QTILE, n_mats);
  mxfp4_to_fp8_kernel<<<grid, 256, 0, s>>>(codes, exps, rows, K, q8, e8);
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

extern "C" moe_status moe_quantize_mxfp4(const moe_bf16* w, int32_t n_mats, int32_t rows, int32_t K, uint8_t* codes,
                                         int8_t* exps, moe_stream_t stream) {
  if (n_mats <= 0 || rows <= 0 || K <= 0 || n_mats > 65535 || K % 32 != 0) return MOE_ERR_INVALID_ARG;
  if (w == nullptr || codes == nullptr || exps == nullptr) return MOE_ERR_INVALID_ARG;
  if ((int64_t)n_mats * rows * K >= (1ll << 40)) return MOE_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(w) & 15u) != 0 || (reinterpret_cast<uintptr_t>(codes) & 15u) != 0)
    return MOE_ERR_ALIGNMENT;
  if (moe::launch_quantize_mxfp4(w, n_mats, rows, K, codes, exps, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

extern "C" moe_status moe_mxfp4_to_fp8(const uint8_t* codes, const int8_t* exps, int32_t n_mats, int32_t rows,
                                       int32_t K, uint8_t* q8, int8_t* e8, moe_stream_t stream) {
  if (n_mats <= 0 || rows <= 0 || K <= 0 || n_mats > 65535 || K % 32 != 0) return MOE_ERR_INVALID_ARG;
  if (codes == nullptr || exps == nullptr || e8 == nullptr) return MOE_ERR_INVALID_ARG;
  if ((int64_t)n_mats * rows * K >= (1ll << 40)) return MOE_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(codes) & 15u) != 0 || (reinterpret_cast<uintptr_t>(q8) & 15u) != 0)
    return MOE_ERR_ALIGNMENT;  // (a NULL q8 passes)
  if (moe::launch_mxfp4_to_fp8(codes, exps, n_mats, rows, K, q8, e8, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
