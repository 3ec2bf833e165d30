// Definitions shared by the grouped-GEMM translation units (the bf16 kernels in
// grouped_gemm.cu, the FP8-weight kernels in fp8_gemm.cu): tile constants, the kernel parameter
// block, the tensor-map set, the device-side tile schedule, the single-CTA epilogue and the bf16
// tensor-map helper.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int BLOCK_M = 128;
constexpr int B_BOX = 16;            // rows per TMA box of the B operand
constexpr int NUM_EPI_WARPS = 8;
constexpr int NUM_THREADS = (2 + NUM_EPI_WARPS) * 32;
constexpr int SMEM_LIMIT = 232448;   // dynamic shared memory per block on sm_103a
enum { EPI_SWIGLU = 0, EPI_F32 = 1 };

struct GemmParams {
  int K;                // reduction length of the weight (A) operand, multiple of 64
  int num_mblocks;      // output-feature blocks per group (128 features, or 128*MBLK for fp32)
  int a_rows_per_group;
  int a_up_offset;      // SwiGLU: row offset of the up rows (W3) after the gate rows (W1)
  int out_features;
  int out_ld;
  int out_rows;         // rows of `out` (per K slice), checked in debug-bounds builds; 0 = unchecked
  void* out;
  const float* row_scale;
  int n_routed;
  int shared_b_shift;
  const int4* grp;      // {row_base, rows, first row tile, 0}; grp[G].z = total row tiles
  const int* rt2g;
  int n_groups_total;   // G (index of the total entry)
  int sched_tn;         // rows per row tile of the schedule (a multiple of the kernel's TN)
  int ksplit;           // dense (router) schedule only: K split into ksplit slices, slice s
                        // writing its partial result at out + s * split_stride
  long long split_stride;
  int dense_rows;
  int* err;
  // FP8 weights: int8 tile exponents [mats, exp_nr, exp_nk] of the routed (a_exp) and shared
  // (a_sh_exp) weight codes, one per 128 x 128 tile of each matrix
  const int8_t* a_exp;
  const int8_t* a_sh_exp;
  int exp_nr, exp_nk;
  // E4M3-piece activations: one power-of-two exponent per B row
  const int32_t* b_exp;
};

// Tensor maps of one launch.  The B operand has one map per box height 16 << i (i < 5), so a
// tile of n rows is loaded with at most five boxes (binary decomposition of n / 16).
constexpr int NUM_BOX_H = 5;
struct GemmMaps {
  CUtensorMap a, a_sh;
  CUtensorMap b[NUM_BOX_H], b_sh[NUM_BOX_H];
};

struct Tile {
  int g, mb, b_row, out_row, rows, n_mma;
  bool shared;
};

// Tile id -> (group, m-block, row sub-tile).  The schedule counts row tiles of sched_tn rows;
// a kernel with a smaller TN splits each into sched_tn / TN sub-tiles, some of which may be
// empty (rows <= 0): every role skips those identically.
template <int TN>
__device__ __forceinline__ Tile decode_tile(int tile, const GemmParams& p) {
  Tile t;
  const int split = p.sched_tn / TN;
  const int per_rt = p.num_mblocks * split;
  const int rt_glob = tile / per_rt;
  int row_base, rows_g, rt_start;
  if (p.grp != nullptr) {
    t.g = __ldg(p.rt2g + rt_glob);
    const int4 gi = __ldg(p.grp + t.g);
    row_base = gi.x;
    rows_g = gi.y;
    rt_start = gi.z;
  } else {
    t.g = 0;
    row_base = 0;
    rows_g = p.dense_rows;
    rt_start = 0;
  }
  const int R = ((rows_g + p.sched_tn - 1) / p.sched_tn) * split;
  const int local = tile - rt_start * per_rt;
  t.mb = local / R;
  const int rt = local - t.mb * R;
  t.rows = min(TN, rows_g - rt * TN);
  t.n_mma = max(16, (t.rows + 15) & ~15);
  t.out_row = row_base + rt * TN;
  t.shared = (p.grp != nullptr) && (t.g == p.n_routed);
  t.b_row = t.out_row + (t.shared ? p.shared_b_shift : 0);
  return t;
}

// Epilogue of one tile of the single-CTA kernels, run by each of the 8 epilogue warps on its TMEM
// lane quadrant (`quad`) and its half of the 16-column chunks (`half`): SwiGLU -> the bf16
// (hi, lo) activation pair, fp32 -> O rows (x optional row scale).  tq = the quadrant's address
// in the tile's accumulator buffer.
template <int EPI, int TN, int NACC, int FEATS>
__device__ __forceinline__ void epilogue_tile(const Tile& t, const GemmParams& p, uint32_t tq, int quad, int half,
                                              int lane, long long out_shift) {
  const int nchunk = (t.rows + 15) >> 4;
  if (EPI == EPI_SWIGLU) {
    const int feat = t.mb * BLOCK_M + quad * 32 + lane;
    // h is stored as an unevaluated pair hi + lo of bf16 values: hi = bf16(h),
    // lo = bf16(h - hi), so the down projection sees h to ~16 significant bits.  Within
    // each 64-feature block, hi occupies columns [128*b, 128*b + 64) and lo the next 64.
    const int col = ((feat >> 6) << 7) + (feat & 63);
    const bool fvalid = feat < p.out_features;
    for (int ci = half; ci < nchunk; ci += 2) {
      const int c0 = ci * 16;
      uint32_t rg[16], ru[16];
      tmem_ld16(tq + c0, rg);
      tmem_ld16(tq + TN + c0, ru);
      tmem_ld_wait();
      reg_fence16(rg);
      reg_fence16(ru);
      const int nr = min(16, t.rows - c0);
      if (fvalid && !(p.out_rows > 0 && (bad_index(t.out_row + c0, p.out_rows, p.err) ||
                                         bad_index(t.out_row + c0 + nr - 1, p.out_rows, p.err)))) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + (size_t)(t.out_row + c0) * p.out_ld + col;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (j < nr) {
            const float g = __uint_as_float(rg[j]);
            const float u = __uint_as_float(ru[j]);
            const float h = __fdividef(g, 1.0f + __expf(-g)) * u;
            const __nv_bfloat16 hi = __float2bfloat16_rn(h);
            const __nv_bfloat16 lo = __float2bfloat16_rn(h - __bfloat162float(hi));
            out[(size_t)j * p.out_ld] = hi;
            out[(size_t)j * p.out_ld + 64] = lo;
          }
        }
      }
    }
  } else {
    const bool scaled = (p.row_scale != nullptr) && !t.shared;
    for (int w = half; w < NACC * nchunk; w += 2) {
      const int a = w / nchunk;
      const int c0 = (w - a * nchunk) * 16;
      const int feat = t.mb * FEATS + a * BLOCK_M + quad * 32 + lane;
      uint32_t r[16];
      tmem_ld16(tq + a * TN + c0, r);
      tmem_ld_wait();
      reg_fence16(r);
      const int nr = min(16, t.rows - c0);
      if (feat < p.out_features && !(p.out_rows > 0 && (bad_index(t.out_row + c0, p.out_rows, p.err) ||
                                                        bad_index(t.out_row + c0 + nr - 1, p.out_rows, p.err)))) {
        float* out = static_cast<float*>(p.out) + out_shift + (size_t)(t.out_row + c0) * p.out_ld + feat;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (j < nr) {
            const float sc = scaled ? __ldg(p.row_scale + t.out_row + c0 + j) : 1.0f;
            out[(size_t)j * p.out_ld] = __uint_as_float(r[j]) * sc;
          }
        }
      }
    }
  }
}

// 2-D bf16 tensor [rows, cols] (cols innermost, contiguous), box bk x box_rows, swizzle of
// 2*bk bytes (bk = 64: 128-byte, bk = 32: 64-byte).
inline bool make_tmap(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_rows, int bk) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)bk, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, bk == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// E4M3 weight codes: 2-D uint8 [rows, cols] with boxes of box_k codes x box_rows rows, and the
// gate/up 3-D view (cols, d_ff, 2*groups) with boxes (box_k, 128, 2).  box_k = 64: 64-byte
// swizzle, so that the converter warps' row-wise 16-byte reads spread over all banks; box_k =
// 128: 128-byte swizzle, the K-major layout the 8-bit MMA reads.
inline bool make_tmap_u8(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_rows, int box_k = 64) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols};
  cuuint32_t box[2] = {(cuuint32_t)box_k, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, box_k == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool make_tmap_u8_gateup(CUtensorMap* m, const void* ptr, int64_t groups, int64_t d_ff, int64_t cols,
                                int box_k = 64, int box_rows = BLOCK_M) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)d_ff, (cuuint64_t)(2 * groups)};
  cuuint64_t strides[2] = {(cuuint64_t)cols, (cuuint64_t)(d_ff * cols)};
  cuuint32_t box[3] = {(cuuint32_t)box_k, (cuuint32_t)box_rows, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, box_k == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E4M3 activation pieces [rows, pieces, K]: 3-D view (K, pieces, rows) with boxes of
// (128, 1, box_rows), i.e. box_rows rows of 128 codes of one piece, 128-byte swizzle.
inline bool make_tmap_pieces(CUtensorMap* m, const void* ptr, int64_t rows, int pieces, int64_t K, int box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)pieces, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)K, (cuuint64_t)(pieces * K)};
  cuuint32_t box[3] = {128, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MXFP4 codes, two E2M1 codes per byte (code 2i in the low nibble of byte i), row-major [rows,
// K]: each group of 16 codes (8 bytes) lands in the low half of a 16-byte chunk of shared memory
// (CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B), the form the block-scaled MMA reads; boxes of 128
// codes (one 128-byte row of shared memory) x box_rows rows, 128-byte swizzle.  The gate/up view
// is 3-D (K, d_ff, 2*groups) with boxes (128, 128, 2).  The type wants K a multiple of 128,
// row strides a multiple of 32 bytes and a 32-byte aligned base.
inline bool make_tmap_e2m1(CUtensorMap* m, const void* ptr, int64_t rows, int64_t K, int box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
  cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool make_tmap_e2m1_gateup(CUtensorMap* m, const void* ptr, int64_t groups, int64_t d_ff, int64_t K,
                                  int box_rows = BLOCK_M) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)d_ff, (cuuint64_t)(2 * groups)};
  cuuint64_t strides[2] = {(cuuint64_t)(K / 2), (cuuint64_t)(d_ff * K / 2)};
  cuuint32_t box[3] = {128, (cuuint32_t)box_rows, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The FP8-weight grouped GEMMs (fp8_gemm.cu) for a launch with L.q8 set: 1 = codes widened to
// bf16 in Tensor Memory, 2 = codes straight into the 8-bit MMA with E4M3-piece activations.
cudaError_t launch_fp8_gemm(const GemmLaunch& L, GemmParams p, int kernel_tn, cudaStream_t s);

// The block-scaled CTA-pair GEMMs (bs_pair_gemm.cu) for FP8 (q8 = 2) or MXFP4 (q8 = 3) weights at
// prefill: codes and their scales into the 2-SM block-scaled MMA, E4M3-piece activations.
cudaError_t launch_bs_pair_gemm(const GemmLaunch& L, GemmParams p, cudaStream_t s);

}  // namespace moe
