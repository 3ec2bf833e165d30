// Grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMEM), fed by TMA.
//
// One persistent kernel serves the three dense contractions of the layer:
//   * router      logits[t, e]  = sum_i x[t, i] W_r[e, i]                       (fp32 out)
//   * gate/up     H[r, j]       = SiLU(sum_i X[r,i] W1_e[j,i]) * sum_i X[r,i] W3_e[j,i]  (bf16 out)
//   * down        O[r, c]       = g_r * sum_j H[r, j] W2_e[c, j]                 (fp32 out)
// ("Mixture of Experts: router, token dispatch, grouped GEMM", section "为什么不能一个一个
// GEMM 地算": many GEMMs with different weights and different row counts M, same K/N, one
// launch that schedules their tiles across SMs.)
//
// Layout: weights are the MMA's A operand (M = 128 output features per tile), the token rows
// of one group are the B operand (N = up to TN rows, rounded up to 16).  Each tile therefore
// streams a 128-row weight slab exactly once and reuses it for every token row of its group,
// which is what the weight-bandwidth-bound MoE layer needs.  D = A * B^T lands in TMEM with one
// lane per output feature and one column per token row.
//
// Warp roles (320 threads): warp 0 = TMA producer, warp 1 = TMEM owner + MMA issuer,
// warps 2..9 = epilogue (two warps per TMEM lane quadrant, splitting the columns).
// Tiles: for group g with R_g = ceil(rows_g / TN) row tiles, tile ids run m-block-major
// (all row tiles of one weight slab are adjacent, so a slab re-read hits L2).
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
  // gathered B (pair gate/up): routed row r of a group is row b_idx[r] of b_x ([*, b_ld] bf16),
  // a shared-expert row r is row r + shared_b_shift of b_x
  const __nv_bfloat16* b_x;
  const int32_t* b_idx;
  int b_ld;
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

// Compile-time shape of one kernel variant.
//   EPI_SWIGLU: A = gate and up slabs of 128 features each, one B tile, two accumulators.
//   EPI_F32:    A = MBLK slabs of 128 features, MBLK accumulators; with HILO the B operand
//               is the activation pair (hi, lo), both multiplied by the same A tile.
//   BK:         K elements per pipeline stage: 64 (128-byte swizzle rows) or 32 (64-byte).
template <int EPI, int TN, int MBLK, bool HILO, int BK>
struct GemmShape {
  static constexpr int BLOCK_K = BK;
  static constexpr int ROW_BYTES = BK * 2;
  static constexpr int A_BYTES = BLOCK_M * BLOCK_K * 2;
  static constexpr int NUM_A = (EPI == EPI_SWIGLU) ? 2 : MBLK;
  static constexpr int NUM_B = HILO ? 2 : 1;
  static constexpr int B_BYTES = TN * BLOCK_K * 2;
  static constexpr int STAGE_BYTES = NUM_A * A_BYTES + NUM_B * B_BYTES;
  static constexpr int NACC = NUM_A;                 // accumulators per buffer, TN columns each
  static constexpr int ACC_COLS = NACC * TN;
  static constexpr int NUM_BUF = (2 * ACC_COLS <= 512) ? 2 : 1;
  static constexpr int USED_COLS = NUM_BUF * ACC_COLS;
  static constexpr int TMEM_COLS = USED_COLS <= 32 ? 32 : USED_COLS <= 64 ? 64 : USED_COLS <= 128 ? 128
                                   : USED_COLS <= 256 ? 256 : 512;
  static constexpr int STAGES_FIT = (SMEM_LIMIT - 1024 - 256) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /* alignment slack */ + 256 /* barriers */;
  static constexpr int FEATS = (EPI == EPI_SWIGLU) ? BLOCK_M : BLOCK_M * MBLK;  // features per tile
  static_assert(USED_COLS <= 512, "TMEM holds 512 columns");
  static_assert(TN % B_BOX == 0 && TN <= 256, "token tile");
  static_assert(STAGES >= 2, "pipeline needs two stages");
  static_assert(EPI == EPI_F32 || (MBLK == 1 && !HILO), "SwiGLU variant");
  static_assert(BK == 64 || BK == 32, "stage K");
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
      if (fvalid) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + (size_t)(t.out_row + c0) * p.out_ld + col;
        const int nr = min(16, t.rows - c0);
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
      if (feat < p.out_features) {
        float* out = static_cast<float*>(p.out) + out_shift + (size_t)(t.out_row + c0) * p.out_ld + feat;
        const int nr = min(16, t.rows - c0);
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

template <int EPI, int TN, int MBLK, bool HILO, int BK>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmParams p) {
  using S = GemmShape<EPI, TN, MBLK, HILO, BK>;
  constexpr int BLOCK_K = S::BLOCK_K;
  constexpr int STAGES = S::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * S::STAGE_BYTES);
  // bars: full[STAGES], empty[STAGES], acc_full[2], acc_empty[2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto accf_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto acce_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf_bar(a), 1);
      mbar_init(acce_bar(a), NUM_EPI_WARPS);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.a);
    tma_prefetch_desc(&maps.a_sh);
    for (int i = 0; i < NUM_BOX_H; ++i) {
      if ((16 << i) <= TN) {
        tma_prefetch_desc(&maps.b[i]);
        tma_prefetch_desc(&maps.b_sh[i]);
      }
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), S::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  int total_tiles;
  if (p.grp != nullptr) {
    total_tiles = __ldg(&p.grp[p.n_groups_total].z) * p.num_mblocks * (p.sched_tn / TN);
  } else {
    total_tiles = ((p.dense_rows + p.sched_tn - 1) / p.sched_tn) * p.num_mblocks * (p.sched_tn / TN);
  }
  // split-K (dense schedule only): tile id = base tile * ksplit + slice
  const int ksplit = p.ksplit;
  total_tiles *= ksplit;
  const int KBS = p.K / BLOCK_K / ksplit;  // k-blocks per slice

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        const Tile t = decode_tile<TN>(tile / ksplit, p);
        if (t.rows <= 0) continue;
        const int kb0 = (tile % ksplit) * KBS;
        const CUtensorMap* ta = t.shared ? &maps.a_sh : &maps.a;
        const CUtensorMap* tb = t.shared ? maps.b_sh : maps.b;
        const int a_row = (t.shared ? 0 : t.g * p.a_rows_per_group) + t.mb * S::FEATS;
        const uint32_t bytes = S::NUM_A * S::A_BYTES + S::NUM_B * t.n_mma * BLOCK_K * 2;
        for (int kb = kb0; kb < kb0 + KBS; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_u32(smem + stage * S::STAGE_BYTES);
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, bytes);
          if (EPI == EPI_SWIGLU) {
            // gate and up slabs in one 3-D box: (k, row within the gate/up half, 2*expert + half)
            tma_load_3d(sa, ta, fb, kb * BLOCK_K, t.mb * BLOCK_M, t.shared ? 0 : 2 * t.g);
          } else {
            // the MBLK weight slabs are consecutive rows: one box of MBLK * 128 rows
            tma_load_2d(sa, ta, fb, kb * BLOCK_K, a_row);
          }
#pragma unroll
          for (int bp = 0; bp < S::NUM_B; ++bp) {
            const uint32_t sb = sa + S::NUM_A * S::A_BYTES + bp * S::B_BYTES;
            // the (hi, lo) pair: per 64 features, 64 hi columns then 64 lo columns
            const int k0 = kb * BLOCK_K;
            const int kc = HILO ? (k0 >> 6) * 128 + (k0 & 63) + bp * 64 : k0;
            int off = 0;
#pragma unroll
            for (int i = NUM_BOX_H - 1; i >= 0; --i) {
              const int h = B_BOX << i;
              if (h <= TN && (t.n_mma - off) >= h) {
                tma_load_2d(sb + off * S::ROW_BYTES, tb + i, fb, kc, t.b_row + off);
                off += h;
              }
            }
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int buf = 0;
      uint32_t buf_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        const Tile t = decode_tile<TN>(tile / ksplit, p);
        if (t.rows <= 0) continue;
        if (!mbar_wait(acce_bar(buf), buf_phase ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(t.n_mma);
        const uint32_t d0 = tmem_base + buf * S::ACC_COLS;
        for (int kb = 0; kb < KBS; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * S::STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < BLOCK_K / 16; ++kk) {
#pragma unroll
            for (int a = 0; a < S::NUM_A; ++a) {
              const uint64_t da = smem_desc_sw(sa + a * S::A_BYTES, S::ROW_BYTES) + 2 * kk;
#pragma unroll
              for (int bp = 0; bp < S::NUM_B; ++bp) {
                // advance 16 bf16 = 32 bytes along K inside the swizzle row: +2 in the >>4 field
                const uint64_t db = smem_desc_sw(sa + S::NUM_A * S::A_BYTES + bp * S::B_BYTES, S::ROW_BYTES) + 2 * kk;
                const uint32_t accum = (kb | kk | bp) ? 1u : 0u;
                tc_mma(d0 + a * TN, da, db, idesc, accum);
              }
            }
          }
          tc_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(accf_bar(buf));
        if (++buf == S::NUM_BUF) {
          buf = 0;
          buf_phase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int quad = warp & 3;      // TMEM lanes this warp may access: 32*quad .. 32*quad+31
    const int half = ew >> 2;       // which 16-column chunks: half, half+2, half+4, ...
    int buf = 0;
    uint32_t buf_phase = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      const Tile t = decode_tile<TN>(tile / ksplit, p);
      if (t.rows <= 0) continue;
      const long long out_shift = (long long)(tile % ksplit) * p.split_stride;
      if (!mbar_wait(accf_bar(buf), buf_phase, abort_flag, p.err)) break;
      tc_fence_after();
      const uint32_t tq = tmem_base + (uint32_t(quad * 32) << 16) + buf * S::ACC_COLS;
      epilogue_tile<EPI, TN, S::NACC, S::FEATS>(t, p, tq, quad, half, lane, out_shift);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce_bar(buf));
      if (++buf == S::NUM_BUF) {
        buf = 0;
        buf_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, S::TMEM_COLS);
  }
}

// ============================================================================ FP8-weight variant
// The single-CTA kernel on FP8 (E4M3) weight codes with one power-of-two scale per 128 x 128
// tile ("DeepSeek-V4 MoE", section "FP4 QAT 怎么做到反量化无损").  TMA brings each stage's codes
// (64-byte rows, 64-byte swizzle) and token rows into a raw ring in shared memory; four
// converter warps, one per TMEM lane quadrant, each widen whole weight rows to bf16 (q * 2^e,
// exact) and store them into a ring of A tiles in Tensor Memory (lane = weight row, two bf16 per
// column); the MMA reads A from Tensor Memory and B from the raw stage, then releases both.  The
// weight bytes a stage streams are half those of the bf16 kernel, and the widened tiles never
// pass through shared memory.
// Two E4M3 codes -> two bf16 values q * 2^e in one word (low half = the first code), exact,
// through the f16 conversion instruction: the path for zero and subnormal codes and very small
// scales.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2_exact(uint32_t two_codes, float scale) {
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two_codes & 0xFFFFu), __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
  const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// Four normal E4M3 codes (one word) -> four bf16 values q * 2^e (two words, low half first),
// exact.  A normal code (exponent field E in 1..15, mantissa M) is (1 + M/8) 2^(E-7), so its
// bf16 bits are the sign, the exponent field E + 120 + e and M as the top three mantissa bits:
// the bytes are spread into 16-bit lanes, shifted, biased (bias2 = (120 + e) in both lanes'
// exponent fields) and signed with integer operations.
__device__ __forceinline__ uint2 e4m3x4_normal_to_bf16x4(uint32_t w, uint32_t bias2) {
  const uint32_t l0 = __byte_perm(w, 0u, 0x4140);  // codes 0, 1 in 16-bit lanes
  const uint32_t l1 = __byte_perm(w, 0u, 0x4342);  // codes 2, 3
  uint2 r;
  r.x = (((l0 & 0x007F007Fu) << 4) + bias2) | ((l0 & 0x00800080u) << 8);
  r.y = (((l1 & 0x007F007Fu) << 4) + bias2) | ((l1 & 0x00800080u) << 8);
  return r;
}

// True when some code of the word has exponent field 0 (zero or subnormal).
__device__ __forceinline__ bool e4m3x4_has_small(uint32_t w) {
  const uint32_t t = w & 0x78787878u;                  // exponent fields, each byte < 0x80
  return ((t - 0x01010101u) & ~t & 0x80808080u) != 0;  // some byte of t is zero
}

template <int EPI, int TN, int MBLK, bool HILO>
struct Fp8Shape {
  static constexpr int BLOCK_K = 64;
  static constexpr int ROW_BYTES = 128;                  // bf16 rows of B
  static constexpr int NUM_A = (EPI == EPI_SWIGLU) ? 2 : MBLK;
  static constexpr int RAW_SLAB = BLOCK_M * BLOCK_K;     // 128 rows x 64 E4M3 codes
  static constexpr int RAW_A = NUM_A * RAW_SLAB;
  static constexpr int NUM_B = HILO ? 2 : 1;
  static constexpr int B_BYTES = TN * ROW_BYTES;
  static constexpr int RAW_STAGE = RAW_A + NUM_B * B_BYTES;
  static constexpr int A_COLS = BLOCK_K / 2;             // TMEM columns of one widened 128 x 64 slab
  static constexpr int CSTAGES = 4;                      // widened-A stages in Tensor Memory
  static constexpr int CVT_GROUPS = CSTAGES;             // group g widens every CSTAGES-th stage into slot g
  static constexpr int NUM_CVT_WARPS = 4 * CVT_GROUPS;   // one warp per TMEM lane quadrant per group
  static constexpr int THREADS = (2 + NUM_EPI_WARPS + NUM_CVT_WARPS) * 32;
  static constexpr int NACC = NUM_A;
  static constexpr int ACC_COLS = NACC * TN;
  static constexpr int NUM_BUF = (2 * ACC_COLS + CSTAGES * NUM_A * A_COLS <= 512) ? 2 : 1;
  static constexpr int USED_COLS = NUM_BUF * ACC_COLS;
  static constexpr int A_COL0 = USED_COLS;               // first column of the A ring
  static constexpr int TMEM_COLS = 512;
  static constexpr int RSTAGES_FIT = (SMEM_LIMIT - 1024 - 512) / RAW_STAGE;
  static constexpr int RSTAGES = RSTAGES_FIT > 8 ? 8 : RSTAGES_FIT;
  static constexpr int SMEM_BYTES = RSTAGES * RAW_STAGE + 1024 + 512;
  static constexpr int FEATS = (EPI == EPI_SWIGLU) ? BLOCK_M : BLOCK_M * MBLK;
  static_assert(USED_COLS + CSTAGES * NUM_A * A_COLS <= TMEM_COLS, "TMEM: accumulators + A ring");
  static_assert(TN % B_BOX == 0 && TN <= 256, "token tile");
  static_assert(RSTAGES >= 2, "pipeline needs two raw stages");
  static_assert(RAW_A % 1024 == 0 && RAW_STAGE % 1024 == 0, "swizzled tiles start on 1024 bytes");
  static_assert((2 * RSTAGES + 2 * CSTAGES + 4) * 8 + 8 <= 512, "barrier area");
  static_assert(EPI == EPI_F32 || (MBLK == 1 && !HILO), "SwiGLU variant");
};

template <int EPI, int TN, int MBLK, bool HILO>
__global__ void __launch_bounds__(Fp8Shape<EPI, TN, MBLK, HILO>::THREADS, 1)
    fp8w_gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmParams p) {
  using S = Fp8Shape<EPI, TN, MBLK, HILO>;
  constexpr int BLOCK_K = S::BLOCK_K;
  constexpr int RST = S::RSTAGES;
  constexpr int CST = S::CSTAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* raw = smem;                                    // RST raw stages (codes + token rows)
  uint64_t* bars = reinterpret_cast<uint64_t*>(raw + RST * S::RAW_STAGE);
  // bars: full[RST], empty[RST], cfull[CST], cempty[CST], acc_full[2], acc_empty[2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * RST + 2 * CST + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (RST + s); };
  auto cfull_bar = [&](int c) { return bar0 + 8u * (2 * RST + c); };
  auto cempty_bar = [&](int c) { return bar0 + 8u * (2 * RST + CST + c); };
  auto accf_bar = [&](int a) { return bar0 + 8u * (2 * RST + 2 * CST + a); };
  auto acce_bar = [&](int a) { return bar0 + 8u * (2 * RST + 2 * CST + 2 + a); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RST; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int c = 0; c < CST; ++c) {
      mbar_init(cfull_bar(c), 4 * 32);  // the four warps of the slot's converter group
      mbar_init(cempty_bar(c), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf_bar(a), 1);
      mbar_init(acce_bar(a), NUM_EPI_WARPS);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.a);
    tma_prefetch_desc(&maps.a_sh);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), S::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  int total_tiles;
  if (p.grp != nullptr) {
    total_tiles = __ldg(&p.grp[p.n_groups_total].z) * p.num_mblocks * (p.sched_tn / TN);
  } else {
    total_tiles = ((p.dense_rows + p.sched_tn - 1) / p.sched_tn) * p.num_mblocks * (p.sched_tn / TN);
  }
  const int KB = p.K / BLOCK_K;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        const Tile t = decode_tile<TN>(tile, p);
        if (t.rows <= 0) continue;
        const CUtensorMap* ta = t.shared ? &maps.a_sh : &maps.a;
        const CUtensorMap* tb = t.shared ? maps.b_sh : maps.b;
        const int a_row = (t.shared ? 0 : t.g * p.a_rows_per_group) + t.mb * S::FEATS;
        const uint32_t bytes = S::RAW_A + S::NUM_B * t.n_mma * S::ROW_BYTES;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t sr = smem_u32(raw + stage * S::RAW_STAGE);
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, bytes);
          if (EPI == EPI_SWIGLU) {
            tma_load_3d(sr, ta, fb, kb * BLOCK_K, t.mb * BLOCK_M, t.shared ? 0 : 2 * t.g);  // gate, up codes
          } else {
            tma_load_2d(sr, ta, fb, kb * BLOCK_K, a_row);                                   // MBLK slabs
          }
#pragma unroll
          for (int bp = 0; bp < S::NUM_B; ++bp) {
            const uint32_t sb = sr + S::RAW_A + bp * S::B_BYTES;
            const int k0 = kb * BLOCK_K;
            const int kc = HILO ? (k0 >> 6) * 128 + (k0 & 63) + bp * 64 : k0;
            int off = 0;
#pragma unroll
            for (int i = NUM_BOX_H - 1; i >= 0; --i) {
              const int h = B_BOX << i;
              if (h <= TN && (t.n_mma - off) >= h) {
                tma_load_2d(sb + off * S::ROW_BYTES, tb + i, fb, kc, t.b_row + off);
                off += h;
              }
            }
          }
          if (++stage == RST) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, cs = 0;
      uint32_t phase = 0, cphase = 0;
      int buf = 0;
      uint32_t buf_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        const Tile t = decode_tile<TN>(tile, p);
        if (t.rows <= 0) continue;
        if (!mbar_wait(acce_bar(buf), buf_phase ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(t.n_mma);
        const uint32_t d0 = tmem_base + buf * S::ACC_COLS;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag, p.err) ||
              !mbar_wait(cfull_bar(cs), cphase, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sr = smem_u32(raw + stage * S::RAW_STAGE);
          const uint32_t ta = tmem_base + S::A_COL0 + cs * (S::NUM_A * S::A_COLS);
#pragma unroll
          for (int kk = 0; kk < BLOCK_K / 16; ++kk) {
#pragma unroll
            for (int a = 0; a < S::NUM_A; ++a) {
#pragma unroll
              for (int bp = 0; bp < S::NUM_B; ++bp) {
                const uint64_t db = smem_desc_sw(sr + S::RAW_A + bp * S::B_BYTES, S::ROW_BYTES) + 2 * kk;
                tc_mma_ta(d0 + a * TN, ta + a * S::A_COLS + kk * 8, db, idesc, (kb | kk | bp) ? 1u : 0u);
              }
            }
          }
          tc_commit(empty_bar(stage));
          tc_commit(cempty_bar(cs));
          if (++stage == RST) {
            stage = 0;
            phase ^= 1u;
          }
          if (++cs == CST) {
            cs = 0;
            cphase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(accf_bar(buf));
        if (++buf == S::NUM_BUF) {
          buf = 0;
          buf_phase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp < 2 + NUM_EPI_WARPS) {
    // ------------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int quad = warp & 3;
    const int half = ew >> 2;
    int buf = 0;
    uint32_t buf_phase = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      const Tile t = decode_tile<TN>(tile, p);
      if (t.rows <= 0) continue;
      if (!mbar_wait(accf_bar(buf), buf_phase, abort_flag, p.err)) break;
      tc_fence_after();
      const uint32_t tq = tmem_base + (uint32_t(quad * 32) << 16) + buf * S::ACC_COLS;
      epilogue_tile<EPI, TN, S::NACC, S::FEATS>(t, p, tq, quad, half, lane, 0);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce_bar(buf));
      if (++buf == S::NUM_BUF) {
        buf = 0;
        buf_phase ^= 1u;
      }
    }
  } else {
    // ------------------------------------------------------------------ code -> bf16 converters
    // CVT_GROUPS groups of four warps; group g widens the stages n with n % CVT_GROUPS == g into
    // A slot g, so that several stages are widened at once (each warp must wait for its Tensor
    // Memory stores before reporting a stage).  Within a group, warp w owns TMEM lane quadrant
    // w % 4, i.e. weight rows r = 32 (w % 4) + lane of every slab: the thread reads that row's 64
    // codes (four 16-byte chunks; chunk c of row r at c ^ ((r >> 1) & 3), the 64-byte swizzle
    // TMA wrote), widens them with the row's scale 2^e and stores the 32 columns of bf16 pairs
    // into the slot's A tile.  A slab spans at most two 128-row tiles: the thread keeps the two
    // exponents of the current 128-wide K tile and loads those of the next one ahead, so no
    // global load sits in a stage's critical path and no converter waits on another.
    const int quad = warp & 3;
    const int group = (warp - 2 - NUM_EPI_WARPS) >> 2;
    const int r = quad * 32 + lane;
    const uint32_t ta = tmem_base + (uint32_t(quad * 32) << 16) + S::A_COL0 + group * (S::NUM_A * S::A_COLS);
    const int nk = p.exp_nk;
    uint32_t n = 0;   // stage counter over all tiles of this CTA
    uint32_t mine = 0; // stages this group has widened
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
      const Tile t = decode_tile<TN>(tile, p);
      if (t.rows <= 0) continue;
      const int8_t* ex = t.shared ? p.a_sh_exp : p.a_exp + (size_t)t.g * p.exp_nr * p.exp_nk;
      int trow[S::NUM_A];  // this row's tile row in each slab (clamped to the matrix)
#pragma unroll
      for (int a = 0; a < S::NUM_A; ++a) {
        const int base = (EPI == EPI_SWIGLU) ? a * p.a_up_offset + t.mb * BLOCK_M : t.mb * S::FEATS + a * BLOCK_M;
        trow[a] = min((base + r) >> 7, p.exp_nr - 1);
      }
      int e_cur[S::NUM_A], e_nxt[S::NUM_A];
#pragma unroll
      for (int a = 0; a < S::NUM_A; ++a) {
        e_cur[a] = __ldg(ex + trow[a] * nk);
        e_nxt[a] = nk > 1 ? __ldg(ex + trow[a] * nk + 1) : 0;
      }
      for (int kb = 0; kb < KB; ++kb, ++n) {
        if (kb > 0 && ((kb * BLOCK_K) & 127) == 0) {  // a new 128-wide K tile: rotate, fetch the next
          const int kn = ((kb * BLOCK_K) >> 7) + 1;
#pragma unroll
          for (int a = 0; a < S::NUM_A; ++a) {
            e_cur[a] = e_nxt[a];
            e_nxt[a] = kn < nk ? __ldg(ex + trow[a] * nk + kn) : 0;
          }
        }
        if ((int)(n % S::CVT_GROUPS) != group) continue;
        const int stage = (int)(n % RST);
        const uint32_t phase = (n / RST) & 1u;
        if (!mbar_wait(full_bar(stage), phase, abort_flag, p.err) ||
            !mbar_wait(cempty_bar(group), (mine & 1u) ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        ++mine;
        tc_fence_after();
        const uint8_t* src = raw + stage * S::RAW_STAGE;
#pragma unroll
        for (int a = 0; a < S::NUM_A; ++a) {
          const int e = e_cur[a];
          const uint32_t bias2 = (uint32_t)(120 + e) * 0x00800080u;
          const float scale = __int_as_float((e + 127) << 23);
          const bool tiny = e < -120;
          const uint8_t* row = src + a * S::RAW_SLAB + r * 64;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t o[16];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              const int c = 2 * h + cc;  // K codes [16 c, 16 c + 16)
              const uint4 q = *reinterpret_cast<const uint4*>(row + ((c ^ ((r >> 1) & 3)) << 4));
              uint2 v0, v1, v2, v3;
              // normal codes and an ordinary scale (the common case): integer path; otherwise (a
              // zero or subnormal code, or a scale below 2^-120, where E + 120 + e could leave the
              // normal bf16 range) the chunk goes through the conversion instruction
              if (!tiny && !(e4m3x4_has_small(q.x) | e4m3x4_has_small(q.y) | e4m3x4_has_small(q.z) |
                             e4m3x4_has_small(q.w))) {
                v0 = e4m3x4_normal_to_bf16x4(q.x, bias2);
                v1 = e4m3x4_normal_to_bf16x4(q.y, bias2);
                v2 = e4m3x4_normal_to_bf16x4(q.z, bias2);
                v3 = e4m3x4_normal_to_bf16x4(q.w, bias2);
              } else {
                v0 = make_uint2(e4m3x2_to_bf16x2_exact(q.x, scale), e4m3x2_to_bf16x2_exact(q.x >> 16, scale));
                v1 = make_uint2(e4m3x2_to_bf16x2_exact(q.y, scale), e4m3x2_to_bf16x2_exact(q.y >> 16, scale));
                v2 = make_uint2(e4m3x2_to_bf16x2_exact(q.z, scale), e4m3x2_to_bf16x2_exact(q.z >> 16, scale));
                v3 = make_uint2(e4m3x2_to_bf16x2_exact(q.w, scale), e4m3x2_to_bf16x2_exact(q.w >> 16, scale));
              }
              o[8 * cc + 0] = v0.x;
              o[8 * cc + 1] = v0.y;
              o[8 * cc + 2] = v1.x;
              o[8 * cc + 3] = v1.y;
              o[8 * cc + 4] = v2.x;
              o[8 * cc + 5] = v2.y;
              o[8 * cc + 6] = v3.x;
              o[8 * cc + 7] = v3.y;
            }
            tmem_st16(ta + a * S::A_COLS + h * 16, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(cfull_bar(group));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, S::TMEM_COLS);
  }
}

// ============================================================================ FP8 MMA variant
// The single-CTA kernel with the E4M3 weight codes as the MMA's A operand as they are (tcgen05
// kind::f8f6f4, twice the bf16 rate), one power-of-two scale per 128 x 128 code tile ("DeepSeek-V4
// MoE", section "FP4 QAT 怎么做到反量化无损").  B holds the token rows as E4M3 pieces with one
// power-of-two scale per row (x: 2 pieces, h: 4; see the split kernel).  The pieces of a tile's
// token rows sit one after another in the stage (piece p at rows p * n .. p * n + n - 1), so one
// MMA per slab and K step multiplies all of them (N = pieces * n) and reads the A tile from
// shared memory once.  A stage is one 128-wide K tile, so a single weight scale 2^e covers each
// slab of it: the MMAs of K tile kt write their own slot of a ring in Tensor Memory, and the
// epilogue warps add (sum of the piece columns) * 2^e(kt) into fp32 registers and release the
// slot; after the last K tile they apply the row scales and write the tile (SwiGLU: fp32 h;
// fp32: O rows x gate weight).  The slabs must start on a scale tile (gate/up: d_ff a multiple
// of 128).
template <int EPI, int MBLK, int TN_>
struct F8Shape {
  static constexpr int TN = TN_;                        // token rows per tile (16, 32 or 64)
  static constexpr int BLOCK_K = 128;                   // codes per stage = one scale tile of K
  static constexpr int NUM_A = (EPI == EPI_SWIGLU) ? 2 : MBLK;
  static constexpr int A_SLAB = BLOCK_M * BLOCK_K;      // 128 weight rows x 128 codes
  static constexpr int PIECES = (EPI == EPI_SWIGLU) ? 2 : 4;
  static constexpr int B_PIECE = TN * BLOCK_K;          // TN token rows x 128 codes
  static constexpr int STAGE_BYTES = NUM_A * A_SLAB + PIECES * B_PIECE;
  static constexpr int SLOT_COLS = NUM_A * PIECES * TN; // partial products of one K tile
  static constexpr int SLOTS = (512 / SLOT_COLS) > 8 ? 8 : (512 / SLOT_COLS);
  static constexpr int STAGES_FIT = (SMEM_LIMIT - 1024 - 512) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 512;
  static constexpr int FEATS = (EPI == EPI_SWIGLU) ? BLOCK_M : BLOCK_M * MBLK;
  static_assert(SLOTS * SLOT_COLS <= 512, "TMEM holds 512 columns");
  static_assert(STAGES >= 2, "pipeline needs two stages");
  static_assert(A_SLAB % 1024 == 0 && B_PIECE % 1024 == 0 && STAGE_BYTES % 1024 == 0, "swizzled tiles on 1024 B");
  static_assert((2 * STAGES + 2 * SLOTS) * 8 + 8 <= 512, "barrier area");
  static_assert(EPI == EPI_F32 || MBLK == 1, "SwiGLU variant");
  static_assert(TN == 16 || TN == 32 || TN == 64, "token tile");
  static_assert(PIECES * TN <= 256, "MMA N");
};

template <int EPI, int MBLK, int TN_>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fp8mma_gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmParams p) {
  using S = F8Shape<EPI, MBLK, TN_>;
  constexpr int TN = S::TN;
  constexpr int ST = S::STAGES;
  constexpr int SL = S::SLOTS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ST * S::STAGE_BYTES);
  // bars: full[ST], empty[ST], slot_full[SL], slot_empty[SL]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * ST + 2 * SL);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (ST + s); };
  auto sfull_bar = [&](int c) { return bar0 + 8u * (2 * ST + c); };
  auto sempty_bar = [&](int c) { return bar0 + 8u * (2 * ST + SL + c); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int c = 0; c < SL; ++c) {
      mbar_init(sfull_bar(c), 1);
      mbar_init(sempty_bar(c), NUM_EPI_WARPS);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.a);
    tma_prefetch_desc(&maps.a_sh);
    for (int i = 0; (B_BOX << i) <= TN; ++i) tma_prefetch_desc(&maps.b[i]);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int row_tiles = p.grp != nullptr ? __ldg(&p.grp[p.n_groups_total].z)
                                         : (p.dense_rows + p.sched_tn - 1) / p.sched_tn;
  const int total_tiles = row_tiles * p.num_mblocks * (p.sched_tn / TN);
  const int KB = p.K / S::BLOCK_K;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        const Tile t = decode_tile<TN>(tile, p);
        if (t.rows <= 0) continue;
        const CUtensorMap* ta = t.shared ? &maps.a_sh : &maps.a;
        const int a_row = (t.shared ? 0 : t.g * p.a_rows_per_group) + t.mb * S::FEATS;
        const uint32_t bytes = S::NUM_A * S::A_SLAB + S::PIECES * t.n_mma * S::BLOCK_K;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_u32(smem + stage * S::STAGE_BYTES);
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, bytes);
          if (EPI == EPI_SWIGLU) {
            tma_load_3d(sa, ta, fb, kb * S::BLOCK_K, t.mb * BLOCK_M, t.shared ? 0 : 2 * t.g);  // gate, up codes
          } else {
            tma_load_2d(sa, ta, fb, kb * S::BLOCK_K, a_row);                                   // MBLK slabs
          }
#pragma unroll
          for (int pc = 0; pc < S::PIECES; ++pc) {
            const uint32_t sb = sa + S::NUM_A * S::A_SLAB + pc * t.n_mma * S::BLOCK_K;
            int off = 0;
#pragma unroll
            for (int i = 2; i >= 0; --i) {  // boxes of 64, 32, 16 rows
              const int h = B_BOX << i;
              if (h <= TN && (t.n_mma - off) >= h) {
                tma_load_3d(sb + off * S::BLOCK_K, &maps.b[i], fb, kb * S::BLOCK_K, pc, t.b_row + off);
                off += h;
              }
            }
          }
          if (++stage == ST) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, slot = 0;
      uint32_t phase = 0, sphase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        const Tile t = decode_tile<TN>(tile, p);
        if (t.rows <= 0) continue;
        const uint32_t idesc = idesc_e4m3_f32(S::PIECES * t.n_mma);  // all pieces in one N
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag, p.err) ||
              !mbar_wait(sempty_bar(slot), sphase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * S::STAGE_BYTES);
          const uint32_t d0 = tmem_base + slot * S::SLOT_COLS;
#pragma unroll
          for (int kk = 0; kk < S::BLOCK_K / 32; ++kk) {
            // advance 32 codes = 32 bytes along K inside the swizzle row: +2 in the >>4 field
            const uint64_t db = smem_desc_sw(sa + S::NUM_A * S::A_SLAB, 128) + 2 * kk;
#pragma unroll
            for (int a = 0; a < S::NUM_A; ++a) {
              const uint64_t da = smem_desc_sw(sa + a * S::A_SLAB, 128) + 2 * kk;
              tc_mma_f8(d0 + a * S::PIECES * TN, da, db, idesc, kk ? 1u : 0u);
            }
          }
          tc_commit(empty_bar(stage));
          tc_commit(sfull_bar(slot));
          if (++stage == ST) {
            stage = 0;
            phase ^= 1u;
          }
          if (++slot == SL) {
            slot = 0;
            sphase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue
    // Warp (quad, half): TMEM lanes 32 quad .. 32 quad + 31 (weight rows), token columns
    // 32 half .. 32 half + 31 of every slab's partial products.
    const int ew = warp - 2;
    const int quad = warp & 3;
    const int half = ew >> 2;
    int slot = 0;
    uint32_t sphase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
      const Tile t = decode_tile<TN>(tile, p);
      if (t.rows <= 0) continue;
      const int cols = min(32, t.rows - half * 32);  // valid token columns of this warp (may be <= 0)
      const int8_t* ex = t.shared ? p.a_sh_exp : p.a_exp + (size_t)t.g * p.exp_nr * p.exp_nk;
      int erow[S::NUM_A];  // each slab's row of scale tiles (clamped to the matrix)
#pragma unroll
      for (int a = 0; a < S::NUM_A; ++a) {
        const int base = (EPI == EPI_SWIGLU) ? a * p.a_up_offset + t.mb * BLOCK_M : t.mb * S::FEATS + a * BLOCK_M;
        erow[a] = min(base >> 7, p.exp_nr - 1) * p.exp_nk;
      }
      float acc[S::NUM_A][32];
#pragma unroll
      for (int a = 0; a < S::NUM_A; ++a)
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[a][j] = 0.0f;
      int e_cur[S::NUM_A];
#pragma unroll
      for (int a = 0; a < S::NUM_A; ++a) e_cur[a] = __ldg(ex + erow[a]);
      const uint32_t tq = tmem_base + (uint32_t(quad * 32) << 16) + half * 32;
      for (int kb = 0; kb < KB; ++kb) {
        int e_nxt[S::NUM_A];  // the next K tile's scales, loaded ahead of the wait
#pragma unroll
        for (int a = 0; a < S::NUM_A; ++a) e_nxt[a] = (kb + 1 < KB) ? __ldg(ex + erow[a] + kb + 1) : 0;
        if (!mbar_wait(sfull_bar(slot), sphase, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (cols > 0) {
          const uint32_t ts = tq + slot * S::SLOT_COLS;
#pragma unroll
          for (int a = 0; a < S::NUM_A; ++a) {
            const float sc = __int_as_float((e_cur[a] + 127) << 23);  // 2^e, e in [-126, 120]
#pragma unroll
            for (int pp = 0; pp < S::PIECES; pp += 2) {  // two pieces' columns per wait
              uint32_t r0[2][16], r1[2][16];
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                const uint32_t c = ts + a * S::PIECES * TN + (pp + q) * t.n_mma;
                tmem_ld16(c, r0[q]);
                if (cols > 16) tmem_ld16(c + 16, r1[q]);
              }
              tmem_ld_wait();
              reg_fence16(r0[0]);
              reg_fence16(r0[1]);
#pragma unroll
              for (int j = 0; j < 16; ++j)
                acc[a][j] = fmaf(__uint_as_float(r0[0][j]) + __uint_as_float(r0[1][j]), sc, acc[a][j]);
              if (cols > 16) {
                reg_fence16(r1[0]);
                reg_fence16(r1[1]);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                  acc[a][16 + j] = fmaf(__uint_as_float(r1[0][j]) + __uint_as_float(r1[1][j]), sc, acc[a][16 + j]);
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sempty_bar(slot));
#pragma unroll
        for (int a = 0; a < S::NUM_A; ++a) e_cur[a] = e_nxt[a];
        if (++slot == SL) {
          slot = 0;
          sphase ^= 1u;
        }
      }
      if (!ok || cols <= 0) continue;
      // row scales 2^e_r (the pieces hold row r times 2^-e_r) and the gate weight: lane l holds
      // those of token column 32 half + l
      const int rl = half * 32 + lane;
      const bool rvalid = rl < t.rows;
      const int er = rvalid ? __ldg(p.b_exp + t.b_row + rl) : 0;
      float cs_l = __int_as_float((127 + er) << 23);  // e_r in [-126, 120]
      if (EPI == EPI_F32 && p.row_scale != nullptr && !t.shared && rvalid) cs_l *= __ldg(p.row_scale + t.out_row + rl);
      float* out = static_cast<float*>(p.out) + (size_t)(t.out_row + half * 32) * p.out_ld;
      if (EPI == EPI_SWIGLU) {
        const int feat = t.mb * BLOCK_M + quad * 32 + lane;
        const bool fvalid = feat < p.out_features;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float cs = __shfl_sync(0xffffffffu, cs_l, j);
          if (j < cols && fvalid) {
            const float g = acc[0][j] * cs, u = acc[1][j] * cs;
            out[(size_t)j * p.out_ld + feat] = __fdividef(g, 1.0f + __expf(-g)) * u;
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float cs = __shfl_sync(0xffffffffu, cs_l, j);
#pragma unroll
          for (int a = 0; a < S::NUM_A; ++a) {
            const int feat = t.mb * S::FEATS + a * BLOCK_M + quad * 32 + lane;
            if (j < cols && feat < p.out_features) out[(size_t)j * p.out_ld + feat] = acc[a][j] * cs;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// ============================================================================ CTA-pair variant
// The same contractions on the 2-SM MMA (tcgen05 .cta_group::2).  A cluster of two CTAs computes
// one tile of 256 weight rows x N token rows: CTA r holds weight rows [128 r, 128 r + 128) of the
// tile and token rows [r N/2, r N/2 + N/2) of B, the even CTA issues the MMAs, and each CTA's
// TMEM receives its 128 accumulator rows for all N columns.  Each SM therefore stores and reads
// only half of B, which keeps its shared-memory bandwidth below what the tensor pipe consumes.
//   SwiGLU: the pair covers 128 features; CTA r's weight rows are the gate rows of features
//           [64 r, 64 r + 64) followed by the up rows of the same features, so gate and up of
//           one feature sit in TMEM lanes i and i + 64 of one CTA (exchanged through smem).
//   fp32:   the pair covers 256 output features, CTA r the features [128 r, 128 r + 128).
// MB = 2 gives each CTA two 128-row weight slabs against the same token rows (twice the MMA work
// per byte of B landed; both accumulators fill the 512 TMEM columns, one buffer):
//   SwiGLU: slab 0 = the gate rows, slab 1 = the up rows of the CTA's 128 features (the pair
//           covers 256), so gate and up of a feature sit in the same TMEM lane of accumulators
//           0 and 1 and the epilogue needs no exchange;
//   fp32:   two adjacent 128-feature blocks (the pair covers 512 output features).
template <int EPI, int TN, bool HILO, int BK, int TMEM_ALLOC, int MB, bool BG>
struct PairShape {
  static constexpr int BLOCK_K = BK;
  static constexpr int ROW_BYTES = BK * 2;
  static constexpr int HALF = TN / 2;
  static constexpr int A_BYTES = BLOCK_M * BK * 2;                  // one 128-row weight slab
  static constexpr int NUM_B = HILO ? 2 : 1;
  static constexpr int B_BYTES = HALF * BK * 2;
  static constexpr int STAGE_BYTES = MB * A_BYTES + NUM_B * B_BYTES;
  static constexpr bool GU = (EPI == EPI_SWIGLU) && MB == 2;       // gate slab + up slab
  static constexpr int XCH = (EPI == EPI_SWIGLU && !GU) ? 4 : 0;    // gate/up warp pairs
  static constexpr int XBUF_BYTES = XCH * 2 * 16 * 32 * 4;          // 2 slots of 16 x 32 fp32
  static constexpr int ACC_COLS = MB * TN;                          // MB accumulators of TN columns
  static constexpr int NUM_BUF = (TMEM_ALLOC / ACC_COLS) >= 2 ? 2 : 1;
  static constexpr int STAGES_FIT = (SMEM_LIMIT - 1024 - 512 - XBUF_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 16 ? 16 : STAGES_FIT;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + XBUF_BYTES + 1024 + 512;
  static constexpr int FEATS = (EPI == EPI_SWIGLU) ? (GU ? 2 * BLOCK_M : BLOCK_M) : 2 * BLOCK_M * MB;
  static constexpr int A_BOX = (EPI == EPI_SWIGLU) ? (GU ? BLOCK_M : BLOCK_M / 2) : BLOCK_M;
  // BG: the token rows are gathered by NBW loader warps with 16-byte cp.async copies, and one
  // relay warp reports their completed stages to the pair's even CTA
  static constexpr int NBW = BG ? 4 : 0;
  static constexpr int THREADS = (2 + NUM_EPI_WARPS + NBW + (BG ? 1 : 0)) * 32;
  static constexpr int CHUNKS = ROW_BYTES / 16;                     // 16-byte chunks per token row
  static constexpr int ROWS_PER_PASS = BG ? NBW * 32 / CHUNKS : 1;
  static constexpr int ROWS_PER_THREAD = BG ? HALF / ROWS_PER_PASS : 0;
  static_assert(!BG || (EPI == EPI_SWIGLU && !HILO && BK == 64 && HALF % ROWS_PER_PASS == 0),
                "gathered token rows: gate/up, 128-byte rows");
  // barriers (full, empty per stage; acc full/empty x2; exchange full/empty x2 per channel;
  // BG: gathered-rows landed per stage), then the TMEM address slot and the abort flag, in the
  // last 512 bytes
  static constexpr int NUM_LBAR = BG ? STAGES : 0;
  static_assert((2 * STAGES + 4 + 4 * XCH + NUM_LBAR) * 8 + 8 <= 512, "barrier area");
  static_assert(TN % 32 == 0 && TN <= 256, "pair token tile");
  static_assert(TMEM_ALLOC >= ACC_COLS && TMEM_ALLOC <= 512, "TMEM allocation");
  static_assert(STAGES >= 2, "pipeline needs two stages");
  static_assert(BK == 64 || BK == 32, "stage K");
  static_assert(MB == 1 || MB == 2, "weight slabs per CTA");
};

// NP = CTA pairs per cluster.  With NP = 2 the two pairs of a cluster work on the same token
// rows and on adjacent feature blocks; each CTA TMA-loads a quarter of the token rows and
// multicasts it to the CTA holding the same half in the other pair, so each SM requests only
// half of its B half.  The multicast's bytes are counted on each destination pair's even-CTA
// barrier, and a stage is refilled only after both pairs' MMAs released it.
template <int EPI, int TN, bool HILO, int BK, int TMEM_ALLOC, int NP, int MB, bool BG>
__global__ void __launch_bounds__(PairShape<EPI, TN, HILO, BK, TMEM_ALLOC, MB, BG>::THREADS, 1)
    pair_gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmParams p) {
  using S = PairShape<EPI, TN, HILO, BK, TMEM_ALLOC, MB, BG>;
  static_assert(!BG || NP == 1, "gathered token rows with one pair per cluster");
  constexpr int STAGES = S::STAGES;
  constexpr int BLOCK_K = S::BLOCK_K;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* xbuf = reinterpret_cast<float*>(smem + STAGES * S::STAGE_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * S::STAGE_BYTES + S::XBUF_BYTES);
  // bars: full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], xfull[XCH][2], xempty[XCH][2],
  // landed[NUM_LBAR]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 4 + 4 * S::XCH + S::NUM_LBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto accf_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto acce_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  auto xfull_bar = [&](int x, int sl) { return bar0 + 8u * (2 * STAGES + 4 + 2 * x + sl); };
  auto xempty_bar = [&](int x, int sl) { return bar0 + 8u * (2 * STAGES + 4 + 2 * S::XCH + 2 * x + sl); };
  auto landed_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + 4 + 4 * S::XCH + s); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const uint32_t rank = crank & 1u;    // position in the CTA pair
  const uint32_t pp = crank >> 1;      // which pair of the cluster
  const uint32_t lrank = crank & ~1u;  // cluster rank of this pair's even CTA
  const bool leader = (rank == 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), BG ? 3 : 1);  // the even CTA's expect-tx arrival (+ both relays)
      mbar_init(empty_bar(s), NP);  // one commit per pair of the cluster
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf_bar(a), 1);
      mbar_init(acce_bar(a), 2 * NUM_EPI_WARPS);
    }
    for (int x = 0; x < S::XCH; ++x)
      for (int sl = 0; sl < 2; ++sl) {
        mbar_init(xfull_bar(x, sl), 32);
        mbar_init(xempty_bar(x, sl), 32);
      }
    for (int s = 0; s < S::NUM_LBAR; ++s) mbar_init(landed_bar(s), S::NBW * 32);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.a);
    tma_prefetch_desc(&maps.a_sh);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), TMEM_ALLOC);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int pair = blockIdx.x / (2 * NP);   // cluster index
  const int npairs = gridDim.x / (2 * NP);  // clusters
  int total_tiles;
  if (p.grp != nullptr) {
    total_tiles = __ldg(&p.grp[p.n_groups_total].z) * p.num_mblocks * (p.sched_tn / TN);
  } else {
    total_tiles = ((p.dense_rows + p.sched_tn - 1) / p.sched_tn) * p.num_mblocks * (p.sched_tn / TN);
  }
  const int KB = p.K / BLOCK_K;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < total_tiles; tile += npairs) {
        const Tile t = decode_tile<TN>(tile, p);
        if (t.rows <= 0) continue;
        const int mb = t.mb * NP + (int)pp;  // this pair's feature block
        const int unit = 32 * NP;
        const int n_mma = max(unit, (t.rows + unit - 1) / unit * unit);
        const int half = n_mma >> 1;         // token rows per CTA
        const int qh = half / NP;            // token rows this CTA loads (NP = 2: multicast)
        const CUtensorMap* ta = t.shared ? &maps.a_sh : &maps.a;
        const CUtensorMap* tb = t.shared ? maps.b_sh : maps.b;
        const int base = t.shared ? 0 : t.g * p.a_rows_per_group;
        const int b_off = (NP == 2) ? (int)pp * qh : 0;  // rows into this CTA's half
        const int b_row = t.b_row + (int)rank * half + b_off;
        const uint32_t b_land = BG ? 0u : S::NUM_B * half * BLOCK_K * 2;  // TMA B bytes landing in one CTA
        const uint32_t expect = 2u * (MB * S::A_BYTES + b_land);  // both CTAs' A and B, on the even CTA
        const uint16_t mc_mask = (uint16_t)((1u << rank) | (1u << (2 + rank)));
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_u32(smem + stage * S::STAGE_BYTES);
          const uint32_t fbc = mapa_shared(full_bar(stage), lrank);  // the pair's even CTA's full barrier
          if (leader) mbar_arrive_expect_tx(full_bar(stage), expect);
          const int k0 = kb * BLOCK_K;
          if (S::GU) {
            // gate rows, then up rows, of this CTA's 128 features: one 3-D box, two slabs
            tma_load_3d_pair(sa, ta, fbc, k0, mb * 2 * BLOCK_M + (int)rank * BLOCK_M, t.shared ? 0 : 2 * t.g);
          } else {
#pragma unroll
            for (int ms = 0; ms < MB; ++ms) {
              const int fb = mb * MB + ms;  // 128-row weight slab of the pair
              if (EPI == EPI_SWIGLU) {
                // this CTA's gate and up slabs (64 features each) in one 3-D box
                tma_load_3d_pair(sa + ms * S::A_BYTES, ta, fbc, k0, fb * BLOCK_M + (int)rank * (BLOCK_M / 2),
                                 t.shared ? 0 : 2 * t.g);
              } else {
                tma_load_2d_pair(sa + ms * S::A_BYTES, ta, fbc, k0,
                                 base + fb * 2 * BLOCK_M + (int)rank * BLOCK_M);
              }
            }
          }
#pragma unroll
          for (int bp = 0; bp < (BG ? 0 : S::NUM_B); ++bp) {
            const uint32_t sb = sa + MB * S::A_BYTES + bp * S::B_BYTES + b_off * S::ROW_BYTES;
            const int kc = HILO ? (k0 >> 6) * 128 + (k0 & 63) + bp * 64 : k0;
            int off = 0;
#pragma unroll
            for (int i = NUM_BOX_H - 1; i >= 0; --i) {
              const int h = B_BOX << i;
              if (h <= S::HALF && (qh - off) >= h) {
                if (NP == 2)
                  tma_load_2d_pair_mc(sb + off * S::ROW_BYTES, tb + i, fbc, kc, b_row + off, mc_mask);
                else
                  tma_load_2d_pair(sb + off * S::ROW_BYTES, tb + i, fbc, kc, b_row + off);
                off += h;
              }
            }
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (even CTA)
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int buf = 0;
      uint32_t buf_phase = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < total_tiles; tile += npairs) {
        const Tile t = decode_tile<TN>(tile, p);
        if (t.rows <= 0) continue;
        const int unit = 32 * NP;
        const int n_mma = max(unit, (t.rows + unit - 1) / unit * unit);
        if (!mbar_wait_cluster(acce_bar(buf), buf_phase ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32_m256(n_mma);
        const uint32_t d = tmem_base + buf * S::ACC_COLS;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_cluster(full_bar(stage), phase, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * S::STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < BLOCK_K / 16; ++kk) {
#pragma unroll
            for (int ms = 0; ms < MB; ++ms) {
              const uint64_t da = smem_desc_sw(sa + ms * S::A_BYTES, S::ROW_BYTES) + 2 * kk;
#pragma unroll
              for (int bp = 0; bp < S::NUM_B; ++bp) {
                const uint64_t db = smem_desc_sw(sa + MB * S::A_BYTES + bp * S::B_BYTES, S::ROW_BYTES) + 2 * kk;
                tc_mma_pair(d + ms * TN, da, db, idesc, (kb | kk | bp) ? 1u : 0u);
              }
            }
          }
          tc_commit_pair_mc(empty_bar(stage), (uint16_t)((1u << (2 * NP)) - 1u));  // every CTA
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(accf_bar(buf), (uint16_t)(0x3u << lrank));
        if (++buf == S::NUM_BUF) {
          buf = 0;
          buf_phase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp < 2 + NUM_EPI_WARPS) {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    const int ew = warp - 2;
    const int quad = warp & 3;
    const int half = ew >> 2;
    const int xch = half * 2 + (quad & 1);  // SwiGLU: exchange channel of this gate/up warp pair
    int buf = 0;
    uint32_t buf_phase = 0;
    uint32_t xiter = 0;                      // SwiGLU: chunks exchanged so far on this channel
    bool ok = true;
    const uint32_t acce_leader0 = mapa_shared(acce_bar(0), lrank);
    const uint32_t acce_leader1 = mapa_shared(acce_bar(1), lrank);
    for (int tile = pair; ok && tile < total_tiles; tile += npairs) {
      const Tile t = decode_tile<TN>(tile, p);
      if (t.rows <= 0) continue;
      if (!mbar_wait_cluster(accf_bar(buf), buf_phase, abort_flag, p.err)) break;
      tc_fence_after();
      const int nchunk = (t.rows + 15) >> 4;
      for (int ms = 0; ok && ms < (S::GU ? 1 : MB); ++ms) {
        const uint32_t tq = tmem_base + (uint32_t(quad * 32) << 16) + buf * S::ACC_COLS + ms * TN;
        const int fb = (t.mb * NP + (int)pp) * MB + ms;  // 128-row weight slab of this accumulator
        if (S::GU) {
          // lane = feature; gate in accumulator 0, up in accumulator 1 of the same lane
          const int feat = (t.mb * NP + (int)pp) * 2 * BLOCK_M + (int)rank * BLOCK_M + quad * 32 + lane;
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
            if (fvalid) {
              __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + (size_t)(t.out_row + c0) * p.out_ld + col;
              const int nr = min(16, t.rows - c0);
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                if (j < nr) {
                  const float g = __uint_as_float(rg[j]);
                  const float h = __fdividef(g, 1.0f + __expf(-g)) * __uint_as_float(ru[j]);
                  const __nv_bfloat16 hi = __float2bfloat16_rn(h);
                  const __nv_bfloat16 lo = __float2bfloat16_rn(h - __bfloat162float(hi));
                  out[(size_t)j * p.out_ld] = hi;
                  out[(size_t)j * p.out_ld + 64] = lo;
                }
              }
            }
          }
        } else if (EPI == EPI_SWIGLU) {
          float* xb = xbuf + xch * (2 * 16 * 32);
          for (int ci = half; ci < nchunk; ci += 2, ++xiter) {
            const int sl = xiter & 1;
            const uint32_t par = (xiter >> 1) & 1u;
            const int c0 = ci * 16;
            if (quad >= 2) {
              // up lanes: hand the 16 up values of this chunk to the gate warp of the channel
              uint32_t ru[16];
              tmem_ld16(tq + c0, ru);
              tmem_ld_wait();
              reg_fence16(ru);
              if (!mbar_wait(xempty_bar(xch, sl), par ^ 1u, abort_flag, p.err)) {
                ok = false;
                break;
              }
#pragma unroll
              for (int j = 0; j < 16; ++j) xb[(sl * 16 + j) * 32 + lane] = __uint_as_float(ru[j]);
              mbar_arrive(xfull_bar(xch, sl));
            } else {
              uint32_t rg[16];
              tmem_ld16(tq + c0, rg);
              tmem_ld_wait();
              reg_fence16(rg);
              if (!mbar_wait(xfull_bar(xch, sl), par, abort_flag, p.err)) {
                ok = false;
                break;
              }
              float u[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) u[j] = xb[(sl * 16 + j) * 32 + lane];
              mbar_arrive(xempty_bar(xch, sl));
              const int feat = fb * BLOCK_M + (int)rank * (BLOCK_M / 2) + quad * 32 + lane;
              if (feat < p.out_features) {
                const int col = ((feat >> 6) << 7) + (feat & 63);
                __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + (size_t)(t.out_row + c0) * p.out_ld + col;
                const int nr = min(16, t.rows - c0);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  if (j < nr) {
                    const float g = __uint_as_float(rg[j]);
                    const float h = __fdividef(g, 1.0f + __expf(-g)) * u[j];
                    const __nv_bfloat16 hi = __float2bfloat16_rn(h);
                    const __nv_bfloat16 lo = __float2bfloat16_rn(h - __bfloat162float(hi));
                    out[(size_t)j * p.out_ld] = hi;
                    out[(size_t)j * p.out_ld + 64] = lo;
                  }
                }
              }
            }
          }
          if (!ok) break;
        } else {
          const bool scaled = (p.row_scale != nullptr) && !t.shared;
          const int feat = fb * 2 * BLOCK_M + (int)rank * BLOCK_M + quad * 32 + lane;
          for (int ci = half; ci < nchunk; ci += 2) {
            const int c0 = ci * 16;
            uint32_t r[16];
            tmem_ld16(tq + c0, r);
            tmem_ld_wait();
            reg_fence16(r);
            if (feat < p.out_features) {
              float* out = static_cast<float*>(p.out) + (size_t)(t.out_row + c0) * p.out_ld + feat;
              const int nr = min(16, t.rows - c0);
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
      if (!ok) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(buf == 0 ? acce_leader0 : acce_leader1);
      if (++buf == S::NUM_BUF) {
        buf = 0;
        buf_phase ^= 1u;
      }
    }
  } else if constexpr (BG) {
    // ------------------------------------------------------------------ token-row loaders (both CTAs)
    // Loader thread b copies 16-byte chunk (b % CHUNKS) of rows b / CHUNKS + j * ROWS_PER_PASS
    // of this CTA's half of the tile's token rows, straight from x by the permuted token ids,
    // into the 128-byte-swizzled layout TMA would have written (chunk c of row r at
    // c ^ (r & 7)), and arrives on the stage's landed barrier when its copies complete.  The
    // relay lane, which issues no copies, waits for each stage to land, fences the writes to the
    // async proxy and reports the stage to the even CTA's full barrier.
    const bool relay = (warp == 2 + NUM_EPI_WARPS + S::NBW);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    if (relay) {
      if (lane == 0) {
        for (int tile = pair; ok && tile < total_tiles; tile += npairs) {
          const Tile t = decode_tile<TN>(tile, p);
          if (t.rows <= 0) continue;
          for (int kb = 0; kb < KB; ++kb) {
            if (!mbar_wait(landed_bar(stage), phase, abort_flag, p.err)) {
              ok = false;
              break;
            }
            fence_proxy_async_smem();
            mbar_arrive_cluster(mapa_shared(full_bar(stage), lrank));
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      __syncwarp();
    } else {
      constexpr int RPT = S::ROWS_PER_THREAD;
      const int b = (warp - 2 - NUM_EPI_WARPS) * 32 + lane;
      const int chunk = b % S::CHUNKS;
      const int r0 = b / S::CHUNKS;
      for (int tile = pair; ok && tile < total_tiles; tile += npairs) {
        const Tile t = decode_tile<TN>(tile, p);
        if (t.rows <= 0) continue;
        const int n_mma = max(32, (t.rows + 31) / 32 * 32);
        const int half = n_mma >> 1;
        const __nv_bfloat16* src[RPT];
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
          const int r = r0 + j * S::ROWS_PER_PASS;  // row within this CTA's half
          const int g = (int)rank * half + r;        // row within the tile
          src[j] = nullptr;
          if (r < half && g < t.rows) {
            const int tok = t.shared ? t.out_row + g + p.shared_b_shift : __ldg(p.b_idx + t.out_row + g);
            src[j] = p.b_x + (size_t)tok * p.b_ld + chunk * 8;
          }
        }
        for (int kb = 0; kb < KB; ++kb) {
          bool got = true;
          if (lane == 0) got = mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.err);
          if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
            ok = false;
            break;
          }
          const uint32_t sb = smem_u32(smem + stage * S::STAGE_BYTES + MB * S::A_BYTES);
#pragma unroll
          for (int j = 0; j < RPT; ++j) {
            const int r = r0 + j * S::ROWS_PER_PASS;
            if (src[j] != nullptr) cp_async16(sb + r * S::ROW_BYTES + ((chunk ^ (r & 7)) << 4), src[j] + kb * BLOCK_K);
          }
          cp_async_arrive_noinc(landed_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      cp_async_commit();  // copies never committed so far form the last group
      cp_async_wait<0>();
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_ALLOC);
  }
}

// ----------------------------------------------------------------------------- host side

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
  }
  return fn;
}

// 2-D bf16 tensor [rows, cols] (cols innermost, contiguous), box bk x box_rows, swizzle of
// 2*bk bytes (bk = 64: 128-byte, bk = 32: 64-byte).
static bool make_tmap(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_rows, int bk) {
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

// The fused gate/up weight [groups, 2*d_ff, K] viewed as 3-D (K, d_ff, 2*groups): one box of
// (bk, box_rows, 2) brings the gate rows and the up rows of the same features.
static bool make_tmap_gateup(CUtensorMap* m, const void* ptr, int64_t groups, int64_t d_ff, int64_t cols,
                             int box_rows, int bk) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)d_ff, (cuuint64_t)(2 * groups)};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)(d_ff * cols * 2)};
  cuuint32_t box[3] = {(cuuint32_t)bk, (cuuint32_t)box_rows, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, bk == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// E4M3 weight codes: 2-D uint8 [rows, cols] with boxes of box_k codes x box_rows rows, and the
// gate/up 3-D view (cols, d_ff, 2*groups) with boxes (box_k, 128, 2).  box_k = 64: 64-byte
// swizzle, so that the converter warps' row-wise 16-byte reads spread over all banks; box_k =
// 128: 128-byte swizzle, the K-major layout the 8-bit MMA reads.
static bool make_tmap_u8(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_rows, int box_k = 64) {
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

static bool make_tmap_u8_gateup(CUtensorMap* m, const void* ptr, int64_t groups, int64_t d_ff, int64_t cols,
                                int box_k = 64) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)d_ff, (cuuint64_t)(2 * groups)};
  cuuint64_t strides[2] = {(cuuint64_t)cols, (cuuint64_t)(d_ff * cols)};
  cuuint32_t box[3] = {(cuuint32_t)box_k, (cuuint32_t)BLOCK_M, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, box_k == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E4M3 activation pieces [rows, pieces, K]: 3-D view (K, pieces, rows) with boxes of
// (128, 1, box_rows), i.e. box_rows rows of 128 codes of one piece, 128-byte swizzle.
static bool make_tmap_pieces(CUtensorMap* m, const void* ptr, int64_t rows, int pieces, int64_t K, int box_rows) {
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

// A-operand maps of a launch: 2-D row slabs, or the gate/up 3-D view for SwiGLU.
static bool make_a_maps(GemmMaps& m, const GemmLaunch& L, bool swiglu, int box_rows, int bk) {
  if (swiglu) {
    const int64_t f = L.a_up_offset;
    if (!make_tmap_gateup(&m.a, L.a_ptr, L.a_rows / (2 * f), f, L.K, box_rows, bk)) return false;
    if (L.a_sh_ptr != nullptr) return make_tmap_gateup(&m.a_sh, L.a_sh_ptr, 1, f, L.K, box_rows, bk);
  } else {
    if (!make_tmap(&m.a, L.a_ptr, L.a_rows, L.K, box_rows, bk)) return false;
    if (L.a_sh_ptr != nullptr) return make_tmap(&m.a_sh, L.a_sh_ptr, L.a_sh_rows, L.K, box_rows, bk);
  }
  m.a_sh = m.a;
  return true;
}

template <int EPI, int TN, int MBLK, bool HILO, int BK>
static cudaError_t launch_variant(const GemmLaunch& L, GemmParams p, cudaStream_t s) {
  using Sh = GemmShape<EPI, TN, MBLK, HILO, BK>;
  static_assert(Sh::SMEM_BYTES <= SMEM_LIMIT, "dynamic shared memory per block");
  if (p.sched_tn % TN != 0 || L.K % BK != 0) return cudaErrorInvalidValue;
  GemmMaps m;
  memset(&m, 0, sizeof(m));
  const int kb_cols = HILO ? 2 * L.K : L.K;  // row length of the activation matrix
  if (!make_a_maps(m, L, EPI == EPI_SWIGLU, EPI == EPI_SWIGLU ? BLOCK_M : BLOCK_M * MBLK, BK))
    return cudaErrorInvalidValue;
  const int KB = L.K / BK;
  if (p.ksplit < 1 || KB % p.ksplit != 0 || (p.ksplit > 1 && p.grp != nullptr)) return cudaErrorInvalidValue;
  for (int i = 0; i < NUM_BOX_H; ++i) {
    const int h = B_BOX << i;
    if (h > TN) break;
    if (!make_tmap(&m.b[i], L.b_ptr, L.b_rows, kb_cols, h, BK)) return cudaErrorInvalidValue;
    if (L.b_sh_ptr != nullptr) {
      if (!make_tmap(&m.b_sh[i], L.b_sh_ptr, L.b_sh_rows, kb_cols, h, BK)) return cudaErrorInvalidValue;
    } else {
      m.b_sh[i] = m.b[i];
    }
  }
  auto kern = grouped_gemm_kernel<EPI, TN, MBLK, HILO, BK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  int grid = L.num_sms;
  const int tiles = L.max_tiles * (p.sched_tn / TN) * p.ksplit;
  if (tiles < grid) grid = tiles;
  if (grid < 1) grid = 1;
  kern<<<grid, NUM_THREADS, Sh::SMEM_BYTES, s>>>(m, p);
  return cudaGetLastError();
}

template <int EPI, int TN, int MBLK, bool HILO>
static cudaError_t launch_fp8_variant(const GemmLaunch& L, GemmParams p, cudaStream_t s) {
  using Sh = Fp8Shape<EPI, TN, MBLK, HILO>;
  static_assert(Sh::SMEM_BYTES <= SMEM_LIMIT, "dynamic shared memory per block");
  if (p.sched_tn % TN != 0 || L.K % 64 != 0 || p.ksplit != 1 || L.a_exp == nullptr) return cudaErrorInvalidValue;
  if (L.a_sh_ptr != nullptr && L.a_sh_exp == nullptr) return cudaErrorInvalidValue;
  GemmMaps m;
  memset(&m, 0, sizeof(m));
  if (EPI == EPI_SWIGLU) {
    const int64_t f = L.a_up_offset;
    if (!make_tmap_u8_gateup(&m.a, L.a_ptr, L.a_rows / (2 * f), f, L.K)) return cudaErrorInvalidValue;
    if (L.a_sh_ptr != nullptr && !make_tmap_u8_gateup(&m.a_sh, L.a_sh_ptr, 1, f, L.K)) return cudaErrorInvalidValue;
  } else {
    if (!make_tmap_u8(&m.a, L.a_ptr, L.a_rows, L.K, BLOCK_M * MBLK)) return cudaErrorInvalidValue;
    if (L.a_sh_ptr != nullptr && !make_tmap_u8(&m.a_sh, L.a_sh_ptr, L.a_sh_rows, L.K, BLOCK_M * MBLK))
      return cudaErrorInvalidValue;
  }
  if (L.a_sh_ptr == nullptr) m.a_sh = m.a;
  const int kb_cols = HILO ? 2 * L.K : L.K;
  for (int i = 0; i < NUM_BOX_H; ++i) {
    const int h = B_BOX << i;
    if (h > TN) break;
    if (!make_tmap(&m.b[i], L.b_ptr, L.b_rows, kb_cols, h, 64)) return cudaErrorInvalidValue;
    if (L.b_sh_ptr != nullptr) {
      if (!make_tmap(&m.b_sh[i], L.b_sh_ptr, L.b_sh_rows, kb_cols, h, 64)) return cudaErrorInvalidValue;
    } else {
      m.b_sh[i] = m.b[i];
    }
  }
  p.a_exp = L.a_exp;
  p.a_sh_exp = L.a_sh_exp != nullptr ? L.a_sh_exp : L.a_exp;
  p.exp_nr = (L.a_rows_per_group + 127) / 128;
  p.exp_nk = (L.K + 127) / 128;
  auto kern = fp8w_gemm_kernel<EPI, TN, MBLK, HILO>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  int grid = L.num_sms;
  const int tiles = L.max_tiles * (p.sched_tn / TN);
  if (tiles < grid) grid = tiles;
  if (grid < 1) grid = 1;
  kern<<<grid, Sh::THREADS, Sh::SMEM_BYTES, s>>>(m, p);
  return cudaGetLastError();
}

template <int EPI, int MBLK, int TN>
static cudaError_t launch_fp8mma_variant(const GemmLaunch& L, GemmParams p, cudaStream_t s) {
  using Sh = F8Shape<EPI, MBLK, TN>;
  static_assert(Sh::SMEM_BYTES <= SMEM_LIMIT, "dynamic shared memory per block");
  if (p.sched_tn % Sh::TN != 0 || L.K % Sh::BLOCK_K != 0 || p.ksplit != 1) return cudaErrorInvalidValue;
  if (L.a_exp == nullptr || L.b_exp == nullptr || (L.a_sh_ptr != nullptr && L.a_sh_exp == nullptr))
    return cudaErrorInvalidValue;
  if (EPI == EPI_SWIGLU && L.a_up_offset % 128 != 0) return cudaErrorInvalidValue;  // slabs on scale tiles
  GemmMaps m;
  memset(&m, 0, sizeof(m));
  if (EPI == EPI_SWIGLU) {
    const int64_t f = L.a_up_offset;
    if (!make_tmap_u8_gateup(&m.a, L.a_ptr, L.a_rows / (2 * f), f, L.K, 128)) return cudaErrorInvalidValue;
    if (L.a_sh_ptr != nullptr && !make_tmap_u8_gateup(&m.a_sh, L.a_sh_ptr, 1, f, L.K, 128))
      return cudaErrorInvalidValue;
  } else {
    if (!make_tmap_u8(&m.a, L.a_ptr, L.a_rows, L.K, BLOCK_M * MBLK, 128)) return cudaErrorInvalidValue;
    if (L.a_sh_ptr != nullptr && !make_tmap_u8(&m.a_sh, L.a_sh_ptr, L.a_sh_rows, L.K, BLOCK_M * MBLK, 128))
      return cudaErrorInvalidValue;
  }
  if (L.a_sh_ptr == nullptr) m.a_sh = m.a;
  for (int i = 0; (B_BOX << i) <= Sh::TN; ++i)
    if (!make_tmap_pieces(&m.b[i], L.b_ptr, L.b_rows, Sh::PIECES, L.K, B_BOX << i)) return cudaErrorInvalidValue;
  p.a_exp = L.a_exp;
  p.a_sh_exp = L.a_sh_exp != nullptr ? L.a_sh_exp : L.a_exp;
  p.exp_nr = (L.a_rows_per_group + 127) / 128;
  p.exp_nk = (L.K + 127) / 128;
  p.b_exp = L.b_exp;
  auto kern = fp8mma_gemm_kernel<EPI, MBLK, TN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  int grid = L.num_sms;
  const int tiles = L.max_tiles * (p.sched_tn / Sh::TN);
  if (tiles < grid) grid = tiles;
  if (grid < 1) grid = 1;
  kern<<<grid, NUM_THREADS, Sh::SMEM_BYTES, s>>>(m, p);
  return cudaGetLastError();
}

template <int EPI, int TN, bool HILO, int BK, int TMEM_ALLOC, int NP, int MB, bool BG = false>
static cudaError_t launch_pair_variant(const GemmLaunch& L, GemmParams p, cudaStream_t s) {
  using Sh = PairShape<EPI, TN, HILO, BK, TMEM_ALLOC, MB, BG>;
  static_assert(Sh::SMEM_BYTES <= SMEM_LIMIT, "dynamic shared memory per block");
  if (p.sched_tn % TN != 0 || L.K % BK != 0) return cudaErrorInvalidValue;
  GemmMaps m;
  memset(&m, 0, sizeof(m));
  const int kb_cols = HILO ? 2 * L.K : L.K;
  if (!make_a_maps(m, L, EPI == EPI_SWIGLU, Sh::A_BOX, BK)) return cudaErrorInvalidValue;
  if (BG) {
    if (L.b_gather_x == nullptr || L.b_gather_idx == nullptr) return cudaErrorInvalidValue;
    p.b_x = static_cast<const __nv_bfloat16*>(L.b_gather_x);
    p.b_idx = L.b_gather_idx;
    p.b_ld = L.K;
  }
  for (int i = 0; i < (BG ? 0 : NUM_BOX_H); ++i) {
    const int h = B_BOX << i;
    if (h > Sh::HALF) break;
    if (!make_tmap(&m.b[i], L.b_ptr, L.b_rows, kb_cols, h, BK)) return cudaErrorInvalidValue;
    if (L.b_sh_ptr != nullptr) {
      if (!make_tmap(&m.b_sh[i], L.b_sh_ptr, L.b_sh_rows, kb_cols, h, BK)) return cudaErrorInvalidValue;
    } else {
      m.b_sh[i] = m.b[i];
    }
  }
  auto kern = pair_gemm_kernel<EPI, TN, HILO, BK, TMEM_ALLOC, NP, MB, BG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  // the schedule counts pair feature blocks of one slab; a CTA of MB slabs, in a cluster of NP
  // pairs, covers MB * NP of them
  p.num_mblocks = (p.num_mblocks + NP * MB - 1) / (NP * MB);
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.blockDim = dim3(Sh::THREADS);
  cfg.dynamicSmemBytes = Sh::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2 * NP;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // as many clusters as can be resident at once (persistent kernel), at most one per tile
  static int max_clusters = 0;
  if (max_clusters == 0) {
    cfg.gridDim = dim3(2 * NP * (L.num_sms / (2 * NP)));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = L.num_sms / (2 * NP);
    }
    max_clusters = n;
  }
  int clusters = max_clusters;
  if (MOE_PAIR_MAX_CLUSTERS > 0 && clusters > MOE_PAIR_MAX_CLUSTERS) clusters = MOE_PAIR_MAX_CLUSTERS;
  const int tiles = (L.max_tiles + NP * MB - 1) / (NP * MB) * (p.sched_tn / TN);
  if (tiles < clusters) clusters = tiles;
  if (clusters < 1) clusters = 1;
  cfg.gridDim = dim3(2 * NP * clusters);
  e = cudaLaunchKernelEx(&cfg, kern, m, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

int gemm_features_per_tile(int epi, int mblk) { return epi == EPI_SWIGLU ? BLOCK_M : BLOCK_M * mblk; }

cudaError_t launch_grouped_gemm(const GemmLaunch& L, cudaStream_t s) {
  const int kernel_tn = L.kernel_tn > 0 ? L.kernel_tn : L.TN;
  GemmParams p;
  p.K = L.K;
  p.num_mblocks = L.num_mblocks;
  p.a_rows_per_group = L.a_rows_per_group;
  p.a_up_offset = L.a_up_offset;
  p.out_features = L.out_features;
  p.out_ld = L.out_ld;
  p.out = L.out;
  p.row_scale = L.row_scale;
  p.n_routed = L.n_routed;
  p.shared_b_shift = L.shared_b_shift;
  p.grp = L.grp;
  p.rt2g = L.rt2g;
  p.n_groups_total = L.n_routed + (L.a_sh_ptr != nullptr ? 1 : 0);
  p.sched_tn = L.TN;
  p.ksplit = L.ksplit > 0 ? L.ksplit : 1;
  p.split_stride = L.split_stride;
  p.dense_rows = L.dense_rows;
  p.err = L.err;
  p.b_x = nullptr;
  p.b_idx = nullptr;
  p.b_ld = 0;
  p.a_exp = nullptr;
  p.a_sh_exp = nullptr;
  p.exp_nr = p.exp_nk = 0;
  p.b_exp = nullptr;
  if (L.q8 == 2) {
    // FP8 weight codes straight into the MMA, E4M3-piece activations, 16-, 32- or 64-row token
    // tiles (the down projection's 64-row tiles on one 128-feature slab: its four pieces then
    // fill N = 256)
    if (L.epi == EPI_SWIGLU && kernel_tn == 16) return launch_fp8mma_variant<EPI_SWIGLU, 1, 16>(L, p, s);
    if (L.epi == EPI_SWIGLU && kernel_tn == 32) return launch_fp8mma_variant<EPI_SWIGLU, 1, 32>(L, p, s);
    if (L.epi == EPI_SWIGLU && kernel_tn == 64) return launch_fp8mma_variant<EPI_SWIGLU, 1, 64>(L, p, s);
    if (L.epi != EPI_SWIGLU && kernel_tn == 16 && L.mblk == 2) return launch_fp8mma_variant<EPI_F32, 2, 16>(L, p, s);
    if (L.epi != EPI_SWIGLU && kernel_tn == 32 && L.mblk == 2) return launch_fp8mma_variant<EPI_F32, 2, 32>(L, p, s);
    if (L.epi != EPI_SWIGLU && kernel_tn == 64 && L.mblk == 1) return launch_fp8mma_variant<EPI_F32, 1, 64>(L, p, s);
    return cudaErrorInvalidValue;
  }
  if (L.q8) {
    // FP8 weight codes: single-CTA kernels with 64-row token sub-tiles
    if (L.epi == EPI_SWIGLU && kernel_tn == 64) return launch_fp8_variant<EPI_SWIGLU, 64, 1, false>(L, p, s);
    if (L.epi != EPI_SWIGLU && L.hilo && kernel_tn == 64 && L.mblk == 2)
      return launch_fp8_variant<EPI_F32, 64, 2, true>(L, p, s);
    return cudaErrorInvalidValue;
  }
  constexpr int TNP = MOE_TN_PREFILL;
  constexpr int TN2 = MOE_TN_DOWN;
  if (L.pair) {
    // two weight slabs per CTA where the pair feature blocks divide evenly, else one
    const bool even = (L.num_mblocks % (2 * (L.epi == EPI_SWIGLU ? MOE_G1_NP : MOE_G2_NP))) == 0;
    if (L.epi == EPI_SWIGLU && kernel_tn == TNP && L.b_gather_x != nullptr) {
      if (MOE_G1_MB == 2 && even)
        return launch_pair_variant<EPI_SWIGLU, TNP, false, MOE_G1_BK, MOE_PAIR_TMEM, 1, 2, true>(L, p, s);
      return launch_pair_variant<EPI_SWIGLU, TNP, false, MOE_G1_BK, MOE_PAIR_TMEM, 1, 1, true>(L, p, s);
    }
    if (L.epi == EPI_SWIGLU && kernel_tn == TNP) {
      if (MOE_G1_MB == 2 && even)
        return launch_pair_variant<EPI_SWIGLU, TNP, false, MOE_G1_BK, MOE_PAIR_TMEM, MOE_G1_NP, 2>(L, p, s);
      return launch_pair_variant<EPI_SWIGLU, TNP, false, MOE_G1_BK, MOE_PAIR_TMEM, MOE_G1_NP, 1>(L, p, s);
    }
    if (L.epi != EPI_SWIGLU && L.hilo && kernel_tn == TN2 && L.mblk == 2) {
      if (MOE_G2_MB == 2 && even)
        return launch_pair_variant<EPI_F32, TN2, true, MOE_G2_BK, MOE_PAIR_TMEM, MOE_G2_NP, 2>(L, p, s);
      return launch_pair_variant<EPI_F32, TN2, true, MOE_G2_BK, MOE_PAIR_TMEM, MOE_G2_NP, 1>(L, p, s);
    }
    return cudaErrorInvalidValue;
  }
  if (L.epi == EPI_SWIGLU) {
    if (kernel_tn == TNP) return launch_variant<EPI_SWIGLU, TNP, 1, false, MOE_G1_BK>(L, p, s);
    if (kernel_tn == 64) return launch_variant<EPI_SWIGLU, 64, 1, false, 64>(L, p, s);
    return cudaErrorInvalidValue;
  }
  if (L.hilo) {
    if (kernel_tn == TN2 && L.mblk == MOE_G2_MBLK) return launch_variant<EPI_F32, TN2, MOE_G2_MBLK, true, MOE_G2_BK>(L, p, s);
    if (kernel_tn == 64 && L.mblk == 1) return launch_variant<EPI_F32, 64, 1, true, 64>(L, p, s);
    if (kernel_tn == 64 && L.mblk == 2) return launch_variant<EPI_F32, 64, 2, true, 64>(L, p, s);
    return cudaErrorInvalidValue;
  }
  if (kernel_tn == TNP && L.mblk == 2) return launch_variant<EPI_F32, TNP, 2, false, 64>(L, p, s);
  if (kernel_tn == TNP && L.mblk == 1) return launch_variant<EPI_F32, TNP, 1, false, 64>(L, p, s);
  if (kernel_tn == 64 && L.mblk == 2) return launch_variant<EPI_F32, 64, 2, false, 64>(L, p, s);
  if (kernel_tn == 64 && L.mblk == 1) return launch_variant<EPI_F32, 64, 1, false, 64>(L, p, s);
  return cudaErrorInvalidValue;
}

}  // namespace moe
