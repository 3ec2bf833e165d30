// FP8 (E4M3) and MXFP4 (E2M1) expert weights in the grouped GEMMs ("DeepSeek-V4 MoE", section
// "FP4 QAT 怎么做到反量化无损": FP8 with one power-of-two scale per 128 x 128 tile, FP4 with one
// per 1 x 32 sub-block, losslessly dequantised to the FP8 form).  Three kernel families:
//   * fp8mma_gemm_kernel: FP8 codes as the 8-bit MMA's A operand, as stored; the activations as
//     E4M3 pieces (d and d_ff multiples of 128);
//   * fp4mma_gemm_kernel: MXFP4 codes as the A operand of the block-scaled MMA, as stored, with
//     their 1 x 32 sub-block scales applied by the tensor cores; the activations as E4M3 pieces;
//   * fp8w_gemm_kernel: FP8 codes widened to bf16 into Tensor Memory and multiplied by the bf16
//     activations (any shape).
#include "gemm_common.cuh"

namespace moe {

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
  sync_and_quiesce(abort_flag);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, S::TMEM_COLS);
  }
}

// ============================================================================ FP8 MMA variant
// The single-CTA kernel with the E4M3 weight codes as the MMA's A operand as they are (tcgen05
// kind::f8f6f4, twice the bf16 rate), one power-of-two scale per 128 x 128 code tile ("DeepSeek-V4
// MoE", section "FP4 QAT 怎么做到反量化无损").  B holds the token rows as E4M3 pieces with one
// power-of-two scale per row and piece p weighted 2^(-4p) (x: 2 pieces, h: 4; see the split
// kernel).  The pieces of a tile's
// token rows sit one after another in the stage (piece p at rows p * n .. p * n + n - 1), so one
// MMA per slab and K step multiplies all of them (N = pieces * n) and reads the A tile from
// shared memory once.  A stage is one 128-wide K tile, so a single weight scale 2^e covers each
// slab of it: the MMAs of K tile kt write their own slot of a ring in Tensor Memory, and the
// epilogue warps add (sum of the piece columns x 2^(-4p)) * 2^e(kt) into fp32 registers and release the
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
  static_assert(PIECES == 2 || PIECES == 4, "pieces are summed in pairs");
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
#if MOE_TEST_UNSET_WAIT
    // test build: wait on a phase nothing completes (only these warps arrive on it), so the
    // wait runs out and the kernel takes its abort path
    if (!mbar_wait(sempty_bar(0), 0, abort_flag, p.err)) ok = false;
#endif
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
              const float scp = sc * (pp == 0 ? 1.0f : 0.00390625f);  // 2^e * 2^(-4 pp), exact
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
                acc[a][j] = fmaf(fmaf(__uint_as_float(r0[1][j]), 0.0625f, __uint_as_float(r0[0][j])), scp, acc[a][j]);
              if (cols > 16) {
                reg_fence16(r1[0]);
                reg_fence16(r1[1]);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                  acc[a][16 + j] =
                      fmaf(fmaf(__uint_as_float(r1[1][j]), 0.0625f, __uint_as_float(r1[0][j])), scp, acc[a][16 + j]);
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
  sync_and_quiesce(abort_flag);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// ============================================================================ MXFP4 variant
// Native MXFP4 weights (E2M1 codes, one power-of-two scale 2^s per 1 x 32 sub-block; "DeepSeek-V4
// MoE", section "FP4 QAT 怎么做到反量化无损": FP4 weights with 1 x 32 sub-block scales used
// natively at inference) on the block-scaled tensor-core MMA (tcgen05.mma kind::mxf8f6f4 with
// block_scale, one UE8M0 scale per row and per 32 K values of each operand).  TMA streams the
// stored codes (two per byte) as 16 x 4-bit groups, each unpacked into the low 8 bytes of a 16-byte
// chunk of shared memory -- the form in which the MMA reads E2M1 -- beside the token rows'
// E4M3 pieces; the codes reach the tensor cores as they are stored.  The sub-block exponents
// become the A scales (2^s, UE8M0 s + 127) in Tensor Memory, written per stage by four scale
// warps; the B scales are the pieces' fixed weights 2^(-4p), so every piece of every stage
// accumulates into one fp32 accumulator per tile, and the epilogue applies the token rows'
// exponents 2^e (and the gate weights) once.
//
// Scale-factor layout in Tensor Memory, as used here for M = 128 (measured on this part: row m
// of A takes its scale from lane m, column c0 + m / 32, byte `sfa_id` of the instruction
// descriptor, c0 the scale address's column; a scale address whose column is not a multiple of
// 4 raised a misaligned-address fault, so every scale address here is a multiple of 4 columns):
// the scale warp of lane quadrant q writes its 32 rows' four sub-block scales of a 128-wide K
// step as one word at column c0 + q, and the four MMAs of the step select bytes 0..3.  The B
// scales are written uniform (every lane, byte and column of an 8-column region per piece), so
// their layout does not matter.

// The parameter block plus the MXFP4 sub-block exponents [mats, rows, K/32] (int8) of the routed
// and the shared weights.
struct Fp4Params : GemmParams {
  const int8_t* a_sub;
  const int8_t* a_sh_sub;
};

// Stages whose A scales a scale writer loads at once (see the writers' loop).
constexpr int F4_SF_CHUNK = 8;

template <int EPI, int MBLK, int TN_>
struct F4Shape {
  static constexpr int TN = TN_;
  static constexpr int BLOCK_K = 128;                    // codes per stage: one TMA box, four MMAs
  static constexpr int NUM_A = (EPI == EPI_SWIGLU) ? 2 : MBLK;
  static constexpr int A_SLAB = BLOCK_M * BLOCK_K;       // 128 rows x 128 bytes (codes in 16-byte chunks)
  static constexpr int A_BYTES = NUM_A * A_SLAB;
  static constexpr int PIECES = (EPI == EPI_SWIGLU) ? 2 : 4;
  static constexpr int B_PIECE = TN * BLOCK_K;           // TN token rows x 128 E4M3 codes
  static constexpr int STAGE = A_BYTES + PIECES * B_PIECE;
  static constexpr int TX_BYTES = A_BYTES / 2 + PIECES * B_PIECE;  // bytes a stage's TMA loads move
  static constexpr int STAGES_FIT = (SMEM_LIMIT - 1024 - 512) / STAGE;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int SMEM_BYTES = STAGES * STAGE + 1024 + 512;
  // Decode-sized tiles (TN <= 32) put the pieces side by side in N: one MMA per slab and K step
  // covers every piece, each into its own accumulator columns, summed by the epilogue (so the
  // B scales are all 1).  Wider tiles issue one MMA per piece into one accumulator per slab, the
  // piece's weight 2^(-4p) applied as its B scale.
  static constexpr bool PIN = TN <= 32;
  static constexpr int ACC_COLS = NUM_A * (PIN ? PIECES : 1) * TN;   // one accumulator buffer
  static constexpr int SFB_REGIONS = PIN ? 1 : PIECES;
  static constexpr int SFB_COLS = 8;                     // one B-scale region
  static constexpr int SFA_COLS = STAGES * NUM_A * 4;    // per stage and slab: one column per lane quadrant
  static constexpr int NUM_BUF = (2 * ACC_COLS + SFB_REGIONS * SFB_COLS + SFA_COLS <= 512) ? 2 : 1;
  static constexpr int SFB_COL0 = NUM_BUF * ACC_COLS;    // after the accumulator buffers
  static constexpr int SFA_COL0 = SFB_COL0 + SFB_REGIONS * SFB_COLS;
  static constexpr int TMEM_COLS = (SFA_COL0 + SFA_COLS <= 256) ? 256 : 512;
  static constexpr int SF_WARP0 = 2 + NUM_EPI_WARPS;     // four scale warps after the epilogue warps
  static constexpr int THREADS = (SF_WARP0 + 4) * 32;
  static constexpr int FEATS = (EPI == EPI_SWIGLU) ? BLOCK_M : BLOCK_M * MBLK;
  static_assert(TN % 16 == 0 && TN <= 64, "token tile");
  static_assert(!PIN || PIECES * TN <= 256, "MMA N");
  static_assert(STAGES >= 2, "pipeline needs two stages");
  static_assert(A_SLAB % 1024 == 0 && B_PIECE % 1024 == 0 && STAGE % 1024 == 0, "swizzled tiles on 1024 B");
  static_assert(SFB_COL0 % 4 == 0 && SFA_COL0 % 4 == 0, "scale addresses on 4-column boundaries");
  static_assert(SFA_COL0 + SFA_COLS <= TMEM_COLS, "TMEM: accumulators + scales");
  static_assert((3 * STAGES + 4) * 8 + 8 <= 512, "barrier area");
  static_assert(EPI == EPI_F32 || MBLK == 1, "SwiGLU variant");
};

template <int EPI, int MBLK, int TN_>
__global__ void __launch_bounds__(F4Shape<EPI, MBLK, TN_>::THREADS, 1)
    fp4mma_gemm_kernel(const __grid_constant__ GemmMaps maps, const Fp4Params p) {
  using S = F4Shape<EPI, MBLK, TN_>;
  constexpr int TN = S::TN;
  constexpr int ST = S::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ST * S::STAGE);
  // bars: full[ST], empty[ST], sfull[ST], accf[2], acce[2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * ST + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (ST + s); };
  auto sfull_bar = [&](int s) { return bar0 + 8u * (2 * ST + s); };
  auto accf_bar = [&](int a) { return bar0 + 8u * (3 * ST + a); };
  auto acce_bar = [&](int a) { return bar0 + 8u * (3 * ST + 2 + a); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(sfull_bar(s), 4);  // one arrival per scale warp
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
    tma_prefetch_desc(&maps.b[0]);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), S::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (warp >= S::SF_WARP0) {
    // B scales: region p holds 2^(-4p) (UE8M0 127 - 4p; a single region of 1 with the pieces
    // along N), the same in every lane, byte and column of the region
    const uint32_t tq = tmem_base + (uint32_t((warp & 3) * 32) << 16) + S::SFB_COL0;
#pragma unroll
    for (int pc = 0; pc < S::SFB_REGIONS; ++pc)
#pragma unroll
      for (int c = 0; c < S::SFB_COLS; ++c) tmem_st1(tq + pc * S::SFB_COLS + c, (127u - 4u * pc) * 0x01010101u);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

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
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t sr = smem_u32(smem + stage * S::STAGE);
          const uint32_t fb = full_bar(stage);
          // transaction bytes: the codes as stored (4 bits each; the gaps in shared memory do not
          // count) and the pieces
          mbar_arrive_expect_tx(fb, S::TX_BYTES);
          if (EPI == EPI_SWIGLU) {
            tma_load_3d(sr, ta, fb, kb * S::BLOCK_K, t.mb * BLOCK_M, t.shared ? 0 : 2 * t.g);  // gate, up
          } else {
            tma_load_2d(sr, ta, fb, kb * S::BLOCK_K, a_row);                                   // MBLK slabs
          }
#pragma unroll
          for (int pc = 0; pc < S::PIECES; ++pc)
            tma_load_3d(sr + S::A_BYTES + pc * S::B_PIECE, &maps.b[0], fb, kb * S::BLOCK_K, pc, t.b_row);
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
      int stage = 0, buf = 0;
      uint32_t phase = 0, buf_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        const Tile t = decode_tile<TN>(tile, p);
        if (t.rows <= 0) continue;
        if (!mbar_wait(acce_bar(buf), buf_phase ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + buf * S::ACC_COLS;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag, p.err) ||
              !mbar_wait(sfull_bar(stage), phase, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sr = smem_u32(smem + stage * S::STAGE);
          const uint32_t sfa0 = tmem_base + S::SFA_COL0 + stage * S::NUM_A * 4;
#pragma unroll
          for (int kk = 0; kk < S::BLOCK_K / 32; ++kk) {
#pragma unroll
            for (int a = 0; a < S::NUM_A; ++a) {
              const uint64_t ad = smem_desc_sw(sr + a * S::A_SLAB, 128) + 2 * kk;
              if (S::PIN) {  // all pieces (PIECES * TN rows of B) into piece-wise accumulator columns
                const uint64_t bd = smem_desc_sw(sr + S::A_BYTES, 128) + 2 * kk;
                tc_mma_mx(d0 + a * S::PIECES * TN, ad, bd, idesc_mx_e2m1_e4m3(S::PIECES * TN, kk), sfa0 + a * 4,
                          tmem_base + S::SFB_COL0, (kb | kk) ? 1u : 0u);
              } else {
#pragma unroll
                for (int pc = 0; pc < S::PIECES; ++pc) {
                  const uint64_t bd = smem_desc_sw(sr + S::A_BYTES + pc * S::B_PIECE, 128) + 2 * kk;
                  tc_mma_mx(d0 + a * TN, ad, bd, idesc_mx_e2m1_e4m3(t.n_mma, kk), sfa0 + a * 4,
                            tmem_base + S::SFB_COL0 + pc * S::SFB_COLS, (kb | kk | pc) ? 1u : 0u);
                }
              }
            }
          }
          tc_commit(empty_bar(stage));
          if (++stage == ST) {
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
  } else if (warp < S::SF_WARP0) {
    // ------------------------------------------------------------------ epilogue
    // Warp w reads TMEM lane quadrant w % 4 (weight rows 32 (w % 4) + lane) and the 16-column
    // chunks of its half; each column (a token row) is scaled by 2^e of the row's pieces (and,
    // in the down projection, by the row's gate weight).
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    int buf = 0;
    uint32_t buf_phase = 0;
#if MOE_TEST_UNSET_WAIT
    // test build: wait on a phase nothing completes (only these warps arrive on it), so the
    // wait runs out and the kernel takes its abort path
    mbar_wait(acce_bar(0), 0, abort_flag, p.err);
#endif
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      const Tile t = decode_tile<TN>(tile, p);
      if (t.rows <= 0) continue;
      if (!mbar_wait(accf_bar(buf), buf_phase, abort_flag, p.err)) break;
      tc_fence_after();
      const uint32_t tq = tmem_base + (uint32_t(quad * 32) << 16) + buf * S::ACC_COLS;
      const int nchunk = (t.rows + 15) >> 4;
      for (int ci = half; ci < nchunk; ci += 2) {
        const int c0 = ci * 16;
        const int nr = min(16, t.rows - c0);
        const bool rvalid = lane < nr;
        float cs_l = rvalid ? __int_as_float((127 + __ldg(p.b_exp + t.b_row + c0 + lane)) << 23) : 0.0f;
        if (EPI == EPI_F32 && p.row_scale != nullptr && !t.shared && rvalid)
          cs_l *= __ldg(p.row_scale + t.out_row + c0 + lane);
        // slab a's 16 columns at c0, the pieces summed with weights 2^(-4p) where they lie along N
        auto load_slab = [&](int a, float(&v)[16]) {
          if (S::PIN) {
            uint32_t r[S::PIECES][16];
#pragma unroll
            for (int pc = 0; pc < S::PIECES; ++pc) tmem_ld16(tq + (a * S::PIECES + pc) * TN + c0, r[pc]);
            tmem_ld_wait();
#pragma unroll
            for (int pc = 0; pc < S::PIECES; ++pc) reg_fence16(r[pc]);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              float x = fmaf(__uint_as_float(r[1][j]), 0.0625f, __uint_as_float(r[0][j]));
              if (S::PIECES == 4)
                x = fmaf(fmaf(__uint_as_float(r[S::PIECES - 1][j]), 0.0625f, __uint_as_float(r[S::PIECES - 2][j])),
                         0.00390625f, x);
              v[j] = x;
            }
          } else {
            uint32_t r[16];
            tmem_ld16(tq + a * TN + c0, r);
            tmem_ld_wait();
            reg_fence16(r);
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
          }
        };
        float cs[16];  // the columns' scales
#pragma unroll
        for (int j = 0; j < 16; ++j) cs[j] = __shfl_sync(0xffffffffu, cs_l, j);
        const bool skip = p.out_rows > 0 && (bad_index(t.out_row + c0, p.out_rows, p.err) ||
                                             bad_index(t.out_row + c0 + nr - 1, p.out_rows, p.err));
        float* out = static_cast<float*>(p.out) + (size_t)(t.out_row + c0) * p.out_ld;
        if (EPI == EPI_SWIGLU) {
          float g[16], u[16];
          load_slab(0, g);
          load_slab(1, u);
          const int feat = t.mb * BLOCK_M + quad * 32 + lane;
          if (!skip && feat < p.out_features) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (j < nr) {
                const float gj = g[j] * cs[j], uj = u[j] * cs[j];
                out[(size_t)j * p.out_ld + feat] = __fdividef(gj, 1.0f + __expf(-gj)) * uj;
              }
            }
          }
        } else {
#pragma unroll
          for (int a = 0; a < S::NUM_A; ++a) {
            float v[16];
            load_slab(a, v);
            const int feat = t.mb * S::FEATS + a * BLOCK_M + quad * 32 + lane;
            if (!skip && feat < p.out_features) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (j < nr) out[(size_t)j * p.out_ld + feat] = v[j] * cs[j];
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce_bar(buf));
      if (++buf == S::NUM_BUF) {
        buf = 0;
        buf_phase ^= 1u;
      }
    }
  } else {
    // ------------------------------------------------------------------ A-scale writers
    // Warp w owns TMEM lane quadrant q = w % 4, i.e. weight rows r = 32 q + lane of every slab.
    // For each stage the thread loads the row's four sub-block exponents s of the stage's 128 K
    // values (one word, byte j = sub-block j), turns them into UE8M0 bytes s + 127 (s below -127,
    // values under 2^-127 * 6, taken as -127) and stores the word at column q of the stage's
    // slot of each slab, once the stage's previous MMAs have completed (the stage's empty barrier).
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int kb32 = p.K / 32;  // sub-blocks per weight row
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
      const Tile t = decode_tile<TN>(tile, p);
      if (t.rows <= 0) continue;
      const int8_t* sub = t.shared ? p.a_sh_sub : p.a_sub + (size_t)t.g * p.a_rows_per_group * kb32;
      const uint32_t* srow[S::NUM_A];
#pragma unroll
      for (int a = 0; a < S::NUM_A; ++a) {
        const int base = (EPI == EPI_SWIGLU) ? a * p.a_up_offset + t.mb * BLOCK_M : t.mb * S::FEATS + a * BLOCK_M;
        const int row = min(base + r, p.a_rows_per_group - 1);  // rows past the matrix: any valid row
        srow[a] = reinterpret_cast<const uint32_t*>(sub + (size_t)row * kb32);
      }
      // The words of F4_SF_CHUNK stages are loaded together and used before the first of those
      // stages reports: the report (an arrive with release semantics) then never waits for a load
      // still in flight, which would put a global-memory latency into every stage.
      for (int kb0 = 0; ok && kb0 < KB; kb0 += F4_SF_CHUNK) {
        uint32_t w[F4_SF_CHUNK][S::NUM_A];
#pragma unroll
        for (int j = 0; j < F4_SF_CHUNK; ++j)
#pragma unroll
          for (int a = 0; a < S::NUM_A; ++a)
            w[j][a] = (kb0 + j < KB) ? __vadd4(__vmaxs4(__ldg(srow[a] + kb0 + j), 0x81818181u), 0x7F7F7F7Fu) : 0u;
#pragma unroll
        for (int j = 0; j < F4_SF_CHUNK; ++j) {
          if (kb0 + j >= KB) break;
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ts = tmem_base + (uint32_t(quad * 32) << 16) + S::SFA_COL0 + stage * S::NUM_A * 4 + quad;
#pragma unroll
          for (int a = 0; a < S::NUM_A; ++a) tmem_st1(ts + a * 4, w[j][a]);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(sfull_bar(stage));
          if (++stage == ST) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  }

  tc_fence_before();
  sync_and_quiesce(abort_flag);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, S::TMEM_COLS);
  }
}

// ============================================================================ CTA-pair FP8 (prefill)
// FP8 weights at prefill batches, on the 2-SM MMA of the bf16 CTA-pair kernels.  TMA streams each
// CTA's 128 weight rows as E4M3 codes (64-byte rows per 64-wide K step: half the bf16 bytes) with
// the token rows as bf16 (the dispatched x rows, or the (hi, lo) activation pair), four converter
// warps per CTA widen the codes to bf16 q * 2^e (exact; e the 128 x 128 tile's exponent) into a
// ring of 128-byte-swizzled A slabs in shared memory, and the even CTA's MMA thread multiplies
// them with bf16 MMAs exactly as the bf16 pair kernel does.  The layer is then the bf16 layer on
// the dequantised weights with bf16 activations, the definition the FP8 weight format has.  Roles
// (704 threads): warp 0 TMA producer, warp 1 TMEM owner + MMA issuer (even CTA), warps 2..9
// epilogue, warps 10..21 converters in three groups of four that take the stages in turn (thread r
// of a group widens weight row r of its stages).  Measured (V4-Flash T=8192): one group 8.28 ms,
// two 5.48, three 4.82 ms per forward (the earlier single-CTA FP8 prefill kernels: 5.87 ms); with
// the conversion replaced by a plain copy, two groups gave 4.35 ms: the conversion's integer work
// and its place in each stage's round trip (codes landed -> widened -> multiplied -> released)
// bound it, not the halved weight stream.
template <int EPI, bool HILO>
struct Fp8PairShape {
  static constexpr int TN = 256;
  static constexpr int HALF = TN / 2;
  static constexpr int BLOCK_K = 64;
  static constexpr int ROW_BYTES = 128;                // bf16 rows of B and of the widened A
  static constexpr int RAW_A = BLOCK_M * BLOCK_K;      // 128 rows x 64 codes (64-byte swizzle)
  static constexpr int NUM_B = HILO ? 2 : 1;
  static constexpr int B_BYTES = HALF * ROW_BYTES;     // one activation operand, this CTA's rows
  static constexpr int RAW_STAGE = RAW_A + NUM_B * B_BYTES;
  static constexpr int A_BYTES = BLOCK_M * ROW_BYTES;  // one widened slab
  static constexpr int CSLOTS = 4;                     // widened slabs in flight
  static constexpr int XCH = (EPI == EPI_SWIGLU) ? 4 : 0;
  static constexpr int XBUF_BYTES = XCH * 2 * 16 * 32 * 4;
  static constexpr int STAGES_FIT = (SMEM_LIMIT - 1024 - 512 - XBUF_BYTES - CSLOTS * A_BYTES) / RAW_STAGE;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int SMEM_BYTES = CSLOTS * A_BYTES + STAGES * RAW_STAGE + XBUF_BYTES + 1024 + 512;
  static constexpr int ACC_COLS = TN;
  static constexpr int NUM_BUF = 2;
  static constexpr int TMEM_COLS = 512;
  static constexpr int CVT_GROUPS = 3;                 // groups of four converter warps, stages in turn
  static constexpr int NUM_CVT_WARPS = 4 * CVT_GROUPS;
  static constexpr int CVT_WARP0 = 2 + NUM_EPI_WARPS;
  static constexpr int THREADS = (2 + NUM_EPI_WARPS + NUM_CVT_WARPS) * 32;
  static constexpr int A_BOX = (EPI == EPI_SWIGLU) ? BLOCK_M / 2 : BLOCK_M;  // code rows per box
  // barriers: full, rfull, empty per stage; cfull, cempty per slab; acc full/empty x2; exchange
  static constexpr int NUM_BARS = 3 * STAGES + 2 * CSLOTS + 4 + 4 * XCH;
  static_assert(NUM_BARS * 8 + 8 <= 512, "barrier area");
  static_assert(STAGES >= 2, "pipeline needs two stages");
  static_assert(RAW_STAGE % 1024 == 0 && A_BYTES % 1024 == 0 && RAW_A % 1024 == 0, "swizzled tiles on 1024 B");
};

template <int EPI, bool HILO>
__global__ void __launch_bounds__(Fp8PairShape<EPI, HILO>::THREADS, 1)
    fp8w_pair_gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmParams p) {
  using S = Fp8PairShape<EPI, HILO>;
  constexpr int TN = S::TN;
  constexpr int STAGES = S::STAGES;
  constexpr int CS = S::CSLOTS;
  constexpr int BLOCK_K = S::BLOCK_K;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* aslab = smem;                                 // CSLOTS widened A slabs
  uint8_t* raw = smem + CS * S::A_BYTES;                 // STAGES x (codes, B)
  float* xbuf = reinterpret_cast<float*>(raw + STAGES * S::RAW_STAGE);
  uint64_t* bars = reinterpret_cast<uint64_t*>(raw + STAGES * S::RAW_STAGE + S::XBUF_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + S::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };                      // B bytes, even CTA
  auto rfull_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };          // this CTA's codes
  auto empty_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };      // stage consumed
  auto cfull_bar = [&](int c) { return bar0 + 8u * (3 * STAGES + c); };      // slab widened (even CTA)
  auto cempty_bar = [&](int c) { return bar0 + 8u * (3 * STAGES + CS + c); };  // slab consumed
  auto accf_bar = [&](int a) { return bar0 + 8u * (3 * STAGES + 2 * CS + a); };
  auto acce_bar = [&](int a) { return bar0 + 8u * (3 * STAGES + 2 * CS + 2 + a); };
  auto xfull_bar = [&](int x, int sl) { return bar0 + 8u * (3 * STAGES + 2 * CS + 4 + 2 * x + sl); };
  auto xempty_bar = [&](int x, int sl) { return bar0 + 8u * (3 * STAGES + 2 * CS + 4 + 2 * S::XCH + 2 * x + sl); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank() & 1u;
  const bool leader = (rank == 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(rfull_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int c = 0; c < CS; ++c) {
      mbar_init(cfull_bar(c), 2 * 4);  // the four warps of one converter group, in both CTAs
      mbar_init(cempty_bar(c), 1);
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
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.a);
    tma_prefetch_desc(&maps.a_sh);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), S::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int pair = blockIdx.x / 2;
  const int npairs = gridDim.x / 2;
  const int total_tiles = __ldg(&p.grp[p.n_groups_total].z) * p.num_mblocks;
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
        const int n_mma = max(32, (t.rows + 31) / 32 * 32);
        const int half = n_mma >> 1;  // token rows per CTA
        const CUtensorMap* ta = t.shared ? &maps.a_sh : &maps.a;
        const CUtensorMap* tb = t.shared ? maps.b_sh : maps.b;
        const int base = t.shared ? 0 : t.g * p.a_rows_per_group;
        const int b_row = t.b_row + (int)rank * half;
        const uint32_t expect = 2u * (uint32_t)(S::NUM_B * half * S::ROW_BYTES);  // both CTAs' token rows
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t sr = smem_u32(raw + stage * S::RAW_STAGE);
          const int k0 = kb * BLOCK_K;
          // this CTA's weight codes, counted on its own barrier (its converters wait there)
          mbar_arrive_expect_tx(rfull_bar(stage), S::RAW_A);
          if (EPI == EPI_SWIGLU) {
            // gate and up codes of this CTA's 64 features in one 3-D box
            tma_load_3d(sr, ta, rfull_bar(stage), k0, t.mb * BLOCK_M + (int)rank * (BLOCK_M / 2),
                        t.shared ? 0 : 2 * t.g);
          } else {
            tma_load_2d(sr, ta, rfull_bar(stage), k0, base + t.mb * 2 * BLOCK_M + (int)rank * BLOCK_M);
          }
          // both CTAs' token rows, counted on the even CTA's barrier (its MMA thread waits there)
          const uint32_t fbc = mapa_shared(full_bar(stage), 0);
          if (leader) mbar_arrive_expect_tx(full_bar(stage), expect);
#pragma unroll
          for (int bp = 0; bp < S::NUM_B; ++bp) {
            const uint32_t sb = sr + S::RAW_A + bp * S::B_BYTES;
            // the (hi, lo) pair: per 64 features, 64 hi columns then 64 lo columns
            const int kc = HILO ? (k0 >> 6) * 128 + (k0 & 63) + bp * 64 : k0;
            int off = 0;
#pragma unroll
            for (int i = NUM_BOX_H - 1; i >= 0; --i) {
              const int h = B_BOX << i;
              if (h <= S::HALF && (half - off) >= h) {
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
      int stage = 0, cs = 0, buf = 0;
      uint32_t phase = 0, cphase = 0, buf_phase = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < total_tiles; tile += npairs) {
        const Tile t = decode_tile<TN>(tile, p);
        if (t.rows <= 0) continue;
        const int n_mma = max(32, (t.rows + 31) / 32 * 32);
        if (!mbar_wait_cluster(acce_bar(buf), buf_phase ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32_m256(n_mma);
        const uint32_t d = tmem_base + buf * S::ACC_COLS;
        for (int kb = 0; kb < KB; ++kb) {
          // both CTAs' token rows have landed, and both CTAs' converters have widened the slab
          if (!mbar_wait_cluster(full_bar(stage), phase, abort_flag, p.err) ||
              !mbar_wait_cluster(cfull_bar(cs), cphase, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(aslab + cs * S::A_BYTES);
          const uint32_t sb = smem_u32(raw + stage * S::RAW_STAGE + S::RAW_A);
#pragma unroll
          for (int kk = 0; kk < BLOCK_K / 16; ++kk) {
            const uint64_t da = smem_desc_sw(sa, S::ROW_BYTES) + 2 * kk;
#pragma unroll
            for (int bp = 0; bp < S::NUM_B; ++bp) {
              const uint64_t db = smem_desc_sw(sb + bp * S::B_BYTES, S::ROW_BYTES) + 2 * kk;
              tc_mma_pair(d, da, db, idesc, (kb | kk | bp) ? 1u : 0u);
            }
          }
          tc_commit_pair_mc(empty_bar(stage), (uint16_t)0x3u);  // the stage, in both CTAs
          tc_commit_pair_mc(cempty_bar(cs), (uint16_t)0x3u);    // the widened slab, in both CTAs
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          if (++cs == CS) {
            cs = 0;
            cphase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(accf_bar(buf), (uint16_t)0x3u);
        if (++buf == S::NUM_BUF) {
          buf = 0;
          buf_phase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp < S::CVT_WARP0) {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    const int ew = warp - 2;
    const int quad = warp & 3;
    const int half = ew >> 2;
    const int xch = half * 2 + (quad & 1);  // SwiGLU: exchange channel of this gate/up warp pair
    int buf = 0;
    uint32_t buf_phase = 0;
#if MOE_TEST_UNSET_WAIT
    // test build: wait on a phase nothing completes (only the epilogue warps arrive on it, the
    // even CTA's), so the wait runs out and both CTAs take their abort path
    mbar_wait(acce_bar(0), 0, abort_flag, p.err);
#endif
    uint32_t xiter = 0;                      // SwiGLU: chunks exchanged so far on this channel
    bool ok = true;
    const uint32_t acce_leader0 = mapa_shared(acce_bar(0), 0);
    const uint32_t acce_leader1 = mapa_shared(acce_bar(1), 0);
    for (int tile = pair; ok && tile < total_tiles; tile += npairs) {
      const Tile t = decode_tile<TN>(tile, p);
      if (t.rows <= 0) continue;
      if (!mbar_wait_cluster(accf_bar(buf), buf_phase, abort_flag, p.err)) break;
      tc_fence_after();
      const int nchunk = (t.rows + 15) >> 4;
      const uint32_t tq = tmem_base + (uint32_t(quad * 32) << 16) + buf * S::ACC_COLS;
      if (EPI == EPI_SWIGLU) {
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
            const int feat = t.mb * BLOCK_M + (int)rank * (BLOCK_M / 2) + quad * 32 + lane;
            const int nr = min(16, t.rows - c0);
            if (feat < p.out_features && !(p.out_rows > 0 && (bad_index(t.out_row + c0, p.out_rows, p.err) ||
                                                              bad_index(t.out_row + c0 + nr - 1, p.out_rows, p.err)))) {
              const int col = ((feat >> 6) << 7) + (feat & 63);
              __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + (size_t)(t.out_row + c0) * p.out_ld + col;
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
        const int feat = t.mb * 2 * BLOCK_M + (int)rank * BLOCK_M + quad * 32 + lane;
        for (int ci = half; ci < nchunk; ci += 2) {
          const int c0 = ci * 16;
          uint32_t r[16];
          tmem_ld16(tq + c0, r);
          tmem_ld_wait();
          reg_fence16(r);
          const int nr = min(16, t.rows - c0);
          if (feat < p.out_features && !(p.out_rows > 0 && (bad_index(t.out_row + c0, p.out_rows, p.err) ||
                                                            bad_index(t.out_row + c0 + nr - 1, p.out_rows, p.err)))) {
            float* out = static_cast<float*>(p.out) + (size_t)(t.out_row + c0) * p.out_ld + feat;
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
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(buf == 0 ? acce_leader0 : acce_leader1);
      if (++buf == S::NUM_BUF) {
        buf = 0;
        buf_phase ^= 1u;
      }
    }
  } else {
    // ------------------------------------------------------------------ code -> bf16 converters
    // Thread r widens weight row r of every stage: its 64 codes (four 16-byte chunks; chunk c at
    // c ^ ((r >> 1) & 3), the 64-byte swizzle TMA wrote) times 2^e of the row's 128 x 128 tile, into
    // row r of the stage's slab (eight 16-byte chunks; chunk c at c ^ (r & 7), the 128-byte swizzle
    // the MMA reads).  The thread keeps the exponents of the current and the next 128-wide K tile.
    const int r = ((warp - S::CVT_WARP0) & 3) * 32 + lane;  // the group's four warps cover 128 rows
    const int group = (warp - S::CVT_WARP0) >> 2;  // widens the stages n with n % CVT_GROUPS == group
    const int nk = p.exp_nk;
    int stage = 0, cs = 0;
    uint32_t phase = 0, cphase = 0;
    uint32_t n = 0;  // stage counter over all tiles of this CTA
    bool ok = true;
    for (int tile = pair; ok && tile < total_tiles; tile += npairs) {
      const Tile t = decode_tile<TN>(tile, p);
      if (t.rows <= 0) continue;
      const int8_t* ex = t.shared ? p.a_sh_exp : p.a_exp + (size_t)t.g * p.exp_nr * nk;
      int mrow;  // this row's row in its weight matrix
      if (EPI == EPI_SWIGLU) {
        const int f0 = t.mb * BLOCK_M + (int)rank * (BLOCK_M / 2);  // first feature of this CTA
        mrow = r < BLOCK_M / 2 ? f0 + r : p.a_up_offset + f0 + (r - BLOCK_M / 2);
      } else {
        mrow = t.mb * 2 * BLOCK_M + (int)rank * BLOCK_M + r;
      }
      const int trow = min(mrow >> 7, p.exp_nr - 1);  // rows past the matrix are zero codes
      int e_cur = __ldg(ex + trow * nk);
      int e_nxt = nk > 1 ? __ldg(ex + trow * nk + 1) : 0;
      for (int kb = 0; kb < KB; ++kb, ++n) {
        if (kb > 0 && ((kb * BLOCK_K) & 127) == 0) {  // a new 128-wide K tile: rotate, fetch the next
          const int kn = ((kb * BLOCK_K) >> 7) + 1;
          e_cur = e_nxt;
          e_nxt = kn < nk ? __ldg(ex + trow * nk + kn) : 0;
        }
        if ((int)(n % S::CVT_GROUPS) == group) {
          if (!mbar_wait(rfull_bar(stage), phase, abort_flag, p.err) ||
              !mbar_wait(cempty_bar(cs), cphase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t row = smem_u32(raw + stage * S::RAW_STAGE + r * BLOCK_K);
          const uint32_t dst = smem_u32(aslab + cs * S::A_BYTES + r * S::ROW_BYTES);
          const int e = e_cur;
          const uint32_t bias2 = (uint32_t)(120 + e) * 0x00800080u;
          const float scale = __int_as_float((e + 127) << 23);
          const bool tiny = e < -120;
#pragma unroll
          for (int c = 0; c < 4; ++c) {  // K codes [16 c, 16 c + 16) -> widened chunks 2c, 2c + 1
            const uint4 q = ld_shared_v4(row + ((c ^ ((r >> 1) & 3)) << 4));
            uint2 v0, v1, v2, v3;
            // normal codes and an ordinary scale (the common case): integer path; otherwise (a zero
            // or subnormal code, or a scale below 2^-120) the conversion instruction
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
            st_shared_v4(dst + (((2 * c) ^ (r & 7)) << 4), v0.x, v0.y, v1.x, v1.y);
            st_shared_v4(dst + (((2 * c + 1) ^ (r & 7)) << 4), v2.x, v2.y, v3.x, v3.y);
          }
          // the widened row is read by the tensor cores (async proxy) once the MMA thread of the
          // even CTA has seen the group's four converter warps of both CTAs arrive
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(cfull_bar(cs), 0));
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        if (++cs == CS) {
          cs = 0;
          cphase ^= 1u;
        }
      }
    }
  }

  tc_fence_before();
  sync_and_quiesce(abort_flag);
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, S::TMEM_COLS);
  }
}

// ----------------------------------------------------------------------------- host side

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

template <int EPI, int MBLK, int TN>
static cudaError_t launch_fp4mma_variant(const GemmLaunch& L, GemmParams base, cudaStream_t s) {
  using Sh = F4Shape<EPI, MBLK, TN>;
  static_assert(Sh::SMEM_BYTES <= SMEM_LIMIT, "dynamic shared memory per block");
  if (base.sched_tn % TN != 0 || L.K % Sh::BLOCK_K != 0 || base.ksplit != 1) return cudaErrorInvalidValue;
  if (L.a_sub == nullptr || L.b_exp == nullptr) return cudaErrorInvalidValue;
  if (L.a_sh_ptr != nullptr && L.a_sh_sub == nullptr) return cudaErrorInvalidValue;
  if (EPI == EPI_SWIGLU && L.a_up_offset % 128 != 0) return cudaErrorInvalidValue;  // slabs on 128-row boundaries
  if (reinterpret_cast<uintptr_t>(L.a_ptr) % 32 != 0 || reinterpret_cast<uintptr_t>(L.a_sh_ptr) % 32 != 0)
    return cudaErrorInvalidValue;  // the 4-bit tensor maps want 32-byte aligned codes
  GemmMaps m;
  memset(&m, 0, sizeof(m));
  if (EPI == EPI_SWIGLU) {
    const int64_t f = L.a_up_offset;
    if (!make_tmap_e2m1_gateup(&m.a, L.a_ptr, L.a_rows / (2 * f), f, L.K)) return cudaErrorInvalidValue;
    if (L.a_sh_ptr != nullptr && !make_tmap_e2m1_gateup(&m.a_sh, L.a_sh_ptr, 1, f, L.K)) return cudaErrorInvalidValue;
  } else {
    if (!make_tmap_e2m1(&m.a, L.a_ptr, L.a_rows, L.K, BLOCK_M * MBLK)) return cudaErrorInvalidValue;
    if (L.a_sh_ptr != nullptr && !make_tmap_e2m1(&m.a_sh, L.a_sh_ptr, L.a_sh_rows, L.K, BLOCK_M * MBLK))
      return cudaErrorInvalidValue;
  }
  if (L.a_sh_ptr == nullptr) m.a_sh = m.a;
  if (!make_tmap_pieces(&m.b[0], L.b_ptr, L.b_rows, Sh::PIECES, L.K, TN)) return cudaErrorInvalidValue;
  Fp4Params p;
  static_cast<GemmParams&>(p) = base;
  p.b_exp = L.b_exp;
  p.a_sub = L.a_sub;
  p.a_sh_sub = L.a_sh_sub != nullptr ? L.a_sh_sub : L.a_sub;
  auto kern = fp4mma_gemm_kernel<EPI, MBLK, TN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  int grid = L.num_sms;
  const int tiles = L.max_tiles * (base.sched_tn / TN);
  if (tiles < grid) grid = tiles;
  if (grid < 1) grid = 1;
  kern<<<grid, Sh::THREADS, Sh::SMEM_BYTES, s>>>(m, p);
  return cudaGetLastError();
}


template <int EPI, bool HILO>
static cudaError_t launch_fp8w_pair_variant(const GemmLaunch& L, GemmParams p, cudaStream_t s) {
  using Sh = Fp8PairShape<EPI, HILO>;
  static_assert(Sh::SMEM_BYTES <= SMEM_LIMIT, "dynamic shared memory per block");
  if (p.sched_tn != Sh::TN || L.K % Sh::BLOCK_K != 0 || p.ksplit != 1 || p.grp == nullptr || L.a_exp == nullptr)
    return cudaErrorInvalidValue;
  if (L.a_sh_ptr != nullptr && L.a_sh_exp == nullptr) return cudaErrorInvalidValue;
  GemmMaps m;
  memset(&m, 0, sizeof(m));
  if (EPI == EPI_SWIGLU) {
    const int64_t f = L.a_up_offset;
    if (!make_tmap_u8_gateup(&m.a, L.a_ptr, L.a_rows / (2 * f), f, L.K, 64, Sh::A_BOX)) return cudaErrorInvalidValue;
    if (L.a_sh_ptr != nullptr && !make_tmap_u8_gateup(&m.a_sh, L.a_sh_ptr, 1, f, L.K, 64, Sh::A_BOX))
      return cudaErrorInvalidValue;
  } else {
    if (!make_tmap_u8(&m.a, L.a_ptr, L.a_rows, L.K, Sh::A_BOX)) return cudaErrorInvalidValue;
    if (L.a_sh_ptr != nullptr && !make_tmap_u8(&m.a_sh, L.a_sh_ptr, L.a_sh_rows, L.K, Sh::A_BOX))
      return cudaErrorInvalidValue;
  }
  if (L.a_sh_ptr == nullptr) m.a_sh = m.a;
  const int kb_cols = HILO ? 2 * L.K : L.K;
  for (int i = 0; i < NUM_BOX_H; ++i) {
    const int h = B_BOX << i;
    if (h > Sh::HALF) break;
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
  auto kern = fp8w_pair_gemm_kernel<EPI, HILO>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.blockDim = dim3(Sh::THREADS);
  cfg.dynamicSmemBytes = Sh::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // as many clusters as can be resident at once (persistent kernel), at most one per tile
  static int max_clusters = 0;
  if (max_clusters == 0) {
    cfg.gridDim = dim3(2 * (L.num_sms / 2));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = L.num_sms / 2;
    }
    max_clusters = n;
  }
  int clusters = max_clusters;
  if (L.max_tiles < clusters) clusters = L.max_tiles;
  if (clusters < 1) clusters = 1;
  cfg.gridDim = dim3(2 * clusters);
  e = cudaLaunchKernelEx(&cfg, kern, m, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_fp8_gemm(const GemmLaunch& L, GemmParams p, int kernel_tn, cudaStream_t s) {
  if ((L.q8 == 2 || L.q8 == 3) && L.pair) return launch_bs_pair_gemm(L, p, s);  // prefill, block-scaled
  if (L.q8 == 1 && L.pair) {
    // prefill: codes widened to bf16 in shared memory, CTA-pair bf16 MMA, 256-row token tiles
    if (L.epi == EPI_SWIGLU && kernel_tn == 256) return launch_fp8w_pair_variant<EPI_SWIGLU, false>(L, p, s);
    if (L.epi != EPI_SWIGLU && L.hilo && kernel_tn == 256 && L.mblk == 2)
      return launch_fp8w_pair_variant<EPI_F32, true>(L, p, s);
    return cudaErrorInvalidValue;
  }
  if (L.q8 == 3) {
    // native MXFP4 codes on the block-scaled MMA, E4M3-piece activations, 16-, 32- or 64-row
    // token tiles (the down projection's 32- and 64-row tiles on one 128-feature slab)
    if (L.epi == EPI_SWIGLU && kernel_tn == 16) return launch_fp4mma_variant<EPI_SWIGLU, 1, 16>(L, p, s);
    if (L.epi == EPI_SWIGLU && kernel_tn == 32) return launch_fp4mma_variant<EPI_SWIGLU, 1, 32>(L, p, s);
    if (L.epi == EPI_SWIGLU && kernel_tn == 64) return launch_fp4mma_variant<EPI_SWIGLU, 1, 64>(L, p, s);
    if (L.epi != EPI_SWIGLU && kernel_tn == 16 && L.mblk == 2) return launch_fp4mma_variant<EPI_F32, 2, 16>(L, p, s);
    if (L.epi != EPI_SWIGLU && kernel_tn == 32 && L.mblk == 1) return launch_fp4mma_variant<EPI_F32, 1, 32>(L, p, s);
    if (L.epi != EPI_SWIGLU && kernel_tn == 64 && L.mblk == 1) return launch_fp4mma_variant<EPI_F32, 1, 64>(L, p, s);
    return cudaErrorInvalidValue;
  }
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
  if (L.q8 == 1) {
    // codes widened to bf16: single-CTA kernels with 64-row token tiles
    if (L.epi == EPI_SWIGLU && kernel_tn == 64) return launch_fp8_variant<EPI_SWIGLU, 64, 1, false>(L, p, s);
    if (L.epi != EPI_SWIGLU && L.hilo && kernel_tn == 64 && L.mblk == 2)
      return launch_fp8_variant<EPI_F32, 64, 2, true>(L, p, s);
    return cudaErrorInvalidValue;
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
