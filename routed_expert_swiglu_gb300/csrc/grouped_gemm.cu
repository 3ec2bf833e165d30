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
#include "gemm_common.cuh"

namespace moe {

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
#if MOE_TEST_UNSET_WAIT
    // test build: wait on a phase nothing completes (only these warps arrive on it), so the
    // wait runs out and the kernel takes its abort path
    mbar_wait(acce_bar(0), 0, abort_flag, p.err);
#endif
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
  sync_and_quiesce(abort_flag);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, S::TMEM_COLS);
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
template <int EPI, int TN, bool HILO, int BK, int TMEM_ALLOC>
struct PairShape {
  static constexpr int BLOCK_K = BK;
  static constexpr int ROW_BYTES = BK * 2;
  static constexpr int HALF = TN / 2;
  static constexpr int A_BYTES = BLOCK_M * BK * 2;                  // one 128-row weight slab
  static constexpr int NUM_B = HILO ? 2 : 1;
  static constexpr int B_BYTES = HALF * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + NUM_B * B_BYTES;
  static constexpr int XCH = (EPI == EPI_SWIGLU) ? 4 : 0;           // gate/up warp pairs
  static constexpr int XBUF_BYTES = XCH * 2 * 16 * 32 * 4;          // 2 slots of 16 x 32 fp32
  static constexpr int ACC_COLS = TN;                               // one accumulator of TN columns
  static constexpr int NUM_BUF = (TMEM_ALLOC / ACC_COLS) >= 2 ? 2 : 1;
  static constexpr int STAGES_FIT = (SMEM_LIMIT - 1024 - 512 - XBUF_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 16 ? 16 : STAGES_FIT;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + XBUF_BYTES + 1024 + 512;
  static constexpr int FEATS = (EPI == EPI_SWIGLU) ? BLOCK_M : 2 * BLOCK_M;
  static constexpr int A_BOX = (EPI == EPI_SWIGLU) ? BLOCK_M / 2 : BLOCK_M;
  static constexpr int THREADS = (2 + NUM_EPI_WARPS) * 32;
  // barriers (full, empty per stage; acc full/empty x2; exchange full/empty x2 per channel),
  // then the TMEM address slot and the abort flag, in the last 512 bytes
  static_assert((2 * STAGES + 4 + 4 * XCH) * 8 + 8 <= 512, "barrier area");
  static_assert(TN % 32 == 0 && TN <= 256, "pair token tile");
  static_assert(TMEM_ALLOC >= ACC_COLS && TMEM_ALLOC <= 512, "TMEM allocation");
  static_assert(STAGES >= 2, "pipeline needs two stages");
  static_assert(BK == 64 || BK == 32, "stage K");
};

template <int EPI, int TN, bool HILO, int BK, int TMEM_ALLOC>
__global__ void __launch_bounds__(PairShape<EPI, TN, HILO, BK, TMEM_ALLOC>::THREADS, 1)
    pair_gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmParams p) {
  using S = PairShape<EPI, TN, HILO, BK, TMEM_ALLOC>;
  constexpr int STAGES = S::STAGES;
  constexpr int BLOCK_K = S::BLOCK_K;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* xbuf = reinterpret_cast<float*>(smem + STAGES * S::STAGE_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * S::STAGE_BYTES + S::XBUF_BYTES);
  // bars: full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], xfull[XCH][2], xempty[XCH][2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 4 + 4 * S::XCH);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto accf_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto acce_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  auto xfull_bar = [&](int x, int sl) { return bar0 + 8u * (2 * STAGES + 4 + 2 * x + sl); };
  auto xempty_bar = [&](int x, int sl) { return bar0 + 8u * (2 * STAGES + 4 + 2 * S::XCH + 2 * x + sl); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank() & 1u;  // position in the CTA pair
  const bool leader = (rank == 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);   // the even CTA's expect-tx arrival
      mbar_init(empty_bar(s), 1);  // the MMA commit
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
    tmem_alloc_pair(smem_u32(tmem_slot), TMEM_ALLOC);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int pair = blockIdx.x / 2;   // cluster index
  const int npairs = gridDim.x / 2;  // clusters
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
        const int n_mma = max(32, (t.rows + 31) / 32 * 32);
        const int half = n_mma >> 1;         // token rows per CTA
        const CUtensorMap* ta = t.shared ? &maps.a_sh : &maps.a;
        const CUtensorMap* tb = t.shared ? maps.b_sh : maps.b;
        const int base = t.shared ? 0 : t.g * p.a_rows_per_group;
        const int b_row = t.b_row + (int)rank * half;
        const uint32_t expect = 2u * (S::A_BYTES + S::NUM_B * half * BLOCK_K * 2);  // both CTAs, on the even CTA
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_u32(smem + stage * S::STAGE_BYTES);
          const uint32_t fbc = mapa_shared(full_bar(stage), 0);  // the pair's even CTA's full barrier
          if (leader) mbar_arrive_expect_tx(full_bar(stage), expect);
          const int k0 = kb * BLOCK_K;
          if (EPI == EPI_SWIGLU) {
            // this CTA's gate and up slabs (64 features each) in one 3-D box
            tma_load_3d_pair(sa, ta, fbc, k0, t.mb * BLOCK_M + (int)rank * (BLOCK_M / 2), t.shared ? 0 : 2 * t.g);
          } else {
            tma_load_2d_pair(sa, ta, fbc, k0, base + t.mb * 2 * BLOCK_M + (int)rank * BLOCK_M);
          }
#pragma unroll
          for (int bp = 0; bp < S::NUM_B; ++bp) {
            const uint32_t sb = sa + S::A_BYTES + bp * S::B_BYTES;
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
      int stage = 0;
      uint32_t phase = 0;
      int buf = 0;
      uint32_t buf_phase = 0;
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
          if (!mbar_wait_cluster(full_bar(stage), phase, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * S::STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < BLOCK_K / 16; ++kk) {
            const uint64_t da = smem_desc_sw(sa, S::ROW_BYTES) + 2 * kk;
#pragma unroll
            for (int bp = 0; bp < S::NUM_B; ++bp) {
              const uint64_t db = smem_desc_sw(sa + S::A_BYTES + bp * S::B_BYTES, S::ROW_BYTES) + 2 * kk;
              tc_mma_pair(d, da, db, idesc, (kb | kk | bp) ? 1u : 0u);
            }
          }
          tc_commit_pair_mc(empty_bar(stage), (uint16_t)0x3u);  // both CTAs
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
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
  } else {
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
  }

  tc_fence_before();
  sync_and_quiesce(abort_flag);
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

template <int EPI, int TN, bool HILO, int BK, int TMEM_ALLOC>
static cudaError_t launch_pair_variant(const GemmLaunch& L, GemmParams p, cudaStream_t s) {
  using Sh = PairShape<EPI, TN, HILO, BK, TMEM_ALLOC>;
  static_assert(Sh::SMEM_BYTES <= SMEM_LIMIT, "dynamic shared memory per block");
  if (p.sched_tn % TN != 0 || L.K % BK != 0) return cudaErrorInvalidValue;
  GemmMaps m;
  memset(&m, 0, sizeof(m));
  const int kb_cols = HILO ? 2 * L.K : L.K;
  if (!make_a_maps(m, L, EPI == EPI_SWIGLU, Sh::A_BOX, BK)) return cudaErrorInvalidValue;
  for (int i = 0; i < NUM_BOX_H; ++i) {
    const int h = B_BOX << i;
    if (h > Sh::HALF) break;
    if (!make_tmap(&m.b[i], L.b_ptr, L.b_rows, kb_cols, h, BK)) return cudaErrorInvalidValue;
    if (L.b_sh_ptr != nullptr) {
      if (!make_tmap(&m.b_sh[i], L.b_sh_ptr, L.b_sh_rows, kb_cols, h, BK)) return cudaErrorInvalidValue;
    } else {
      m.b_sh[i] = m.b[i];
    }
  }
  auto kern = pair_gemm_kernel<EPI, TN, HILO, BK, TMEM_ALLOC>;
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
  const int tiles = L.max_tiles * (p.sched_tn / TN);
  if (tiles < clusters) clusters = tiles;
  if (clusters < 1) clusters = 1;
  cfg.gridDim = dim3(2 * clusters);
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
  p.out_rows = L.out_rows;
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
  p.a_exp = nullptr;
  p.a_sh_exp = nullptr;
  p.exp_nr = p.exp_nk = 0;
  p.b_exp = nullptr;
  if (L.q8) return launch_fp8_gemm(L, p, kernel_tn, s);
  constexpr int TNP = MOE_TN_PREFILL;
  constexpr int TN2 = MOE_TN_PREFILL;
  if (L.pair) {
    if (L.epi == EPI_SWIGLU && kernel_tn == TNP)
      return launch_pair_variant<EPI_SWIGLU, TNP, false, 64, MOE_PAIR_TMEM>(L, p, s);
    if (L.epi != EPI_SWIGLU && L.hilo && kernel_tn == TN2 && L.mblk == 2)
      return launch_pair_variant<EPI_F32, TN2, true, 64, MOE_PAIR_TMEM>(L, p, s);
    return cudaErrorInvalidValue;
  }
  if (L.epi == EPI_SWIGLU) {
    if (kernel_tn == 64) return launch_variant<EPI_SWIGLU, 64, 1, false, 64>(L, p, s);
    return cudaErrorInvalidValue;
  }
  if (L.hilo) {
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
