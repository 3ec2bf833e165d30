// Block-scaled CTA-pair GEMMs for FP8 (E4M3) and MXFP4 (E2M1) expert weights at prefill
// ("DeepSeek-V4 MoE", section "FP4 QAT 怎么做到反量化无损": FP8 weights with one scale per 128 x
// 128 tile, FP4 weights with one per 1 x 32 sub-block).  The stored codes are the A operand of the
// 2-SM block-scaled MMA (tcgen05.mma.cta_group::2 kind::mxf8f6f4 with block_scale), their scales
// (the tile's 2^E, or each sub-block's 2^s) applied by the tensor cores as UE8M0 A scales; the
// activations are E4M3 pieces (two for the dispatched rows, four for h; row r = 2^e_r *
// sum_p piece_p * 2^(-4p)), one MMA per piece with the piece's weight 2^(-4p) as its B scale, so
// that every piece of every K step accumulates into one fp32 accumulator per tile, and the
// epilogue applies 2^e_r (and the gate weights) once.  The layer is then the bf16 layer on the
// dequantised weights up to the pieces' precision, as on the single-CTA FP8 / MXFP4 kernels.
//
// Tiles: 224 token rows (112 per CTA) by 256 weight rows (128 per CTA); SwiGLU: each CTA holds 64
// gate and the matching 64 up rows (the epilogue pairs them through shared memory, as the bf16
// pair kernel does).  The weight codes and the token rows have rings of their own (the codes come
// from HBM and want more of their stream in flight).  Roles (480 threads per CTA): warp 0 TMA
// producer of the codes, warp 14 of the token rows, warp 1 TMEM owner + MMA issuer (even CTA),
// warps 2..9 epilogue, warps 10..13 A-scale writers (lane quadrant w % 4 of this CTA's Tensor
// Memory: one word of four UE8M0 scales per K step, at column c0 + quadrant of a slot of their own
// ring, the layout the MMA reads for M = 128 rows per CTA; reported to the even CTA once per four
// K steps).  Scale addresses lie on 4-column boundaries.
#include "gemm_common.cuh"

namespace moe {

// D[tmem of both CTAs] (+)= (A . 2^SFA) * (B . 2^SFB)^T on 8-bit / 4-bit operands, M = 256, K = 32,
// scales read from each CTA's Tensor Memory at sfa / sfb; issued by one thread of the even CTA.
__device__ __forceinline__ void tc_mma_pair_mx(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of the pair MMA: A format afmt (0 = E4M3, 5 = E2M1), B E4M3, fp32
// accumulator, K-major, UE8M0 scales, M = 256, N = n, B scale byte 0, A scale byte `ida`.
__device__ __forceinline__ uint32_t idesc_mx_m256(uint32_t afmt, uint32_t n, uint32_t ida) {
  return (afmt << 7) | ((n >> 3) << 17) | (1u << 23) | ((256u >> 4) << 24) | (ida << 29);
}

struct BsParams : GemmParams {
  const int8_t* a_sub;     // MXFP4: sub-block exponents [mats, rows, K/32] of the routed weights
  const int8_t* a_sh_sub;  // and of the shared expert's
};

// K steps whose A scales a scale writer loads at once (see the writers' loop).
constexpr int SF_CHUNK = 16;

template <int EPI, bool F4>
struct BsPairShape {
  static constexpr int TN = BS_PAIR_TN;                 // token rows per tile, both CTAs (224)
  static constexpr int HALF = TN / 2;                   // B rows per CTA at most
  static constexpr int BLOCK_K = 128;                   // K per stage: one TMA box, four MMAs
  static constexpr int A_BYTES = BLOCK_M * BLOCK_K;     // this CTA's 128 weight rows in shared memory
  static constexpr int A_TX = F4 ? A_BYTES / 2 : A_BYTES;  // bytes their load moves (4-bit codes: half)
  static constexpr int PIECES = (EPI == EPI_SWIGLU) ? 2 : 4;
  static constexpr int B_PIECE = HALF * BLOCK_K;        // one piece of this CTA's token rows
  static constexpr int B_STAGE = PIECES * B_PIECE;
  static constexpr int XCH = (EPI == EPI_SWIGLU) ? 4 : 0;
  static constexpr int XBUF_BYTES = XCH * 2 * 16 * 32 * 4;
  // Two rings: the weight codes (from HBM, long latency) in ASTAGES slots, the token rows (from
  // L2) in BSTAGES slots, each with its own producer, so that more of the weight stream is in
  // flight than a joint stage of both would allow.
  static constexpr int BSTAGES = 3;
  static constexpr int AFIT = (SMEM_LIMIT - 1024 - 1024 - XBUF_BYTES - BSTAGES * B_STAGE) / A_BYTES;
  static constexpr int ASTAGES = AFIT > 8 ? 8 : AFIT;
  static constexpr int BAR_BYTES = 1024;                // barriers, the TMEM slot and the abort flag
  static constexpr int SMEM_BYTES = ASTAGES * A_BYTES + BSTAGES * B_STAGE + XBUF_BYTES + 1024 + BAR_BYTES;
  static constexpr int ACC_COLS = TN;
  static constexpr int NUM_BUF = 2;
  static constexpr int SFB_COLS = 8;                    // B-scale region of one piece
  static constexpr int SFB_COL0 = NUM_BUF * ACC_COLS;
  static constexpr int SFA_COL0 = SFB_COL0 + PIECES * SFB_COLS;
  static constexpr int TMEM_COLS = 512;
  // A scales have a ring of their own in the Tensor Memory left over (four columns a slot, one per
  // lane quadrant), deeper than the code ring, so that their writers run ahead of the codes.
  // The scale writers report in groups of SF_GROUP K steps: each report is an arrive with release
  // semantics on the even CTA's barrier, which costs about a microsecond, longer than a K step of
  // MMAs; one report per group keeps the writers ahead of the tensor cores.
  static constexpr int SF_GROUP = 4;
  static constexpr int SF_FIT = (TMEM_COLS - SFA_COL0) / 4 / SF_GROUP * SF_GROUP;
  static constexpr int SFSLOTS = SF_FIT > 16 ? 16 : SF_FIT;
  static constexpr int SF_GROUPS = SFSLOTS / SF_GROUP;
  static constexpr int SFA_COLS = SFSLOTS * 4;
  static constexpr int SF_WARP0 = 2 + NUM_EPI_WARPS;
  static constexpr int BPROD_WARP = SF_WARP0 + 4;       // the token-row producer
  static constexpr int THREADS = (BPROD_WARP + 1) * 32;
  static constexpr int A_BOX = (EPI == EPI_SWIGLU) ? BLOCK_M / 2 : BLOCK_M;  // rows per box
  // barriers: full, empty per A slot, per B slot and per group of scale slots; acc full/empty
  // x2; SwiGLU exchange
  static constexpr int NUM_BARS = 2 * ASTAGES + 2 * BSTAGES + 2 * SF_GROUPS + 4 + 4 * XCH;
  static_assert(NUM_BARS * 8 + 8 <= BAR_BYTES, "barrier area");
  static_assert(ASTAGES >= 2 && BSTAGES >= 2 && SF_GROUPS >= 2, "pipelines need two slots");
  static_assert(B_PIECE % 1024 == 0 && A_BYTES % 1024 == 0, "swizzled tiles on 1024 B");
  static_assert(SFB_COL0 % 4 == 0 && SFA_COL0 % 4 == 0, "scale addresses on 4-column boundaries");
  static_assert(SFA_COL0 + SFA_COLS <= TMEM_COLS, "TMEM: accumulators + scales");
  static_assert(TN % 32 == 0 && HALF <= 128, "token tile");
};

template <int EPI, bool F4>
__global__ void __launch_bounds__(BsPairShape<EPI, F4>::THREADS, 1)
    bs_pair_gemm_kernel(const __grid_constant__ GemmMaps maps, const BsParams p) {
  using S = BsPairShape<EPI, F4>;
  constexpr int TN = S::TN;
  constexpr int AST = S::ASTAGES;
  constexpr int BST = S::BSTAGES;
  constexpr int BLOCK_K = S::BLOCK_K;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* aring = smem;                                  // AST slots of this CTA's weight codes
  uint8_t* bring = smem + AST * S::A_BYTES;               // BST slots of this CTA's token-row pieces
  float* xbuf = reinterpret_cast<float*>(bring + BST * S::B_STAGE);
  uint64_t* bars = reinterpret_cast<uint64_t*>(bring + BST * S::B_STAGE + S::XBUF_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + S::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  constexpr int NSF = S::SFSLOTS;
  constexpr int SG = S::SF_GROUP;
  constexpr int NSG = S::SF_GROUPS;
  auto afull_bar = [&](int s) { return bar0 + 8u * s; };                // both CTAs' codes (even CTA)
  auto aempty_bar = [&](int s) { return bar0 + 8u * (AST + s); };       // A slot consumed
  auto bfull_bar = [&](int s) { return bar0 + 8u * (2 * AST + s); };   // both CTAs' rows (even CTA)
  auto bempty_bar = [&](int s) { return bar0 + 8u * (2 * AST + BST + s); };  // B slot consumed
  auto sfull_bar = [&](int g) { return bar0 + 8u * (2 * AST + 2 * BST + g); };  // a group's scales (even CTA)
  auto sempty_bar = [&](int g) { return bar0 + 8u * (2 * AST + 2 * BST + NSG + g); };  // group consumed
  const uint32_t bar1 = bar0 + 8u * (2 * AST + 2 * BST + 2 * NSG);
  auto accf_bar = [&](int a) { return bar1 + 8u * a; };
  auto acce_bar = [&](int a) { return bar1 + 8u * (2 + a); };
  auto xfull_bar = [&](int x, int sl) { return bar1 + 8u * (4 + 2 * x + sl); };
  auto xempty_bar = [&](int x, int sl) { return bar1 + 8u * (4 + 2 * S::XCH + 2 * x + sl); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank() & 1u;
  const bool leader = (rank == 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < AST; ++s) {
      mbar_init(afull_bar(s), 1);
      mbar_init(aempty_bar(s), 1);
    }
    for (int g = 0; g < NSG; ++g) {
      mbar_init(sfull_bar(g), 2 * 4);  // the four scale warps of both CTAs
      mbar_init(sempty_bar(g), 1);
    }
    for (int s = 0; s < BST; ++s) {
      mbar_init(bfull_bar(s), 1);
      mbar_init(bempty_bar(s), 1);
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
  if (warp >= S::SF_WARP0 && warp < S::BPROD_WARP) {
    // B scales of this CTA: region p holds 2^(-4p) (UE8M0 127 - 4p) in every lane, byte and column
    const uint32_t tq = tmem_base + (uint32_t((warp & 3) * 32) << 16) + S::SFB_COL0;
#pragma unroll
    for (int pc = 0; pc < S::PIECES; ++pc)
#pragma unroll
      for (int c = 0; c < S::SFB_COLS; ++c) tmem_st1(tq + pc * S::SFB_COLS + c, (127u - 4u * pc) * 0x01010101u);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' B scales are in place before the first MMA
  tc_fence_after();

  const int pair = blockIdx.x / 2;
  const int npairs = gridDim.x / 2;
  const int total_tiles = __ldg(&p.grp[p.n_groups_total].z) * p.num_mblocks;
  const int KB = p.K / BLOCK_K;

  if (warp == 0 || warp == S::BPROD_WARP) {
    // ------------------------------------------------------------------ TMA producers (both CTAs)
    // warp 0: this CTA's weight codes into the A ring; the last warp: this CTA's token rows (each
    // piece) into the B ring.  Both count on the even CTA's barriers, whose MMA thread waits there.
    if (lane == 0) {
      const bool is_a = (warp == 0);
      const int NS = is_a ? AST : BST;
      int slot = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < total_tiles; tile += npairs) {
        const Tile t = decode_tile<TN>(tile, p);
        if (t.rows <= 0) continue;
        const int n_mma = max(32, (t.rows + 31) / 32 * 32);
        const int half = n_mma >> 1;  // token rows per CTA
        const CUtensorMap* ta = t.shared ? &maps.a_sh : &maps.a;
        const int base = t.shared ? 0 : t.g * p.a_rows_per_group;
        const int b_row = t.b_row + (int)rank * half;
        const uint32_t expect = is_a ? 2u * (uint32_t)S::A_TX : 2u * (uint32_t)(S::PIECES * half * BLOCK_K);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(is_a ? aempty_bar(slot) : bempty_bar(slot), phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t fb = is_a ? afull_bar(slot) : bfull_bar(slot);
          const uint32_t fbc = mapa_shared(fb, 0);
          if (leader) mbar_arrive_expect_tx(fb, expect);
          const int k0 = kb * BLOCK_K;
          if (is_a) {
            const uint32_t sa = smem_u32(aring + slot * S::A_BYTES);
            if (EPI == EPI_SWIGLU) {
              // gate and up codes of this CTA's 64 features in one 3-D box
              tma_load_3d_pair(sa, ta, fbc, k0, t.mb * BLOCK_M + (int)rank * (BLOCK_M / 2), t.shared ? 0 : 2 * t.g);
            } else {
              tma_load_2d_pair(sa, ta, fbc, k0, base + t.mb * 2 * BLOCK_M + (int)rank * BLOCK_M);
            }
          } else {
#pragma unroll
            for (int pc = 0; pc < S::PIECES; ++pc) {
              const uint32_t sb = smem_u32(bring + slot * S::B_STAGE + pc * S::B_PIECE);
              int off = 0;
#pragma unroll
              for (int i = NUM_BOX_H - 1; i >= 0; --i) {
                const int h = B_BOX << i;
                if (h <= S::HALF && (half - off) >= h) {
                  tma_load_3d_pair(sb + off * BLOCK_K, &maps.b[i], fbc, k0, pc, b_row + off);
                  off += h;
                }
              }
            }
          }
          if (++slot == NS) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (even CTA)
    if (leader && lane == 0) {
      int as = 0, bs = 0, buf = 0;
      uint32_t aphase = 0, bphase = 0, buf_phase = 0;
      uint32_t n = 0;  // K steps so far (scale slot n % NSF, group n / SG % NSG)
      bool ok = true;
      for (int tile = pair; ok && tile < total_tiles; tile += npairs) {
        const Tile t = decode_tile<TN>(tile, p);
        if (t.rows <= 0) continue;
        const int n_mma = max(32, (t.rows + 31) / 32 * 32);
        if (!mbar_wait_cluster(acce_bar(buf), buf_phase ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * S::ACC_COLS;
        for (int kb = 0; kb < KB; ++kb) {
          // both CTAs' codes, A scales and token rows of this K step are in place
          const bool w1 = mbar_wait_cluster(afull_bar(as), aphase, abort_flag, p.err);
          const int ss = (int)(n % NSF), sg = (int)((n / SG) % NSG);
          const bool w2 = w1 && ((n % SG) != 0 || mbar_wait_cluster(sfull_bar(sg), (n / NSF) & 1u, abort_flag, p.err));
          const bool w3 = w2 && mbar_wait_cluster(bfull_bar(bs), bphase, abort_flag, p.err);
          if (!w3) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(aring + as * S::A_BYTES);
          const uint32_t sb = smem_u32(bring + bs * S::B_STAGE);
          const uint32_t sfa = tmem_base + S::SFA_COL0 + ss * 4;
#pragma unroll
          for (int kk = 0; kk < BLOCK_K / 32; ++kk) {
            const uint64_t da = smem_desc_sw(sa, 128) + 2 * kk;
            const uint32_t idesc = idesc_mx_m256(F4 ? 5u : 0u, n_mma, kk);
#pragma unroll
            for (int pc = 0; pc < S::PIECES; ++pc) {
              const uint64_t db = smem_desc_sw(sb + pc * S::B_PIECE, 128) + 2 * kk;
              tc_mma_pair_mx(d, da, db, idesc, sfa, tmem_base + S::SFB_COL0 + pc * S::SFB_COLS,
                             (kb | kk | pc) ? 1u : 0u);
            }
          }
          tc_commit_pair_mc(aempty_bar(as), (uint16_t)0x3u);  // the slots, in both CTAs
          tc_commit_pair_mc(bempty_bar(bs), (uint16_t)0x3u);
          if (n % SG == SG - 1) tc_commit_pair_mc(sempty_bar(sg), (uint16_t)0x3u);
          ++n;
          if (++as == AST) {
            as = 0;
            aphase ^= 1u;
          }
          if (++bs == BST) {
            bs = 0;
            bphase ^= 1u;
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
  } else if (warp < S::SF_WARP0) {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    // Column j of a chunk is token row out_row + c0 + j: its value is scaled by the row's 2^e
    // (and, in the down projection, the row's gate weight).
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
      for (int ci = half; ci < nchunk; ci += 2, ++xiter) {
        const int c0 = ci * 16;
        const int nr = min(16, t.rows - c0);
        uint32_t r[16];
        tmem_ld16(tq + c0, r);
        tmem_ld_wait();
        reg_fence16(r);
        const bool skip = p.out_rows > 0 && (bad_index(t.out_row + c0, p.out_rows, p.err) ||
                                             bad_index(t.out_row + c0 + nr - 1, p.out_rows, p.err));
        if (EPI == EPI_SWIGLU) {
          const int sl = xiter & 1;
          const uint32_t par = (xiter >> 1) & 1u;
          float* xb = xbuf + xch * (2 * 16 * 32);
          if (quad >= 2) {
            // up lanes: hand the 16 up values of this chunk to the gate warp of the channel
            if (!mbar_wait(xempty_bar(xch, sl), par ^ 1u, abort_flag, p.err)) {
              ok = false;
              break;
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) xb[(sl * 16 + j) * 32 + lane] = __uint_as_float(r[j]);
            mbar_arrive(xfull_bar(xch, sl));
          } else {
            const float cs_l = lane < nr ? __int_as_float((127 + __ldg(p.b_exp + t.b_row + c0 + lane)) << 23) : 0.0f;
            if (!mbar_wait(xfull_bar(xch, sl), par, abort_flag, p.err)) {
              ok = false;
              break;
            }
            float u[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) u[j] = xb[(sl * 16 + j) * 32 + lane];
            mbar_arrive(xempty_bar(xch, sl));
            const int feat = t.mb * BLOCK_M + (int)rank * (BLOCK_M / 2) + quad * 32 + lane;
            float* out = static_cast<float*>(p.out) + (size_t)(t.out_row + c0) * p.out_ld + feat;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float cs = __shfl_sync(0xffffffffu, cs_l, j);
              if (j < nr && feat < p.out_features && !skip) {
                const float g = __uint_as_float(r[j]) * cs, uj = u[j] * cs;
                out[(size_t)j * p.out_ld] = __fdividef(g, 1.0f + __expf(-g)) * uj;
              }
            }
          }
        } else {
          float cs_l = lane < nr ? __int_as_float((127 + __ldg(p.b_exp + t.b_row + c0 + lane)) << 23) : 0.0f;
          if (p.row_scale != nullptr && !t.shared && lane < nr) cs_l *= __ldg(p.row_scale + t.out_row + c0 + lane);
          const int feat = t.mb * 2 * BLOCK_M + (int)rank * BLOCK_M + quad * 32 + lane;
          float* out = static_cast<float*>(p.out) + (size_t)(t.out_row + c0) * p.out_ld + feat;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float cs = __shfl_sync(0xffffffffu, cs_l, j);
            if (j < nr && feat < p.out_features && !skip) out[(size_t)j * p.out_ld] = __uint_as_float(r[j]) * cs;
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
  } else if (warp < S::BPROD_WARP) {
    // ------------------------------------------------------------------ A-scale writers (both CTAs)
    // Warp w owns lane quadrant q = w % 4 of this CTA's Tensor Memory, i.e. the CTA's weight rows
    // r = 32 q + lane (SwiGLU: rows 0..63 gate features, 64..127 the matching up features).  For K
    // step n the thread writes one word at column q of scale slot n % NSF: four UE8M0 bytes, one
    // per 32-wide K block -- FP8: the row's 128 x 128 tile exponent E + 127 in all four; MXFP4: the
    // row's four sub-block exponents s + 127 (s below -127 taken as -127) -- once the slots' group
    // has been consumed, and reports each group of SG steps to the even CTA's MMA thread.
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int kb32 = p.K / 32;
    uint32_t n = 0;  // K steps so far
    bool ok = true;
    const uint32_t ts = tmem_base + (uint32_t(quad * 32) << 16) + S::SFA_COL0 + quad;
    auto report = [&](uint32_t step) {  // the group of `step` is written
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(sfull_bar((int)((step / SG) % NSG)), 0));
    };
    for (int tile = pair; ok && tile < total_tiles; tile += npairs) {
      const Tile t = decode_tile<TN>(tile, p);
      if (t.rows <= 0) continue;
      int mrow;  // this lane's row in its weight matrix
      if (EPI == EPI_SWIGLU) {
        const int f0 = t.mb * BLOCK_M + (int)rank * (BLOCK_M / 2);
        mrow = r < BLOCK_M / 2 ? f0 + r : p.a_up_offset + f0 + (r - BLOCK_M / 2);
      } else {
        mrow = t.mb * 2 * BLOCK_M + (int)rank * BLOCK_M + r;
      }
      mrow = min(mrow, p.a_rows_per_group - 1);  // rows past the matrix: any valid row (zero codes)
      const int8_t* ex = nullptr;
      const uint32_t* sub = nullptr;
      if (F4) {
        const int8_t* s0 = t.shared ? p.a_sh_sub : p.a_sub + (size_t)t.g * p.a_rows_per_group * kb32;
        sub = reinterpret_cast<const uint32_t*>(s0 + (size_t)mrow * kb32);
      } else {
        ex = (t.shared ? p.a_sh_exp : p.a_exp + (size_t)t.g * p.exp_nr * p.exp_nk) + (size_t)(mrow >> 7) * p.exp_nk;
      }
      auto word = [&](int kb) -> uint32_t {
        if (F4) return __vadd4(__vmaxs4(__ldg(sub + kb), 0x81818181u), 0x7F7F7F7Fu);
        const int e = min(max((int)__ldg(ex + kb) + 127, 0), 254);
        return (uint32_t)e * 0x01010101u;
      };
      // The scales of SF_CHUNK K steps are loaded together and used before the first of those
      // steps reports: a report (release semantics) then never waits for a load in flight.
      for (int kb0 = 0; ok && kb0 < KB; kb0 += SF_CHUNK) {
        uint32_t w[SF_CHUNK];
#pragma unroll
        for (int j = 0; j < SF_CHUNK; ++j) w[j] = (kb0 + j < KB) ? word(kb0 + j) : 0u;
#pragma unroll
        for (int j = 0; j < SF_CHUNK; ++j) {
          if (kb0 + j >= KB) break;
          if (n % SG == 0 &&
              !mbar_wait(sempty_bar((int)((n / SG) % NSG)), ((n / NSF) & 1u) ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          tmem_st1(ts + (n % NSF) * 4, w[j]);
          if (n % SG == SG - 1) report(n);
          ++n;
        }
      }
    }
    if (ok && n % SG != 0) report(n - 1);  // the last, partial group
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

template <int EPI, bool F4>
static cudaError_t launch_bs_pair_variant(const GemmLaunch& L, GemmParams base, cudaStream_t s) {
  using Sh = BsPairShape<EPI, F4>;
  static_assert(Sh::SMEM_BYTES <= SMEM_LIMIT, "dynamic shared memory per block");
  if (base.sched_tn != Sh::TN || L.K % Sh::BLOCK_K != 0 || base.ksplit != 1 || base.grp == nullptr ||
      L.b_exp == nullptr)
    return cudaErrorInvalidValue;
  if (F4 ? (L.a_sub == nullptr || (L.a_sh_ptr != nullptr && L.a_sh_sub == nullptr))
         : (L.a_exp == nullptr || (L.a_sh_ptr != nullptr && L.a_sh_exp == nullptr)))
    return cudaErrorInvalidValue;
  if (EPI == EPI_SWIGLU && L.a_up_offset % 128 != 0) return cudaErrorInvalidValue;  // 128-row scale tiles
  if (F4 && (reinterpret_cast<uintptr_t>(L.a_ptr) % 32 != 0 || reinterpret_cast<uintptr_t>(L.a_sh_ptr) % 32 != 0))
    return cudaErrorInvalidValue;
  GemmMaps m;
  memset(&m, 0, sizeof(m));
  auto amap = [&](CUtensorMap* t, const void* ptr, int64_t rows_or_groups) {
    if (EPI == EPI_SWIGLU) {
      const int64_t f = L.a_up_offset;
      return F4 ? make_tmap_e2m1_gateup(t, ptr, rows_or_groups, f, L.K, Sh::A_BOX)
                : make_tmap_u8_gateup(t, ptr, rows_or_groups, f, L.K, 128, Sh::A_BOX);
    }
    return F4 ? make_tmap_e2m1(t, ptr, rows_or_groups, L.K, Sh::A_BOX) : make_tmap_u8(t, ptr, rows_or_groups, L.K, Sh::A_BOX, 128);
  };
  const int64_t a_n = (EPI == EPI_SWIGLU) ? L.a_rows / (2 * L.a_up_offset) : L.a_rows;
  const int64_t a_sh_n = (EPI == EPI_SWIGLU) ? 1 : L.a_sh_rows;
  if (!amap(&m.a, L.a_ptr, a_n)) return cudaErrorInvalidValue;
  if (L.a_sh_ptr != nullptr) {
    if (!amap(&m.a_sh, L.a_sh_ptr, a_sh_n)) return cudaErrorInvalidValue;
  } else {
    m.a_sh = m.a;
  }
  for (int i = 0; i < NUM_BOX_H; ++i) {
    const int h = B_BOX << i;
    if (h > Sh::HALF) break;
    if (!make_tmap_pieces(&m.b[i], L.b_ptr, L.b_rows, Sh::PIECES, L.K, h)) return cudaErrorInvalidValue;
  }
  BsParams p;
  static_cast<GemmParams&>(p) = base;
  p.a_exp = L.a_exp;
  p.a_sh_exp = L.a_sh_exp != nullptr ? L.a_sh_exp : L.a_exp;
  p.exp_nr = (L.a_rows_per_group + 127) / 128;
  p.exp_nk = (L.K + 127) / 128;
  p.b_exp = L.b_exp;
  p.a_sub = L.a_sub;
  p.a_sh_sub = L.a_sh_sub != nullptr ? L.a_sh_sub : L.a_sub;
  auto kern = bs_pair_gemm_kernel<EPI, F4>;
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

cudaError_t launch_bs_pair_gemm(const GemmLaunch& L, GemmParams p, cudaStream_t s) {
  const bool f4 = L.q8 == 3;
  if (L.epi == EPI_SWIGLU)
    return f4 ? launch_bs_pair_variant<EPI_SWIGLU, true>(L, p, s) : launch_bs_pair_variant<EPI_SWIGLU, false>(L, p, s);
  if (L.mblk == 2)
    return f4 ? launch_bs_pair_variant<EPI_F32, true>(L, p, s) : launch_bs_pair_variant<EPI_F32, false>(L, p, s);
  return cudaErrorInvalidValue;
}

}  // namespace moe
