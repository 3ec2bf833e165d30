// Per-SM ingest rate of asynchronous copies into shared memory (test infrastructure, not part of
// the library).  One CTA per SM streams 16 KB stages into a ring of shared-memory slots: a
// producer lane issues the copies, a consumer lane releases each stage as soon as it has landed,
// so the rate measured is what the memory system delivers into the SMs with nothing else
// running.  Forms: (0) 2-D tiled TMA boxes of 128 rows x 128 bytes over contiguous rows, (1) one
// 16 KB cp.async.bulk per stage, (2) 2-D tiled TMA boxes over rows 2 KB (L2 case) or 8 KB (HBM
// case) apart, like the rows of a weight matrix, (3) four 4 KB cp.async.bulk per stage.  Sources:
// each SM re-reading its own 256 KB (L2-resident) or streaming its own 16 MB once (HBM).  Every
// wait is bounded (the library's mbarrier helpers), and every copy stays inside its SM's region.
//
// Prints one line per (source, form, ring depth): "<L2|HBM> <form> <stages> <GB/s total> <GB/s per SM> <err>".
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#include "../routed_expert_swiglu_gb300/csrc/common.cuh"

using namespace moe;

namespace {

constexpr int STAGE = 16384;
constexpr int MAXST = 14;

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__global__ void __launch_bounds__(64, 1)
    ingest(const __grid_constant__ CUtensorMap map0, const __grid_constant__ CUtensorMap map2, const uint8_t* src,
           int form, int stages, int loads, int wrap, long long cta_bytes, int kbs, int rbs, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bars[2 * MAXST];
  __shared__ int abort_flag;
  const uint32_t b0 = smem_u32(bars);
  auto full = [&](int s) { return b0 + 8u * s; };
  auto empty = [&](int s) { return b0 + 8u * (MAXST + s); };
  if (threadIdx.x == 0) {
    for (int s = 0; s < MAXST; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const int c = blockIdx.x;
  if (threadIdx.x == 0) {
    int s = 0;
    uint32_t ph = 0;
    for (int i = 0; i < loads; ++i) {
      if (!mbar_wait(empty(s), ph ^ 1u, &abort_flag, err)) break;
      const uint32_t dst = smem_u32(smem + s * STAGE);
      mbar_arrive_expect_tx(full(s), STAGE);
      const uint8_t* g = src + c * cta_bytes + (long long)(i % wrap) * STAGE;
      if (form == 0) {
        tma_load_2d(dst, &map0, full(s), 0, (int)(c * (cta_bytes / 128) + (i % wrap) * 128));
      } else if (form == 1) {
        bulk_load(dst, g, STAGE, full(s));
      } else if (form == 2) {
        tma_load_2d(dst, &map2, full(s), (i % kbs) * 64, (c * rbs + (i / kbs) % rbs) * 128);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) bulk_load(dst + q * 4096, g + q * 4096, 4096, full(s));
      }
      if (++s == stages) {
        s = 0;
        ph ^= 1u;
      }
    }
  } else if (threadIdx.x == 32) {
    int s = 0;
    uint32_t ph = 0;
    for (int i = 0; i < loads; ++i) {
      if (!mbar_wait(full(s), ph, &abort_flag, err)) break;
      mbar_arrive(empty(s));
      if (++s == stages) {
        s = 0;
        ph ^= 1u;
      }
    }
  }
  __syncthreads();
  if (abort_flag && threadIdx.x == 0) {  // a wait gave up: let copies in flight land first
    const unsigned long long t0 = global_timer_ns();
    while (global_timer_ns() - t0 < QUIET_NS) __nanosleep(1000);
  }
  __syncthreads();
}

typedef CUresult (*EncFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*, const cuuint64_t*,
                          const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                          CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// bf16 matrix [rows, cols] (row stride cols * 2 bytes), box 64 x 128, 128-byte swizzle
bool encode(EncFn enc, CUtensorMap* m, void* p, uint64_t cols, uint64_t rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace

#define CK(x)                                                            \
  do {                                                                   \
    cudaError_t e_ = (x);                                                \
    if (e_ != cudaSuccess) {                                             \
      printf("CUDA error %s at line %d\n", cudaGetErrorString(e_), __LINE__); \
      return 1;                                                          \
    }                                                                    \
  } while (0)

int main() {
  int sms = 0;
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  void* fp = nullptr;
  cudaDriverEntryPointQueryResult q;
  CK(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fp, 12000, cudaEnableDefault, &q));
  if (q != cudaDriverEntryPointSuccess || fp == nullptr) {
    printf("no cuTensorMapEncodeTiled\n");
    return 1;
  }
  EncFn enc = reinterpret_cast<EncFn>(fp);
  const long long l2_cta = 256ll << 10, hbm_cta = 16ll << 20;
  uint8_t* buf = nullptr;
  CK(cudaMalloc(&buf, (size_t)sms * hbm_cta));
  CK(cudaMemset(buf, 1, (size_t)sms * hbm_cta));
  int* err = nullptr;
  CK(cudaMalloc(&err, sizeof(int)));
  CK(cudaMemset(err, 0, sizeof(int)));
  CK(cudaFuncSetAttribute(ingest, cudaFuncAttributeMaxDynamicSharedMemorySize, MAXST * STAGE + 1024));
  cudaEvent_t e0, e1;
  CK(cudaEventCreate(&e0));
  CK(cudaEventCreate(&e1));
  const char* names[4] = {"tiled_contiguous", "bulk_16K", "tiled_strided", "bulk_4Kx4"};
  for (int hbm = 0; hbm < 2; ++hbm) {
    const long long cta = hbm ? hbm_cta : l2_cta;
    const int wrap = (int)(cta / STAGE);       // stages in one SM's region
    const uint64_t cols2 = hbm ? 4096 : 1024;  // strided form: row length in bf16 elements
    const int kbs = (int)(cols2 / 64);         // boxes along a row
    const int rbs = (int)(cta / (cols2 * 2) / 128);  // 128-row blocks in one SM's region
    CUtensorMap m0, m2;
    if (!encode(enc, &m0, buf, 64, (uint64_t)sms * cta / 128) || !encode(enc, &m2, buf, cols2, (uint64_t)sms * rbs * 128)) {
      printf("tensor map encoding failed\n");
      return 1;
    }
    for (int form = 0; form < 4; ++form) {
      for (int stages : {6, 10, 14}) {
        const int loads = hbm ? wrap : 4096;
        float ms = 0.0f;
        for (int rep = 0; rep < 2; ++rep) {
          CK(cudaEventRecord(e0));
          ingest<<<sms, 64, MAXST * STAGE + 1024>>>(m0, m2, buf, form, stages, loads, wrap, cta, kbs, rbs, err);
          CK(cudaGetLastError());
          CK(cudaEventRecord(e1));
          CK(cudaEventSynchronize(e1));
          CK(cudaEventElapsedTime(&ms, e0, e1));
        }
        int herr = 0;
        CK(cudaMemcpy(&herr, err, sizeof(int), cudaMemcpyDeviceToHost));
        const double gbs = (double)sms * loads * STAGE / (ms * 1e-3) / 1e9;
        printf("%s %s %d %.1f %.2f %d\n", hbm ? "HBM" : "L2", names[form], stages, gbs, gbs / sms, herr);
      }
    }
  }
  CK(cudaFree(buf));
  CK(cudaFree(err));
  return 0;
}
