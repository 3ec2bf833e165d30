// moe_permute_noalloc: the dispatch permutation of moe_permute for callers that cannot
// allocate device memory.
//
// Some callers are handed only their input and output buffers and may not allocate: a plugin
// running inside a host framework that owns all device memory through its own allocator, or a
// latency-critical serving loop where cudaMalloc (which can synchronise the device) is not
// allowed.  Such a caller cannot provide the workspace moe_permute needs.  This entry point
// runs the same histogram / scan / scatter kernels with their scratch (per-chunk histograms,
// the grouped-GEMM schedule and the error word) in a fixed-size array of device memory that
// belongs to the library itself: it is a file-scope __device__ variable, so every GPU that
// loads the library holds it until the process exits, and no call allocates anything.
//
// The array is shared by every call on a device and keeps the last call's contents; the
// entry point clears the one word that must start at zero (the error word) on every call.
// An expert id outside [0, E) is clamped into range (as moe_permute does) and flagged in that
// word, which moe_permute_noalloc_status reads back.
// Two calls whose work overlaps on the GPU (different streams, no ordering between them)
// race on the array.  The first call on a device looks up the array's device address
// (cudaGetSymbolAddress, once per device, with that device current); make that first call
// before any stream capture.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// Largest batch this entry point accepts: T * top_k <= 131072 assignments (e.g. T = 16384 at
// top_k = 8), with E <= 512 experts (the plan limit).
constexpr int NOALLOC_MAX_ASSIGN = 131072;
constexpr int NOALLOC_MAX_BLOCKS = NOALLOC_MAX_ASSIGN / PERMUTE_CHUNK;
constexpr int NOALLOC_MAX_GROUPS = MAX_EXPERTS + 1;  // routed + shared
// row tiles of the schedule: at most E + ceil(N / 64) + ceil(T / 64) + 1 with T <= N, for the
// schedule's row tiles of at least 64 rows (token_tile_for gives 64 or MOE_TN_PREFILL)
static_assert(MOE_TN_PREFILL >= 64, "the fixed scratch is sized for row tiles of at least 64 rows");
constexpr int NOALLOC_MAX_ROWTILES = MAX_EXPERTS + 2 * (NOALLOC_MAX_ASSIGN / 64) + 2;

constexpr size_t OFF_ERR = 0;
constexpr size_t OFF_HIST = 256;
constexpr size_t OFF_GRP = OFF_HIST + (size_t)NOALLOC_MAX_BLOCKS * MAX_EXPERTS * 4;
constexpr size_t OFF_RT2G = OFF_GRP + (size_t)(NOALLOC_MAX_GROUPS + 1) * 16;
constexpr size_t SCRATCH_BYTES = OFF_RT2G + (size_t)NOALLOC_MAX_ROWTILES * 4;  // ~0.33 MB

static __device__ __align__(256) unsigned char g_permute_scratch[SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_mutex;
void* g_scratch_ptr[MAX_DEVICES] = {nullptr};

// Device address of g_permute_scratch on the current device, looked up once per device.
moe_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= MAX_DEVICES) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_permute_scratch) != cudaSuccess || ptr == nullptr) return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_permute_noalloc(moe_plan* plan, int32_t T, const int32_t* topk_ids, int32_t* counts,
                                          int32_t* offsets, int32_t* perm_tok, int32_t* inv,
                                          moe_stream_t stream) {
  using namespace moe;
  if (plan == nullptr) return MOE_ERR_INVALID_ARG;
  const moe_config& c = *plan_config(plan);
  if (T < 0 || T > c.max_tokens) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (topk_ids == nullptr || counts == nullptr || offsets == nullptr || perm_tok == nullptr || inv == nullptr)
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(topk_ids) | reinterpret_cast<uintptr_t>(counts) |
       reinterpret_cast<uintptr_t>(offsets) | reinterpret_cast<uintptr_t>(perm_tok) |
       reinterpret_cast<uintptr_t>(inv)) & 3u)
    return MOE_ERR_ALIGNMENT;
  const int64_t N = (int64_t)T * c.top_k;
  if (N > NOALLOC_MAX_ASSIGN) return MOE_ERR_UNSUPPORTED;  // beyond the static scratch
  void* scratch = nullptr;
  const moe_status st = scratch_for_current_device(&scratch);
  if (st != MOE_OK) return st;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(scratch);
  int* err = reinterpret_cast<int*>(base + OFF_ERR);
  if (cudaMemsetAsync(err, 0, sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
  PermuteLaunch pm;
  memset(&pm, 0, sizeof(pm));
  pm.topk_ids = topk_ids;
  pm.T = T;
  pm.k = c.top_k;
  pm.E = c.n_experts;
  pm.n_shared = c.n_shared;
  pm.TN = token_tile_for(T, c.top_k, c.n_experts);
  pm.nblk = (int)((N + PERMUTE_CHUNK - 1) / PERMUTE_CHUNK);
  pm.blockhist = reinterpret_cast<int32_t*>(base + OFF_HIST);
  pm.counts = counts;
  pm.offsets = offsets;
  pm.grp = reinterpret_cast<int4*>(base + OFF_GRP);
  pm.rt2g = reinterpret_cast<int32_t*>(base + OFF_RT2G);
  pm.perm_tok = perm_tok;
  pm.inv = inv;
  pm.err = err;
  pm.num_sms = sms;
  if (launch_permute(pm, s) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

extern "C" moe_status moe_permute_noalloc_status(moe_stream_t stream) {
  using namespace moe;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= MAX_DEVICES) return MOE_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    scratch = g_scratch_ptr[dev];
  }
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  if (scratch == nullptr) return MOE_OK;  // no call on this device yet: nothing flagged
  int v = 0;
  if (cudaMemcpy(&v, static_cast<char*>(scratch) + OFF_ERR, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  return v != 0 ? MOE_ERR_DEVICE_INPUT : MOE_OK;
}
