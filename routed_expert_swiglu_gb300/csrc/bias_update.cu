// Aux-loss-free load balancing, the inference-side half of its control loop: after a step,
// each expert's selection bias moves by gamma against its load -- an expert that received
// more than the mean load T*k/E loses gamma, one that received fewer gains gamma, one exactly
// at the mean keeps its bias ("MoE compute and communication", section 七.3; "DeepSeek-V4
// MoE", section on auxiliary-loss-free balancing, update speed 0.001).  The load is the
// dispatch histogram (tokens_per_expert) that moe_permute / moe_forward already produce.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

__global__ void __launch_bounds__(256) bias_update_kernel(const int32_t* __restrict__ counts, float* __restrict__ bias,
                                                          int E, long long total, float gamma) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const long long excess = (long long)counts[e] * E - total;  // sign of count - total/E, exactly
  const float step = excess > 0 ? -gamma : (excess < 0 ? gamma : 0.0f);
  bias[e] = bias[e] + step;
}

}  // namespace moe

extern "C" moe_status moe_update_bias(moe_plan* plan, int32_t T, const int32_t* counts, float* bias, float gamma,
                                      moe_stream_t stream) {
  using namespace moe;
  if (plan == nullptr || counts == nullptr || bias == nullptr) return MOE_ERR_INVALID_ARG;
  const moe_config& c = *plan_config(plan);
  if (T < 0 || T > c.max_tokens || !(gamma >= 0.0f)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(counts) | reinterpret_cast<uintptr_t>(bias)) & 3u) return MOE_ERR_ALIGNMENT;
  const int E = c.n_experts;
  bias_update_kernel<<<(E + 255) / 256, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      counts, bias, E, (long long)T * c.top_k, gamma);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
