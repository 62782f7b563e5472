// Load balancing without an auxiliary loss (page "MoE 的分水岭——DeepSeek
// 配方与 2026 年的主流形态", ch. 7 §7.4): after a step, each expert's load is
// compared with the mean load T·k / E; an overloaded expert's selection bias
// is lowered by gamma, an underloaded one's raised by gamma, one exactly at
// the mean is kept.  The comparison is exact (load · E against T·k in
// integers) and the update is one fp32 addition, so the result does not depend
// on the order of anything.
#pragma once

#include "common.cuh"

namespace moe {

// One thread per expert; loads come from the dispatch offsets.
__global__ void __launch_bounds__(256) bias_update_kernel(const int32_t* __restrict__ offsets,
                                                          int E, long long routed_rows,
                                                          float gamma, float* __restrict__ bias,
                                                          int32_t* __restrict__ loads) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const int load = offsets[e + 1] - offsets[e];
  if (loads != nullptr) loads[e] = load;
  const long long scaled = static_cast<long long>(load) * E;
  float b = bias[e];
  if (scaled > routed_rows) b = __fsub_rn(b, gamma);
  else if (scaled < routed_rows) b = __fadd_rn(b, gamma);
  bias[e] = b;
}

}  // namespace moe
