// Load balancing without an auxiliary loss (page "MoE 的分水岭——DeepSeek
// 配方与 2026 年的主流形态", ch. 7 §7.4): after a step, each expert's load is
// compared with the mean load T·k / E; an overloaded expert's selection bias
// is lowered by gamma, an underloaded one's raised by gamma, one exactly at
// the mean is kept.  The comparison is exact (load · E against T·k in
// integers) and the update is one fp32 addition, so the result does not depend
// on the order of anything.
#pragma once

#include "common.cuh"
#include "route.cuh"

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

// Statistics of the expert-level balance loss (page "19-deepseek-moe",
// ai.tomabc.com, load-balance section; the loss is proportional to
// Σ_i f_i P_i):
//   f_i = E · load_i / (k · T), the routing distribution counted over all E
//         routed experts (an even routing gives f_i = 1);
//   P_i = (1/T) Σ_t p_{i,t}, p_t the token's gate distribution over the E
//         routed experts: softmax scores, or sigmoid scores divided by their
//         sum over all E.
// P is reduced in two fixed-order passes (per 256-token chunk in fp32, over
// chunks in fp64), so it does not depend on scheduling.
constexpr int kStatChunk = 256;

// Block = one chunk of kStatChunk tokens.  Warps first find each token's
// normaliser (softmax: max and 1/Σexp; sigmoid: 1/Σσ), then thread e sums
// p_{e,t} over the chunk's tokens in order.
__global__ void __launch_bounds__(256) balance_partial_kernel(const float* __restrict__ logits,
                                                              int T, int E, int sigmoid,
                                                              float* __restrict__ partial) {
  __shared__ float s_max[kStatChunk], s_inv[kStatChunk];
  const int t0 = blockIdx.x * kStatChunk;
  const int nt = min(kStatChunk, T - t0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j = warp; j < nt; j += blockDim.x >> 5) {
    const float* z = logits + static_cast<size_t>(t0 + j) * E;
    float m = 0.0f, d = 0.0f;
    if (sigmoid) {
      for (int e = lane; e < E; e += 32) d += 1.0f / (1.0f + expf(-__ldg(z + e)));
    } else {
      m = -CUDART_INF_F;
      for (int e = lane; e < E; e += 32) m = fmaxf(m, __ldg(z + e));
      m = warp_max(m);
      for (int e = lane; e < E; e += 32) d += expf(__ldg(z + e) - m);
    }
    d = warp_sum(d);
    if (lane == 0) {
      s_max[j] = m;
      s_inv[j] = 1.0f / d;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float acc = 0.0f;
    for (int j = 0; j < nt; ++j) {
      const float v = __ldg(logits + static_cast<size_t>(t0 + j) * E + e);
      const float q = sigmoid ? 1.0f / (1.0f + expf(-v)) : expf(v - s_max[j]);
      acc += q * s_inv[j];
    }
    partial[static_cast<size_t>(blockIdx.x) * E + e] = acc;
  }
}

// One thread per expert: P_e from the chunk partials (fp64, chunk order) and
// f_e from the dispatch offsets (one fp64 division of exact integers).
__global__ void __launch_bounds__(256) balance_final_kernel(const float* __restrict__ partial,
                                                            int n_chunks,
                                                            const int32_t* __restrict__ offsets,
                                                            int T, int E, int k,
                                                            float* __restrict__ f,
                                                            float* __restrict__ p) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  double acc = 0.0;
  for (int c = 0; c < n_chunks; ++c) acc += partial[static_cast<size_t>(c) * E + e];
  p[e] = T > 0 ? static_cast<float>(acc / T) : 0.0f;
  const long long load = offsets[e + 1] - offsets[e];
  const long long rows = static_cast<long long>(k) * T;
  f[e] = rows > 0 ? static_cast<float>(static_cast<double>(load * E) / static_cast<double>(rows))
                  : 0.0f;
}

}  // namespace moe
