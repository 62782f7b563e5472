// Router scores, top-k choice and gate weights: one warp per token.
//
// Softmax gate (page "02 · 细粒度 MoE：从 Mixtral 到 DeepSeekMoE", §2.1
// Eq. 6–8): s_i = softmax_i(z) over the routed experts; the top-k of s are the
// top-k of z (softmax is increasing in the logit), so the choice is taken on
// the fp32 logits exactly; g = s for the chosen, not renormalised.
// Sigmoid gate (§3.1 Eq. 12–15; page "MoE 的分水岭", ch. 7 §7.4):
// s_i = sigmoid(z_i); the choice is taken on fp32(s_i) + b_i, the weights are
// the raw s_i of the chosen divided by their sum.
// Ties go to the lower expert index.  The sum reductions use a fixed
// butterfly order, so the result does not depend on scheduling.
// Group-limited routing (§4, node-limited routing): with n_groups > 0 the
// experts form groups of E / n_groups consecutive indices; a group's score is
// the sum (float64) of its experts' softmax scores, or keys s + b; the
// topk_groups best groups are kept (ties to the lower group index) and the
// top-k is taken among their experts only.
#pragma once

#include <math_constants.h>

#include "common.cuh"

namespace moe {

struct Best {
  float key;
  float score;
  int idx;
};

// (a beats b): larger key, or equal key and lower index.
__device__ __forceinline__ bool beats(float ka, int ia, float kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

__device__ __forceinline__ Best warp_best(Best b) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float k = __shfl_xor_sync(0xffffffffu, b.key, off);
    const float s = __shfl_xor_sync(0xffffffffu, b.score, off);
    const int i = __shfl_xor_sync(0xffffffffu, b.idx, off);
    if (beats(k, i, b.key, b.idx)) b = Best{k, s, i};
  }
  return b;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

__device__ __forceinline__ double warp_sum_f64(double x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
  return x;
}

// Router logits cut along H into S contraction ranges (few-token batches):
// logits[t, e] = (part[0][t, e] + ... + part[S-1][t, e]) + o_e, the ranges
// added in order so that the result is the same on every run.
__global__ void __launch_bounds__(256) sum_logit_partials_kernel(
    const float* __restrict__ part, int S, long long n, int E, const float* __restrict__ offset,
    float* __restrict__ logits) {
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < n; i += gridDim.x * 256LL) {
    float acc = __ldg(part + i);
    for (int sp = 1; sp < S; ++sp) acc += __ldg(part + static_cast<long long>(sp) * n + i);
    if (offset != nullptr) acc += __ldg(offset + i % E);
    logits[i] = acc;
  }
}

// NPL logits per lane: expert e = lane + 32 * i.  Requires E <= 32 * NPL and
// top_k <= 32.
template <int NPL>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits,
                                                    const float* __restrict__ bias, int T,
                                                    int E, int k, int gate, int n_groups,
                                                    int topk_groups,
                                                    int32_t* __restrict__ topk_idx,
                                                    float* __restrict__ topk_w,
                                                    float* __restrict__ kth_gap) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps) {
    const float* z = logits + static_cast<size_t>(t) * E;
    float key[NPL], score[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      key[i] = e < E ? __ldg(z + e) : -CUDART_INF_F;
    }
    if (gate == 0) {  // softmax
      float m = -CUDART_INF_F;
#pragma unroll
      for (int i = 0; i < NPL; ++i) m = fmaxf(m, key[i]);
      m = warp_max(m);
      float part = 0.0f;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        score[i] = (lane + 32 * i < E) ? expf(key[i] - m) : 0.0f;
        part += score[i];
      }
      const float denom = warp_sum(part);
#pragma unroll
      for (int i = 0; i < NPL; ++i) score[i] = score[i] / denom;
    } else {  // sigmoid + selection bias
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
          score[i] = 1.0f / (1.0f + expf(-key[i]));
          key[i] = score[i] + (bias != nullptr ? __ldg(bias + e) : 0.0f);
        } else {
          score[i] = 0.0f;
        }
      }
    }

    if (n_groups > 0) {
      // lane g ends up holding group g's score
      const int gs = E / n_groups;
      double my_group = -CUDART_INF;
      for (int g = 0; g < n_groups; ++g) {
        double part = 0.0;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
          const int e = lane + 32 * i;
          if (e < E && e / gs == g) part += static_cast<double>(gate == 0 ? score[i] : key[i]);
        }
        const double sum = warp_sum_f64(part);
        if (lane == g) my_group = sum;
      }
      uint32_t keep = 0;  // bit g: group g kept
      for (int r = 0; r < topk_groups; ++r) {
        double best = my_group;
        int best_g = lane < n_groups && !((keep >> lane) & 1u) ? lane : 0x7fffffff;
        if (best_g == 0x7fffffff) best = -CUDART_INF;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const double ob = __shfl_xor_sync(0xffffffffu, best, off);
          const int og = __shfl_xor_sync(0xffffffffu, best_g, off);
          if (ob > best || (ob == best && og < best_g)) { best = ob; best_g = og; }
        }
        keep |= 1u << best_g;
      }
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((keep >> (e / gs)) & 1u)) key[i] = -CUDART_INF_F;
      }
    }

    uint32_t taken = 0;
    float my_score = 0.0f;
    int my_idx = 0;
    Best last{0.0f, 0.0f, 0};
    for (int r = 0; r < k; ++r) {
      Best b{-CUDART_INF_F, 0.0f, 0x7fffffff};
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && beats(key[i], e, b.key, b.idx))
          b = Best{key[i], score[i], e};
      }
      b = warp_best(b);
      if ((b.idx & 31) == lane) taken |= 1u << (b.idx >> 5);
      if (lane == r) { my_score = b.score; my_idx = b.idx; }
      last = b;
    }
    if (kth_gap != nullptr) {
      float gap = CUDART_INF_F;
      if (k > 0 && k < E) {
        Best b{-CUDART_INF_F, 0.0f, 0x7fffffff};
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
          const int e = lane + 32 * i;
          if (e < E && !((taken >> i) & 1u) && beats(key[i], e, b.key, b.idx))
            b = Best{key[i], score[i], e};
        }
        b = warp_best(b);
        // no (k+1)-th expert among the kept groups: no competitor
        gap = b.key == -CUDART_INF_F ? CUDART_INF_F
                                      : (gate == 0) ? last.score - b.score : last.key - b.key;
      }
      if (lane == 0) kth_gap[t] = gap;
    }
    float w = my_score;
    if (gate != 0) {
      const float tot = warp_sum(lane < k ? my_score : 0.0f);
      w = my_score / tot;
    }
    if (lane < k) {
      topk_idx[static_cast<size_t>(t) * k + lane] = my_idx;
      topk_w[static_cast<size_t>(t) * k + lane] = w;
    }
  }
}

}  // namespace moe
