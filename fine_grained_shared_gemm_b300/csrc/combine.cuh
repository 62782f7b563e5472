// Combine: h_t = u_t + Σ_{j<Ks} y_shared[j, t] + Σ_{s<k} g[t, s] · y_perm[slot_row[t, s]]
// (page "02 · 细粒度 MoE：从 Mixtral 到 DeepSeekMoE", §3.1 Eq. 9–11: shared
// experts, gate-weighted routed experts, residual).  fp32 accumulation in this
// fixed order and one rounding to the output type, so the result is the same
// on every run.  A warp takes one (token, segment of the row) work item at a
// time, 16-byte vectors along H: one segment per token for large batches,
// several for small ones so that enough warps are busy (each vector's sum is
// the same whichever warp computes it).
#pragma once

#include "common.cuh"

namespace moe {

template <typename T>
__global__ void __launch_bounds__(256) combine_kernel(
    const T* __restrict__ u, const T* __restrict__ y_perm, const T* __restrict__ y_shared,
    const float* __restrict__ topk_w, const int32_t* __restrict__ slot_row, int n_tokens, int H,
    int k, int Ks, int nseg, int seg_vecs, T* __restrict__ h) {
  constexpr int V = Vec16<T>::N;
  __shared__ int s_row[8][32];
  __shared__ float s_w[8][32];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int nvec = H / V;
  const long long items = static_cast<long long>(n_tokens) * nseg;
  for (long long it = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; it < items; it += warps) {
    const int t = static_cast<int>(it / nseg);
    const int v0 = static_cast<int>(it - static_cast<long long>(t) * nseg) * seg_vecs;
    const int v1 = min(nvec, v0 + seg_vecs);
    __syncwarp();
    if (lane < k) {  // k <= 32: slot s's row and weight, broadcast through shared memory
      s_row[wib][lane] = __ldg(slot_row + static_cast<size_t>(t) * k + lane);
      s_w[wib][lane] = __ldg(topk_w + static_cast<size_t>(t) * k + lane);
    }
    __syncwarp();
    // two vectors a lane per pass: the loads of the second are issued with
    // the first's, doubling the bytes in flight (V3-shaped batch: 291 -> 236
    // us, 0.70 -> 0.87 of the copy rate; unrolling by 4 gained nothing)
#pragma unroll 2
    for (int v = v0 + lane; v < v1; v += 32) {
      float acc[V], y[V];
      Vec16<T>::load(u + static_cast<size_t>(t) * H + v * V, acc);
      for (int j = 0; j < Ks; ++j) {
        Vec16<T>::load(y_shared + (static_cast<size_t>(j) * n_tokens + t) * H + v * V, y);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] += y[i];
      }
      // routed slots in groups of 8: all loads of a group are issued before
      // any is used (independent predicated loads), then accumulated in slot
      // order, so the sum is the same as one slot at a time
      for (int s0 = 0; s0 < k; s0 += 8) {
        uint4 raw[8];
#pragma unroll
        for (int d = 0; d < 8; ++d) {
          const int row = s0 + d < k ? s_row[wib][s0 + d] : -1;
          raw[d] = row >= 0 ? __ldg(reinterpret_cast<const uint4*>(y_perm + static_cast<size_t>(row) * H + v * V))
                            : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int d = 0; d < 8; ++d) {
          if (s0 + d >= k || s_row[wib][s0 + d] < 0) continue;
          const float w = s_w[wib][s0 + d];
          Vec16<T>::load(reinterpret_cast<const T*>(&raw[d]), y);
#pragma unroll
          for (int i = 0; i < V; ++i) acc[i] = fmaf(w, y[i], acc[i]);
        }
      }
      Vec16<T>::store(h + static_cast<size_t>(t) * H + v * V, acc);
    }
  }
}

}  // namespace moe
