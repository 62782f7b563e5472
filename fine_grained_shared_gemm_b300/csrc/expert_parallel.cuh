// Expert parallelism: the row regrouping between the all-to-all exchange and
// the local expert GEMMs.
//
// With the routed experts split contiguously over D ranks (E_loc = E / D per
// rank; page "02 · 细粒度 MoE：从 Mixtral 到 DeepSeekMoE", §3.2: routed
// experts are spread over devices and tokens reach them through all-to-all,
// the shared experts are replicated and need no exchange), the rows a rank
// receives arrive source-major: for each source rank s, for each of this
// rank's experts e, the rows s sends to e (in s's dispatch order).  The
// grouped GEMM wants them expert-major: for each expert e, for each source s.
// Both orders are fixed by the count matrix counts[s][e] alone, so one kernel
// moves rows either way: source-major -> expert-major before the expert
// FFN, expert-major -> source-major after it (the inverse permutation), and
// writes the expert offsets of the expert-major order.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kRegroupThreads = 1024;   // D · E_loc <= 1024 segments

// Exclusive prefix of v over the block's 1024 threads (thread order).
__device__ __forceinline__ int block_exclusive_scan_1024(int v, int* warp_tot) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  __syncthreads();
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  if (w == 0) {
    int s = warp_tot[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += y;
    }
    warp_tot[lane] = s;
  }
  __syncthreads();
  return incl - v + (w > 0 ? warp_tot[w - 1] : 0);
}

// counts: [D][E_loc] rows source s sends to local expert e.  Segment (s, e)
// has index s · E_loc + e.  Every block computes both segment-offset tables
// (source-major and expert-major) in shared memory, then its warps move rows:
// row r of the source-major order goes to (or comes from) row
// exp_off[seg] + (r - src_off[seg]) of the expert-major order.
template <typename T>
__global__ void __launch_bounds__(kRegroupThreads)
    ep_regroup_kernel(const int32_t* __restrict__ counts, int D, int El, int H,
                      const T* __restrict__ src, T* __restrict__ dst,
                      int32_t* __restrict__ expert_offsets, int to_expert_major) {
  __shared__ int src_off[kRegroupThreads];
  __shared__ int exp_off[kRegroupThreads];
  __shared__ int warp_tot[32];
  __shared__ int total;
  const int n = D * El, t = threadIdx.x;
  const int v = t < n ? __ldg(counts + t) : 0;
  const int so = block_exclusive_scan_1024(v, warp_tot);
  if (t < n) src_off[t] = so;
  if (t == kRegroupThreads - 1) total = so + v;
  // expert-major order: position t is (e = t / D, s = t % D)
  const int seg2 = t < n ? (t % D) * El + t / D : 0;
  const int v2 = t < n ? __ldg(counts + seg2) : 0;
  const int eo = block_exclusive_scan_1024(v2, warp_tot);
  if (t < n) exp_off[seg2] = eo;
  __syncthreads();
  if (blockIdx.x == 0 && expert_offsets != nullptr) {
    if (t < El) expert_offsets[t] = exp_off[t];  // segment (s = 0, e = t)
    if (t == 0) expert_offsets[El] = total;
  }
  const int rows = total;
  constexpr int V = Vec16<T>::N;
  const int nvec = H / V;
  const int lane = t & 31;
  const int warps = gridDim.x * (kRegroupThreads / 32);
  for (int r = blockIdx.x * (kRegroupThreads / 32) + (t >> 5); r < rows; r += warps) {
    // the last segment starting at or before r is the non-empty one holding r
    int lo = 0, hi = n;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (src_off[mid] <= r) lo = mid; else hi = mid;
    }
    const int e_row = exp_off[lo] + (r - src_off[lo]);
    const int from = to_expert_major ? r : e_row, to = to_expert_major ? e_row : r;
    const uint4* s = reinterpret_cast<const uint4*>(src + static_cast<size_t>(from) * H);
    uint4* d = reinterpret_cast<uint4*>(dst + static_cast<size_t>(to) * H);
    for (int q = lane; q < nvec; q += 32) d[q] = __ldg(s + q);
  }
}

}  // namespace moe
