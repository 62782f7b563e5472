// Dispatch: group the T·k (token, slot) entries by expert, without dropping
// any (page "02 · 细粒度 MoE", §4: no token dropping), and gather the token
// rows into expert-contiguous order.
//
// Rows are ordered by expert, then token; every step is deterministic:
//   1. dispatch_count   per chunk of tokens, a per-expert histogram
//   2. dispatch_scan    per expert, exclusive prefix over chunks; exclusive
//                       prefix over experts -> expert_offsets
//   3. dispatch_scatter each chunk assigns stable ranks (warp match + popc)
//                       and writes slot_row / row_token
//   4. scatter_token_rows  u_perm[slot_row[t, s]] = u[t]: each token row is
//                       read once and written to its k rows (16-byte vectors)
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kDispatchChunk = 256;   // tokens per chunk
constexpr int kDispatchWarps = 8;     // warps per chunk block

__global__ void __launch_bounds__(256) dispatch_count(const int32_t* __restrict__ idx, int T,
                                                      int k, int E,
                                                      int32_t* __restrict__ chunk_hist) {
  extern __shared__ int hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int t0 = blockIdx.x * kDispatchChunk;
  const int n = min(kDispatchChunk, T - t0) * k;
  const int32_t* src = idx + static_cast<size_t>(t0) * k;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const int e = __ldg(src + j);
    if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    else raise_device_error(DEV_ERR_BAD_EXPERT);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_hist[static_cast<size_t>(blockIdx.x) * E + e] = hist[e];
}

// One block of 1024 threads; E <= 1024.
__global__ void __launch_bounds__(1024) dispatch_scan(const int32_t* __restrict__ chunk_hist,
                                                      int n_chunks, int E,
                                                      int32_t* __restrict__ chunk_base,
                                                      int32_t* __restrict__ offsets) {
  __shared__ int warp_tot[32];
  const int e = threadIdx.x;
  int total = 0;
  if (e < E) {
    for (int c = 0; c < n_chunks; ++c) {
      const int v = chunk_hist[static_cast<size_t>(c) * E + e];
      chunk_base[static_cast<size_t>(c) * E + e] = total;
      total += v;
    }
  }
  // exclusive scan of per-expert totals over e
  const int lane = e & 31, w = e >> 5;
  int incl = total;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  if (w == 0) {
    int s = warp_tot[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += y;
    }
    warp_tot[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const int excl = incl - total + (w > 0 ? warp_tot[w - 1] : 0);
  if (e < E) {
    offsets[e] = excl;
    for (int c = 0; c < n_chunks; ++c) chunk_base[static_cast<size_t>(c) * E + e] += excl;
  }
  if (e == E - 1) offsets[E] = excl + total;
}

// One block (kDispatchWarps warps) per chunk; dynamic smem kDispatchWarps * E ints.
__global__ void __launch_bounds__(kDispatchWarps * 32)
    dispatch_scatter(const int32_t* __restrict__ idx, int T, int k, int E,
                     const int32_t* __restrict__ chunk_base, int32_t* __restrict__ row_token,
                     int32_t* __restrict__ slot_row) {
  extern __shared__ int cnt[];  // [warp][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kDispatchWarps * E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const int t0 = blockIdx.x * kDispatchChunk;
  const int n = min(kDispatchChunk, T - t0) * k;
  const int per = ((n + kDispatchWarps - 1) / kDispatchWarps + 31) & ~31;
  const int j_begin = min(n, warp * per), j_end = min(n, j_begin + per);
  const int32_t* src = idx + static_cast<size_t>(t0) * k;
  int* my = cnt + warp * E;
  const uint32_t lt_mask = (1u << lane) - 1u;

  // pass 1: per-warp counts of its contiguous range
  for (int j0 = j_begin; j0 < j_end; j0 += 32) {
    const int j = j0 + lane;
    int e = (j < j_end) ? __ldg(src + j) : -1;
    if (e >= E) e = -1;
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (same & lt_mask) == 0) my[e] += __popc(same);
  }
  __syncthreads();
  // exclusive prefix over warps, starting at this chunk's base for the expert
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = chunk_base[static_cast<size_t>(blockIdx.x) * E + e];
    for (int w = 0; w < kDispatchWarps; ++w) {
      const int c = cnt[w * E + e];
      cnt[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  // pass 2: stable ranks in entry order (token-major), so rows ascend in token
  for (int j0 = j_begin; j0 < j_end; j0 += 32) {
    const int j = j0 + lane;
    const bool in_range = j < j_end;
    int e = in_range ? __ldg(src + j) : -1;
    if (e >= E) e = -1;
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    int row = 0;
    if (e >= 0) row = my[e] + __popc(same & lt_mask);
    __syncwarp();
    if (e >= 0 && (same & lt_mask) == 0) my[e] += __popc(same);
    __syncwarp();
    if (in_range) {
      const int jg = t0 * k + j;
      slot_row[jg] = e >= 0 ? row : -1;  // an invalid expert index maps to no row
      if (e >= 0) row_token[row] = jg / k;
    }
  }
}

// u_perm[slot_row[t·k + s]] = u[t] for every token t and slot s (entries of
// -1, an invalid expert, are skipped); one warp per token.  Each token row is
// read from HBM once and written k times, instead of being read once per
// permuted row as a gather by row_token would (which re-reads rows that the
// stream of writes has pushed out of L2).
template <typename T>
__global__ void __launch_bounds__(256) scatter_token_rows(const T* __restrict__ u, int T_tokens,
                                                          int k,
                                                          const int32_t* __restrict__ slot_row,
                                                          int H, int nseg, int seg_vecs,
                                                          T* __restrict__ u_perm) {
  constexpr int kMaxK = 32;
  __shared__ int s_row[8][kMaxK];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int nvec = H * static_cast<int>(sizeof(T)) / 16;
  // work items (token, segment of its row), as in the combine
  const long long items = static_cast<long long>(T_tokens) * nseg;
  for (long long it = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; it < items; it += warps) {
    const int t = static_cast<int>(it / nseg);
    const int v0 = static_cast<int>(it - static_cast<long long>(t) * nseg) * seg_vecs;
    const int v1 = min(nvec, v0 + seg_vecs);
    __syncwarp();
    if (lane < k) s_row[wib][lane] = __ldg(slot_row + static_cast<size_t>(t) * k + lane);
    __syncwarp();
    const uint4* src = reinterpret_cast<const uint4*>(u + static_cast<size_t>(t) * H);
    for (int v = v0 + lane; v < v1; v += 32) {
      const uint4 x = __ldg(src + v);
      for (int j = 0; j < k; ++j) {
        const int r = s_row[wib][j];
        if (r >= 0) reinterpret_cast<uint4*>(u_perm + static_cast<size_t>(r) * H)[v] = x;
      }
    }
  }
}

}  // namespace moe
