// fp32 grouped GEMM on the CUDA cores, for layers stored in fp32 (their
// tolerance, 1e-4 of the output scale, rules out TF32 tensor-core inputs).
//
//   out[c, j] = epi( Σ_k X[c, k] · W[j, k] )   per expert group
//
// with the same group table as the tensor-core path.  64 x 64 output tile per
// 256-thread block, 4 x 4 per thread, K staged through shared memory.
// Also serves the fp32 router logits (one dense group, per-column offset).
#pragma once

#include "common.cuh"

namespace moe {

enum SimtEpi : int { SIMT_SWIGLU = 0, SIMT_RELU = 1, SIMT_PLAIN = 2, SIMT_LOGITS = 3 };

struct SimtParams {
  const float* a[2];        // weight stacks [rows, K]
  const float* a3[2];       // SwiGLU up-projection stacks
  const float* b[2];        // token sources [rows, K]
  float* out[2];
  const GroupDesc* groups;  // or null: one dense group of dense_count rows
  int dense_count;
  int K;
  int n_cols;               // output columns per group
  int out_ld;
  const float* col_offset;  // SIMT_LOGITS: per-column addend, may be null
};

constexpr int kSimtTile = 64;
constexpr int kSimtK = 16;

template <int EPI>
__global__ void __launch_bounds__(256) simt_gemm_kernel(const SimtParams p) {
  constexpr bool kTwo = EPI == SIMT_SWIGLU;
  __shared__ float xs[kSimtK][kSimtTile + 1];
  __shared__ float ws[kSimtK][kSimtTile + 1];
  __shared__ float ws3[kTwo ? kSimtK : 1][kSimtTile + 1];

  GroupDesc d = (p.groups == nullptr) ? GroupDesc{0, 0, 0, 0, 0, 0, p.dense_count, 0}
                                      : p.groups[blockIdx.z];
  const int c0 = blockIdx.y * kSimtTile, j0 = blockIdx.x * kSimtTile;
  if (c0 >= d.count) return;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const float* X = p.b[d.b_src] + static_cast<size_t>(d.b_row0) * p.K;
  const float* Wm = p.a[d.a_sel] + static_cast<size_t>(d.a_row0) * p.K;
  const float* W3 = kTwo ? p.a3[d.a_sel] + static_cast<size_t>(d.a_row0) * p.K : nullptr;

  float acc[4][4] = {}, acc3[4][4] = {};
  for (int k0 = 0; k0 < p.K; k0 += kSimtK) {
    for (int i = threadIdx.x; i < kSimtK * kSimtTile; i += 256) {
      const int r = i / kSimtK, kk = i % kSimtK;
      const bool kin = k0 + kk < p.K;
      xs[kk][r] = (kin && c0 + r < d.count) ? X[static_cast<size_t>(c0 + r) * p.K + k0 + kk] : 0.f;
      const bool jin = kin && j0 + r < p.n_cols;
      ws[kk][r] = jin ? Wm[static_cast<size_t>(j0 + r) * p.K + k0 + kk] : 0.f;
      if (kTwo) ws3[kk][r] = jin ? W3[static_cast<size_t>(j0 + r) * p.K + k0 + kk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kSimtK; ++kk) {
      float xv[4], wv[4], wv3[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xv[i] = xs[kk][ty * 4 + i];
        wv[i] = ws[kk][tx * 4 + i];
        if (kTwo) wv3[i] = ws3[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
          if (kTwo) acc3[i][j] = fmaf(xv[i], wv3[j], acc3[i][j]);
        }
    }
    __syncthreads();
  }
  float* O = p.out[d.out_sel];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = c0 + ty * 4 + i;
    if (c >= d.count) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = j0 + tx * 4 + j;
      if (col >= p.n_cols) continue;
      float v = acc[i][j];
      if (EPI == SIMT_SWIGLU) v = v / (1.0f + expf(-v)) * acc3[i][j];
      if (EPI == SIMT_RELU) v = fmaxf(v, 0.0f);
      if (EPI == SIMT_LOGITS && p.col_offset != nullptr) v += p.col_offset[col];
      O[static_cast<size_t>(d.out_row0 + c) * p.out_ld + col] = v;
    }
  }
}

// Per-group descriptors of the two expert GEMMs and the prefix of token
// tiles (of `bn` rows) per group.  A group is a routed expert on its permuted
// rows, or a piece of `piece` consecutive tokens of a shared expert.  The
// n_pieces pieces of every shared expert are spread evenly between the routed
// experts (pieces of different shared experts alternate), so that tiles whose
// weights stream from HBM and tiles that reuse their weights from L2 run side
// by side all through the launch instead of one kind after the other.  For
// the same reason, with `by_load` (weights read by few token tiles), the
// routed experts are taken by load, alternately from the most and the least
// loaded (ranks by row count, ties to the lower index): largest, smallest,
// second largest, ...
//   GEMM1 (up/gate):  A = w1/w3 stacks, B source 0 = u_perm, 1 = u; out = act
//   GEMM2 (down):     A = w2 stacks,    B source 0 = act;              out 0 =
//                     y_perm, out 1 = y_shared
// act rows: routed rows first (same row numbers as u_perm), then shared
// expert j's T rows at T·k + j·T.  One thread per group, up to 1024 groups.
__global__ void __launch_bounds__(1024) ffn_plan_kernel(const int32_t* __restrict__ offsets,
                                                        int E, int Ks, int T, int Tk, int I,
                                                        int H, int bn, int n_pieces, int piece,
                                                        int by_load,
                                                        GroupDesc* g1, GroupDesc* g2,
                                                        int* tile_prefix) {
  __shared__ int warp_tot[32];
  __shared__ int s_count[1024];
  __shared__ int s_by_rank[1024];
  const int S = Ks * n_pieces;  // shared pieces
  const int g = threadIdx.x, G = E + S;
  if (g < E) s_count[g] = offsets[g + 1] - offsets[g];
  __syncthreads();
  if (by_load && g < E) {
    const int c = s_count[g];
    int rank = 0;
    for (int j = 0; j < E; ++j) rank += (s_count[j] > c) || (s_count[j] == c && j < g);
    s_by_rank[rank] = g;
  }
  __syncthreads();
  int routed = -1, shared_piece = -1;
  if (g < G) {
    const int q = S > 0 ? E / S : 0;  // routed experts before each shared piece
    const int blk = q + 1;
    if (S == 0) routed = g;
    else if (g < S * blk) {
      if (g % blk < q) routed = (g / blk) * q + g % blk;
      else shared_piece = g / blk;
    } else {
      routed = S * q + (g - S * blk);
    }
  }
  int cnt = 0;
  if (routed >= 0) {
    if (by_load) routed = s_by_rank[(routed & 1) ? E - 1 - (routed >> 1) : (routed >> 1)];
    const int b = offsets[routed];
    cnt = offsets[routed + 1] - b;
    g1[g] = GroupDesc{0, routed * I, 0, b, 0, b, cnt, 0};
    g2[g] = GroupDesc{0, routed * H, 0, b, 0, b, cnt, 0};
  } else if (shared_piece >= 0) {
    const int j = shared_piece % Ks, p0 = (shared_piece / Ks) * piece;
    cnt = max(0, min(piece, T - p0));
    g1[g] = GroupDesc{1, j * I, 1, p0, 0, Tk + j * T + p0, cnt, 0};
    g2[g] = GroupDesc{1, j * H, 0, Tk + j * T + p0, 1, j * T + p0, cnt, 0};
  }
  const int nt = (cnt + bn - 1) / bn;
  const int lane = g & 31, w = g >> 5;
  int incl = nt;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  if (w == 0) {
    int s = (lane < (blockDim.x >> 5)) ? warp_tot[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += y;
    }
    warp_tot[lane] = s;
  }
  __syncthreads();
  const int excl = incl - nt + (w > 0 ? warp_tot[w - 1] : 0);
  if (g < G) tile_prefix[g] = excl;
  if (g == G - 1) tile_prefix[G] = excl + nt;
}

}  // namespace moe
