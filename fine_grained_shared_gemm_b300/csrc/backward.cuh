// Kernels of the layer backward (bf16 layers).  The layer is
//   h_t = u_t + Σ_j FFN_j^shared(u_t) + Σ_s g_{t,s} FFN_{idx[t,s]}(u_t)
// (page "02 · 细粒度 MoE：从 Mixtral 到 DeepSeekMoE", §3.1 Eq. 9–15; expert FFN
// as on page "19-deepseek-moe"), differentiated with the chosen experts held
// fixed: the top-k choice is piecewise constant in the logits and the
// selection bias only changes the choice, so neither passes a gradient.
//
// The tensor-core grouped GEMM does the contractions (the input-gradient
// GEMMs read the weights MN-major, in their stored layout; the weight
// gradients read the token rows x, dh and u MN-major, in theirs); the kernels
// here produce its other operands and consume its outputs:
//   row_gate_kernel        each routed row's gate weight
//   relu_backward_kernel   ReLU derivative per row and the gate-scaled
//                          activation, written row-major into a padded row
//                          space (each expert's rows padded with zero rows:
//                          the weight gradients contract over each expert's
//                          own rows), and the per-row <dy, y> for the gate
//                          gradient (for SwiGLU the dm GEMM's epilogue
//                          computes the same)
//   gate_backward_kernel   dL/dz from dL/dg through softmax or the normalised
//                          sigmoid (dz · centroids and dzᵀ · u are grouped
//                          GEMMs too)
//   sum_partials_kernel    adds the contraction ranges' partial sums of
//                          dzᵀ · u in range order
//   grad_combine_kernel    du = dh + Σ shared dx + Σ slot dx + router term
//   wgrad_plan_kernel      padded per-expert segments and the weight-gradient
//                          GEMMs' groups
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "route.cuh"

namespace moe {

// Each expert's token rows start on a multiple of this in the K-major
// (transposed) operands of the weight-gradient GEMMs: one pipeline stage of
// the grouped GEMM (two 64-element k-blocks).
constexpr int kSegAlign = 128;

// ---------------------------------------------------------------- per-row derivative

// For row r of the expert inputs (routed rows [0, Tk), then shared rows) of a
// ReLU layer with a = x W1ᵀ and dm = dh W2 for the row's token (NOT yet
// scaled by the row's gate weight g; g = 1 for shared rows):
//   dh1[r]  = g dm ⊙ [a > 0]
//   g act   with act = ReLU(a)
//   <dm, act> (= dL/dg of the row)
// (A SwiGLU layer gets the same quantities from the dm GEMM's epilogue.)
// One block per 64 rows x 64 features.  dh1 and g act are written row-major
// into the padded row space the weight-gradient and input-gradient GEMMs
// read: each shared expert's T rows padded with zero rows to Tpad, then each
// routed expert's rows padded with zero rows to kSegAlign (dh1p [KA, I],
// gactp [KA, I]; the block's padded rows start at prow0 + blockIdx.x · 64).
// The block's source rows: a run of rows_total rows from row_base (seg_start
// == nullptr; row(j) = row_base + j), or the routed rows by expert segment
// (expert e owns padded rows [seg_start[e], seg_start[e+1]) of the routed
// region and row(j) = offsets[e] + j - seg_start[e] while that is below
// offsets[e+1]); padded rows with no source row are written as zeros.  The
// 64 features' share of <dm, act> goes to dg_part[r · (I / 64) + blockIdx.y]
// (routed rows only), summed later in block order.
__global__ void __launch_bounds__(256) relu_backward_kernel(
    const __nv_bfloat16* __restrict__ a, const __nv_bfloat16* __restrict__ dm,
    const float* __restrict__ row_gate, long long Tk, int I, long long row_base, int rows_total,
    const int32_t* __restrict__ seg_start, const int32_t* __restrict__ offsets, int E,
    __nv_bfloat16* __restrict__ dh1p, __nv_bfloat16* __restrict__ gactp, long long prow0,
    float* __restrict__ dg_part) {
  const int j0 = blockIdx.x * 64;
  const int f0 = blockIdx.y * 64;
  const int nb = I / 64;
  long long row0;
  int valid;
  if (seg_start == nullptr) {
    row0 = row_base + j0;
    valid = max(0, min(64, rows_total - j0));
  } else {
    if (j0 >= seg_start[E]) return;
    int lo = 0, hi = E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (seg_start[mid] <= j0) lo = mid; else hi = mid;
    }
    const int local = j0 - seg_start[lo];
    row0 = offsets[lo] + local;
    valid = max(0, min(64, offsets[lo + 1] - offsets[lo] - local));
  }
  for (int i = threadIdx.x; i < 64 * 8; i += blockDim.x) {   // two (row, 8 features) per thread
    const int r = i >> 3, v = i & 7;
    float da[8], ag[8];
    float dot = 0.0f;
    if (r < valid) {
      const long long R = row0 + r;
      const float g = R < Tk ? __ldg(row_gate + R) : 1.0f;
      const size_t off = static_cast<size_t>(R) * I + f0 + v * 8;
      float fa[8], fd[8];
      Vec16<__nv_bfloat16>::load(a + off, fa);
      Vec16<__nv_bfloat16>::load(dm + off, fd);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float act = fmaxf(fa[q], 0.0f);
        dot = fmaf(fd[q], act, dot);
        da[q] = fa[q] > 0.0f ? g * fd[q] : 0.0f;
        ag[q] = g * act;
      }
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) da[q] = ag[q] = 0.0f;
    }
    const size_t prow = static_cast<size_t>(prow0 + j0 + r);
    Vec16<__nv_bfloat16>::store(dh1p + prow * I + f0 + v * 8, da);
    Vec16<__nv_bfloat16>::store(gactp + prow * I + f0 + v * 8, ag);
    // the row's 8 vectors sit in 8 consecutive lanes: add them in a fixed order
    dot += __shfl_xor_sync(0xffffffffu, dot, 1);
    dot += __shfl_xor_sync(0xffffffffu, dot, 2);
    dot += __shfl_xor_sync(0xffffffffu, dot, 4);
    if (v == 0 && r < valid && row0 + r < Tk)
      dg_part[static_cast<size_t>(row0 + r) * nb + blockIdx.y] = dot;
  }
}

// row_gate[slot_row[i]] = topk_w[i]: the gate weight of each permuted row.
__global__ void __launch_bounds__(256) row_gate_kernel(const int32_t* __restrict__ slot_row,
                                                       const float* __restrict__ topk_w, int n,
                                                       float* __restrict__ row_gate) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int r = slot_row[i];
  if (r >= 0 && r < n) row_gate[r] = topk_w[i];
}

// ---------------------------------------------------------------- gate

// dL/dz for one token per warp from dg[t, s] = Σ_b dg_part[slot_row[t, s], b],
// written in bf16 with row pitch ld (>= E, zeros past E) as the operand of
// the router-gradient GEMMs:
//   softmax (g = s for the chosen): dz_e = s_e (dg_e [e chosen] − Σ_s dg_s g_s)
//   sigmoid (g = s / S over the chosen): dz_e = (dg_e − Σ_s dg_s g_s) / S ·
//            s_e (1 − s_e) for chosen e, 0 otherwise.
// The scores are recomputed from the logits as the router computes them; g
// is the router's output.  NPL logits per lane (expert e = lane + 32 i).
template <int NPL>
__global__ void __launch_bounds__(256) gate_backward_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ idx,
    const float* __restrict__ topk_w, const int32_t* __restrict__ slot_row,
    const float* __restrict__ dg_part, int n_parts, int T, int E, int k, int gate, int ld,
    __nv_bfloat16* __restrict__ dz) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps) {
    const float* z = logits + static_cast<size_t>(t) * E;
    // slot lane < k: its expert, weight and gradient
    int my_e = -1;
    float my_g = 0.0f, my_dg = 0.0f, my_s = 0.0f;
    if (lane < k) {
      const size_t i = static_cast<size_t>(t) * k + lane;
      my_e = idx[i];
      my_g = topk_w[i];
      const float* part = dg_part + static_cast<size_t>(slot_row[i]) * n_parts;
      for (int b = 0; b < n_parts; ++b) my_dg += part[b];   // feature blocks in order
      if (gate != 0) my_s = 1.0f / (1.0f + expf(-__ldg(z + my_e)));
    }
    const float cdot = warp_sum(my_dg * my_g);   // Σ_s dg_s g_s
    float out[NPL];
    if (gate == 0) {
      float key[NPL];
      float m = -CUDART_INF_F;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        key[i] = e < E ? __ldg(z + e) : -CUDART_INF_F;
        m = fmaxf(m, key[i]);
      }
      m = warp_max(m);
      float part = 0.0f;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        out[i] = (lane + 32 * i < E) ? expf(key[i] - m) : 0.0f;
        part += out[i];
      }
      const float denom = warp_sum(part);
      float ds[NPL];
#pragma unroll
      for (int i = 0; i < NPL; ++i) ds[i] = 0.0f;
      for (int s = 0; s < k; ++s) {
        const int e = __shfl_sync(0xffffffffu, my_e, s);
        const float d = __shfl_sync(0xffffffffu, my_dg, s);
#pragma unroll
        for (int i = 0; i < NPL; ++i)
          if (e == lane + 32 * i) ds[i] = d;
      }
#pragma unroll
      for (int i = 0; i < NPL; ++i) out[i] = (out[i] / denom) * (ds[i] - cdot);
    } else {
      const float S = warp_sum(my_s);
#pragma unroll
      for (int i = 0; i < NPL; ++i) out[i] = 0.0f;
      for (int s = 0; s < k; ++s) {
        const int e = __shfl_sync(0xffffffffu, my_e, s);
        const float d = __shfl_sync(0xffffffffu, my_dg, s);
        const float sc = __shfl_sync(0xffffffffu, my_s, s);
        const float v = (d - cdot) / S * (sc * (1.0f - sc));
#pragma unroll
        for (int i = 0; i < NPL; ++i)
          if (e == lane + 32 * i) out[i] = v;
      }
    }
    __nv_bfloat16* o = dz + static_cast<size_t>(t) * ld;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) o[e] = __float2bfloat16_rn(out[i]);
    }
    for (int e = E + lane; e < ld; e += 32) o[e] = __float2bfloat16_rn(0.0f);
  }
}

// ---------------------------------------------------------------- du

// out[i] = Σ_{s<S} part[s · n4 + i] over float4 elements, s in order (a fixed
// summation order, so the result does not depend on scheduling).
__global__ void __launch_bounds__(256) sum_partials_kernel(const float4* __restrict__ part,
                                                           int S, long long n4,
                                                           float4* __restrict__ out) {
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < n4; i += gridDim.x * 256LL) {
    float4 acc = __ldg(part + i);
    for (int sp = 1; sp < S; ++sp) {
      const float4 v = __ldg(part + sp * n4 + i);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    out[i] = acc;
  }
}

// du_t = dh_t + Σ_{j<Ks} dx_shared[j, t] + Σ_{s<k} dx_perm[slot_row[t, s]] + du_router_t,
// fp32 in this order, one rounding to bf16.  The routed rows were computed
// from gate-scaled upstream gradients, so they add with weight 1.
__global__ void __launch_bounds__(256) grad_combine_kernel(
    const __nv_bfloat16* __restrict__ dh, const __nv_bfloat16* __restrict__ dx_perm,
    const __nv_bfloat16* __restrict__ dx_shared, const int32_t* __restrict__ slot_row,
    const float* __restrict__ du_router, int n_tokens, int H, int k, int Ks,
    __nv_bfloat16* __restrict__ du) {
  using V16 = Vec16<__nv_bfloat16>;
  constexpr int V = V16::N;
  constexpr int kVecsPerItem = 128;  // work item: a token's 128-vector stretch
  __shared__ int s_row[8][32];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int nvec = H / V;
  const int per_tok = (nvec + kVecsPerItem - 1) / kVecsPerItem;
  const long long items = static_cast<long long>(n_tokens) * per_tok;
  int t_loaded = -1;
  for (long long it = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; it < items; it += warps) {
    const int t = static_cast<int>(it / per_tok);
    const int v0 = static_cast<int>(it % per_tok) * kVecsPerItem;
    const int v1 = min(nvec, v0 + kVecsPerItem);
    if (t != t_loaded) {
      __syncwarp();
      if (lane < k) s_row[wib][lane] = __ldg(slot_row + static_cast<size_t>(t) * k + lane);
      __syncwarp();
      t_loaded = t;
    }
#pragma unroll 2
    for (int v = v0 + lane; v < v1; v += 32) {
      float acc[V], y[V];
      V16::load(dh + static_cast<size_t>(t) * H + v * V, acc);
      for (int j = 0; j < Ks; ++j) {
        V16::load(dx_shared + (static_cast<size_t>(j) * n_tokens + t) * H + v * V, y);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] += y[i];
      }
      // slots in groups of 8: the group's loads are issued before any is
      // used, then added in slot order
      for (int s0 = 0; s0 < k; s0 += 8) {
        uint4 raw[8];
#pragma unroll
        for (int d = 0; d < 8; ++d) {
          const int row = s0 + d < k ? s_row[wib][s0 + d] : -1;
          raw[d] = row >= 0 ? __ldg(reinterpret_cast<const uint4*>(dx_perm + static_cast<size_t>(row) * H + v * V))
                            : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int d = 0; d < 8; ++d) {
          if (s0 + d >= k || s_row[wib][s0 + d] < 0) continue;
          V16::load(reinterpret_cast<const __nv_bfloat16*>(&raw[d]), y);
#pragma unroll
          for (int i = 0; i < V; ++i) acc[i] += y[i];
        }
      }
      const float4* rr = reinterpret_cast<const float4*>(du_router + static_cast<size_t>(t) * H + v * V);
      const float4 r0 = __ldg(rr), r1 = __ldg(rr + 1);
      acc[0] += r0.x; acc[1] += r0.y; acc[2] += r0.z; acc[3] += r0.w;
      acc[4] += r1.x; acc[5] += r1.y; acc[6] += r1.z; acc[7] += r1.w;
      V16::store(du + static_cast<size_t>(t) * H + v * V, acc);
    }
  }
}

// ---------------------------------------------------------------- plan

// One block.  Per-expert segments of the weight-gradient operands:
// seg_start[e] = Σ_{e' < e} roundup(L_e', kSegAlign) (L = rows of the expert),
// seg_start[E] = the total.  And the two weight-gradient GEMMs' groups, their
// contraction ranges (in rows) and their tile prefixes (nt2 / nt13 token
// tiles per group):
//   dW2 (out[n = h, m = i] over A = g act, B = dh rows):
//     shared j:    g act rows from j·Tpad, dh rows from 0,              Tpad / 64 chunks
//     routed e:    g act rows from Ks·Tpad + seg, d_perm rows from off_e, padded L_e / 64
//   dW1 / dW3 (out[n = i, m = h] over A = x rows, B = dh1, one group per
//   expert and part; part 1 (up) reads dh1 columns I..2I):
//     shared (j, part): u rows from 0, dh1 rows from j·Tpad
//     routed (e, part): x_perm rows from off_e, dh1 rows from Ks·Tpad + seg
// Shared groups come first (their contraction is the longest).  Also the
// input-gradient GEMM's groups (dx_groups): the forward's down-projection
// groups fwd2 with token rows in dh1's padded row space; and the fused
// dm GEMM's groups (dm_groups): the forward's gate/up groups fwd1 with their
// first padded row in GroupDesc.pad.
__global__ void __launch_bounds__(1024) wgrad_plan_kernel(
    const int32_t* __restrict__ offsets, int E, int Ks, int Tpad, int H, int I, int parts,
    int32_t* __restrict__ seg_start, GroupDesc* __restrict__ g2, int4* __restrict__ k2,
    GroupDesc* __restrict__ g13, int4* __restrict__ k13, int nt2, int nt13,
    int* __restrict__ p2, int* __restrict__ p13, const GroupDesc* __restrict__ fwd2, int G,
    int Tk, int T, GroupDesc* __restrict__ dx_groups, const GroupDesc* __restrict__ fwd1,
    GroupDesc* __restrict__ dm_groups) {
  __shared__ int s_seg[1025];
  __shared__ int warp_tot[32];
  const int e = threadIdx.x;
  const int len = e < E ? (offsets[e + 1] - offsets[e] + kSegAlign - 1) / kSegAlign * kSegAlign : 0;
  // block-wide exclusive scan of len
  const int lane = e & 31, w = e >> 5;
  int incl = len;
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
  const int excl = incl - len + (w > 0 ? warp_tot[w - 1] : 0);
  if (e <= E) s_seg[e] = excl;   // thread E holds len 0: its exclusive sum is the total
  __syncthreads();
  if (e <= E) seg_start[e] = s_seg[e];
  // static tile prefixes: every group of a weight-gradient GEMM has the same
  // token-side width
  for (int g = threadIdx.x; g <= E + Ks; g += blockDim.x) p2[g] = g * nt2;
  for (int g = threadIdx.x; g <= (E + Ks) * parts; g += blockDim.x) p13[g] = g * nt13;
  // Every operand is read MN-major from a row-major matrix; krange = {first
  // row of the weight side, first row of the token side, k-chunks}.  g act
  // and dh1 sit in the padded row space (zero rows after each expert's own);
  // x, u, dh and d_perm are the unpadded stored rows: the rows past an
  // expert's own that its padded contraction reaches belong to the next
  // expert (or lie past the matrix) and meet the padding's zeros.
  constexpr int kc = 64;         // elements per k-chunk
  if (e < Ks) {
    // dW2: g act rows of shared expert e, dh rows from 0 (token source 1)
    g2[e] = GroupDesc{0, 0, 1, 0, 1, e * H, H, 0};
    k2[e] = make_int4(e * Tpad, 0, Tpad / kc, 0);
    for (int p = 0; p < parts; ++p) {
      // dW1/dW3: u rows from 0 (weight-side source 1), dh1 rows of expert e
      g13[e * parts + p] = GroupDesc{1, 0, 0, p * I, 2 + p, e * I, I, 0};
      k13[e * parts + p] = make_int4(0, e * Tpad, Tpad / kc, 0);
    }
  }
  if (e < E) {
    const int seg = s_seg[e], n = (s_seg[e + 1] - seg) / kc;
    g2[Ks + e] = GroupDesc{0, 0, 0, 0, 0, e * H, H, 0};
    k2[Ks + e] = make_int4(Ks * Tpad + seg, offsets[e], n, 0);
    for (int p = 0; p < parts; ++p) {
      g13[(Ks + e) * parts + p] = GroupDesc{0, 0, 0, p * I, p, e * I, I, 0};
      k13[(Ks + e) * parts + p] = make_int4(offsets[e], Ks * Tpad + seg, n, 0);
    }
  }
  // the input-gradient GEMM's groups: the forward's down-projection groups
  // with their token rows moved into the padded row space of dh1
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    GroupDesc d = fwd2[g];
    if (d.a_sel == 0) {            // routed expert a_row0 / H, from its first row
      const int ex = d.a_row0 / H;
      d.b_row0 = Ks * Tpad + s_seg[ex] + (d.b_row0 - offsets[ex]);
    } else {                       // shared expert j's piece from token p0
      const int rel = d.b_row0 - Tk, j = rel / T;
      d.b_row0 = j * Tpad + (rel - j * T);
    }
    dx_groups[g] = d;
    // the fused dm GEMM's groups: the forward's gate/up groups (output rows
    // = the rows of a and c), each with its first row in the padded space
    GroupDesc d1 = fwd1[g];
    if (d1.a_sel == 0) {           // routed expert a_row0 / I, from its first row
      const int ex = d1.a_row0 / I;
      d1.pad = Ks * Tpad + s_seg[ex] + (d1.b_row0 - offsets[ex]);
    } else {                       // shared expert j's piece from token b_row0
      d1.pad = (d1.a_row0 / I) * Tpad + d1.b_row0;
    }
    dm_groups[g] = d1;
  }
}

}  // namespace moe
