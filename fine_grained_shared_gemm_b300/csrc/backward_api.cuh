// Host side of the layer backward: workspace layout, the launch sequence of
// moe_layer_backward and its C entry points.  Included by moe_api.cu at the
// point where the forward's host steps (tensor maps, launches, workspace
// carving, the FFN plan) are already defined; not a stand-alone header.
#pragma once

// ---------------------------------------------------------------- backward

// Workspace of the layer backward.  Rall = T·k + Ks·T expert input rows
// (routed rows, then each shared expert's T rows); P = 2 (SwiGLU) or 1 (ReLU)
// pre-activation blocks per row.  The weight-gradient GEMMs' row-major
// operands g act (gactp) and dh1 (dh1p) sit in a padded row space: each
// shared expert's T rows padded to Tpad, then each routed expert's rows
// padded to kSegAlign.  KX is one shared block plus all routed segments, KA
// every shared block plus the routed segments.
struct BwdWs {
  float* logits;
  int32_t* idx;
  float* w;
  int32_t* offsets;
  int32_t* row_token;
  int32_t* slot_row;
  void* dispatch_ws;
  GroupDesc* g1;
  GroupDesc* g2;
  int* tile_prefix;
  __nv_bfloat16 *x_perm, *d_perm;        // [Tk, H]
  __nv_bfloat16 *a, *c, *dm;             // [Rall, I]
  __nv_bfloat16* dh1p;                   // [KA, P·I]: padded row space
  float* row_gate;                       // [Tk]
  float* dg_part;                        // [Tk, I / 32]: <dm, act> per feature block
                                         // (32 features: SwiGLU; 64: ReLU)
  __nv_bfloat16* dz;                     // [T, Epad], zeros past E
  int Epad;                              // E rounded up to 64
  float* du_router;                      // [T, H]
  __nv_bfloat16 *dx_perm, *dx_sh;        // [Tk, H], [Ks·T, H]
  int32_t* seg_start;                    // [E + 1]
  GroupDesc *wg2, *wg13;
  int4 *wk2, *wk13;
  int *wp2, *wp13;
  __nv_bfloat16* gactp;                  // [KA, I]: g act, padded row space
  GroupDesc* dxg;                        // the input-gradient GEMM's groups
  GroupDesc* dmg;                        // the fused dm GEMM's groups (SwiGLU)
  float* dc_part;                        // [dc_splits, E, H]: d_centroids partial sums
  int dc_splits, dc_split_blocks;        // contraction ranges of d_centroids, k-chunks each
  long long Tpad, KX, KA;
  size_t total;
};

// d_centroids = dzᵀ u contracts over all T tokens but has only
// ceil(Epad / 256) · ceil(H / 256) output tiles: the contraction is cut into
// ranges so that about one wave of CTA pairs (kDcTiles tiles) is busy, each
// range's partial sum written apart and the ranges added in order after.
constexpr int kDcTiles = 72;
// The fused dm GEMM runs its derivative epilogue on eight warps up to this
// contraction length (H), on four above (both with three pipeline stages):
// at H = 2048 eight warps take 0.79 ms against 0.93, at H = 7168 both 2.16.
constexpr int kBwdEpi8MaxK = 4096;
constexpr int kDcMaxSplits = 16;

void dcent_splits(const moe_shape* s, long long Tpad, int Epad, int* splits, int* blocks) {
  const int tiles = cdiv(Epad, 256) * cdiv(s->H, 256);
  const int nkb = static_cast<int>(Tpad / tc::kBK);
  int want = std::max(1, std::min({kDcMaxSplits, kDcTiles / tiles, nkb / tc::kKPS}));
  const int per = cdiv(cdiv(nkb, want), tc::kKPS) * tc::kKPS;
  *blocks = std::max(per, tc::kKPS);
  *splits = std::max(1, cdiv(nkb, *blocks));
}

BwdWs carve_bwd(void* ws, const moe_shape* s) {
  const size_t T = s->T, E = s->n_routed, k = s->top_k, Ks = s->n_shared, H = s->H,
               I = s->inter;
  const size_t P = s->act == MOE_ACT_SWIGLU ? 2 : 1;
  const size_t Tk = T * k, Rall = Tk + Ks * T;
  const size_t Tpad = (T + kSegAlign - 1) / kSegAlign * kSegAlign;
  // routed region: every expert's rows padded to kSegAlign; a multiple of
  // kSegAlign itself, so row pitches stay 16-byte multiples and tensor maps
  // cover whole k-chunks
  const size_t Rmax = (Tk + kSegAlign - 1) / kSegAlign * kSegAlign + static_cast<size_t>(kSegAlign) * E;
  char* base = static_cast<char*>(ws);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = base + off;
    off += align256(bytes);
    return static_cast<void*>(p);
  };
  auto bf = [&](size_t n) { return static_cast<__nv_bfloat16*>(take(n * 2)); };
  BwdWs B;
  B.Tpad = static_cast<long long>(Tpad);
  B.KX = static_cast<long long>(Tpad + Rmax);
  B.KA = static_cast<long long>(Ks * Tpad + Rmax);
  B.logits = static_cast<float*>(take(T * E * 4));
  B.idx = static_cast<int32_t*>(take(Tk * 4));
  B.w = static_cast<float*>(take(Tk * 4));
  B.offsets = static_cast<int32_t*>(take((E + 1) * 4));
  B.row_token = static_cast<int32_t*>(take(Tk * 4));
  B.slot_row = static_cast<int32_t*>(take(Tk * 4));
  B.dispatch_ws = take(dispatch_ws_bytes(s));
  const size_t G = ffn_groups(s);
  B.g1 = static_cast<GroupDesc*>(take(G * sizeof(GroupDesc)));
  B.g2 = static_cast<GroupDesc*>(take(G * sizeof(GroupDesc)));
  B.tile_prefix = static_cast<int*>(take((G + 1) * 4));
  B.x_perm = bf(Tk * H);
  B.d_perm = bf(Tk * H);
  B.a = bf(Rall * I);
  B.c = P == 2 ? bf(Rall * I) : nullptr;
  B.dm = P == 2 ? nullptr : bf(Rall * I);   // SwiGLU: dm stays in the GEMM's accumulator

  B.row_gate = static_cast<float*>(take(Tk * 4));
  B.dg_part = static_cast<float*>(take(Tk * (I / 32) * 4));
  B.Epad = static_cast<int>((E + tc::kBK - 1) / tc::kBK * tc::kBK);
  B.dz = bf(T * static_cast<size_t>(B.Epad));
  B.du_router = static_cast<float*>(take(T * H * 4));
  B.dx_perm = bf(Tk * H);
  B.dx_sh = bf(Ks * T * H);
  B.seg_start = static_cast<int32_t*>(take((E + 1) * 4));
  const size_t G2 = E + Ks, G13 = (E + Ks) * P;
  B.wg2 = static_cast<GroupDesc*>(take(G2 * sizeof(GroupDesc)));
  B.wk2 = static_cast<int4*>(take(G2 * sizeof(int4)));
  B.wp2 = static_cast<int*>(take((G2 + 1) * 4));
  B.wg13 = static_cast<GroupDesc*>(take(G13 * sizeof(GroupDesc)));
  B.wk13 = static_cast<int4*>(take(G13 * sizeof(int4)));
  B.wp13 = static_cast<int*>(take((G13 + 1) * 4));
  B.dh1p = bf(P * I * static_cast<size_t>(B.KA));
  B.gactp = bf(I * static_cast<size_t>(B.KA));
  B.dxg = static_cast<GroupDesc*>(take(G * sizeof(GroupDesc)));
  B.dmg = static_cast<GroupDesc*>(take(G * sizeof(GroupDesc)));
  dcent_splits(s, B.Tpad, B.Epad, &B.dc_splits, &B.dc_split_blocks);
  B.dc_part = static_cast<float*>(take(static_cast<size_t>(B.dc_splits) * E * H * 4));
  B.total = off;
  return B;
}

moe_status check_backward(const moe_shape* s) {
  MOE_TRY(check_shape(s));
  if (s->dtype != MOE_DTYPE_BF16 || s->inter % 128 != 0) return MOE_ERR_UNSUPPORTED;
  const int P = s->act == MOE_ACT_SWIGLU ? 2 : 1;
  if ((s->n_routed + s->n_shared) * P > tc::kMaxGroups) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

MOE_API size_t moe_layer_backward_workspace_size(const moe_shape* s) {
  return check_backward(s) == MOE_OK ? carve_bwd(nullptr, s).total : 0;
}

moe_status layer_backward(const moe_shape* s, const moe_weights* wt, const void* u,
                          const void* dh, void* du, const moe_weight_grads* gr,
                          const void* saved, size_t saved_bytes, void* ws, size_t ws_bytes,
                          cudaStream_t st) {
  MOE_TRY(check_backward(s));
  MOE_TRY(check_weights_ffn(s, wt));
  if (!ok_ptr(wt->centroids) || !ok_opt(wt->logit_offset) || !ok_opt(wt->select_bias))
    return MOE_ERR_INVALID_ARG;
  const bool swiglu = s->act == MOE_ACT_SWIGLU;
  const int T = s->T, E = s->n_routed, Ks = s->n_shared, k = s->top_k, H = s->H, I = s->inter;
  const int P = swiglu ? 2 : 1;
  if (gr == nullptr || !ok_ptr(gr->d_centroids) || !ok_ptr(gr->dw1) || !ok_ptr(gr->dw2) ||
      (swiglu && !ok_ptr(gr->dw3)))
    return MOE_ERR_INVALID_ARG;
  if (Ks > 0 && (!ok_ptr(gr->dsw1) || !ok_ptr(gr->dsw2) || (swiglu && !ok_ptr(gr->dsw3))))
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!ok_ptr(u) || !ok_ptr(dh) || !ok_ptr(du))) return MOE_ERR_INVALID_ARG;
  if (saved != nullptr && (!al16(saved) || saved_bytes < carve_saved(nullptr, s).total))
    return MOE_ERR_INVALID_ARG;
  BwdWs B = carve_bwd(nullptr, s);
  if (ws == nullptr || !al16(ws) || ws_bytes < B.total) return MOE_ERR_WORKSPACE;
  B = carve_bwd(ws, s);
  if (saved != nullptr) {  // the forward's routing, permuted rows and pre-activations
    SavedLayout S = carve_saved(const_cast<void*>(saved), s);
    B.logits = S.logits;
    B.idx = S.idx;
    B.w = S.w;
    B.offsets = S.offsets;
    B.row_token = S.row_token;
    B.slot_row = S.slot_row;
    B.x_perm = static_cast<__nv_bfloat16*>(S.x_perm);
    B.a = static_cast<__nv_bfloat16*>(S.a);
    B.c = static_cast<__nv_bfloat16*>(S.c);
  }
  const size_t wsz = static_cast<size_t>(I) * H * 4;
  if (T == 0) {  // no tokens: every gradient is zero
    MOE_CUDA(cudaMemsetAsync(gr->d_centroids, 0, static_cast<size_t>(E) * H * 4, st));
    MOE_CUDA(cudaMemsetAsync(gr->dw1, 0, E * wsz, st));
    MOE_CUDA(cudaMemsetAsync(gr->dw2, 0, E * wsz, st));
    if (swiglu) MOE_CUDA(cudaMemsetAsync(gr->dw3, 0, E * wsz, st));
    if (Ks > 0) {
      MOE_CUDA(cudaMemsetAsync(gr->dsw1, 0, Ks * wsz, st));
      MOE_CUDA(cudaMemsetAsync(gr->dsw2, 0, Ks * wsz, st));
      if (swiglu) MOE_CUDA(cudaMemsetAsync(gr->dsw3, 0, Ks * wsz, st));
    }
    return MOE_OK;
  }
  const int Tk = T * k;
  const long long Rall = static_cast<long long>(Tk) + static_cast<long long>(Ks) * T;
  const int Epad = B.Epad;

  // ---- the forward's routing, recomputed unless saved
  if (saved == nullptr) {
    const float* bias = s->gate == MOE_GATE_SIGMOID_BIAS ? wt->select_bias : nullptr;
    MOE_TRY(do_router_logits(s, u, wt->centroids, wt->logit_offset, B.logits, nullptr, st));
    MOE_TRY(do_route(s, B.logits, bias, B.idx, B.w, nullptr, st));
    MOE_TRY(do_dispatch(s, B.idx, u, B.offsets, B.row_token, B.slot_row, B.x_perm,
                        B.dispatch_ws, st));
  }
  if (Tk > 0) {
    const RowSplit rs = row_split(T, H / 8, 16);
    scatter_token_rows<__nv_bfloat16><<<rs.blocks, 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(dh), T, s->top_k, B.slot_row, H, rs.nseg,
        rs.seg_vecs, B.d_perm);
    MOE_CUDA(cudaGetLastError());
    row_gate_kernel<<<cdiv(Tk, 256), 256, 0, st>>>(B.slot_row, B.w, Tk, B.row_gate);
    MOE_CUDA(cudaGetLastError());
  }
  const int bn = ffn_bn(s);
  const int pair = bn == 256 ? 2 : 1;
  const int G = static_cast<int>(ffn_groups(s));
  const int by_load = static_cast<long long>(Tk) <= 2LL * bn * E ? 1 : 0;
  ffn_plan_kernel<<<1, cdiv(G, 32) * 32, 0, st>>>(B.offsets, E, Ks, T, Tk, I, H, bn,
                                                   shared_pieces(s), shared_piece_rows(s),
                                                   by_load, B.g1, B.g2, B.tile_prefix);
  MOE_CUDA(cudaGetLastError());
  // per-expert segments of the weight gradients' K-major operands and the
  // weight-gradient GEMMs' groups
  const int nt2 = cdiv(H, 256), nt13 = cdiv(I, 256);
  wgrad_plan_kernel<<<1, 1024, 0, st>>>(B.offsets, E, Ks, static_cast<int>(B.Tpad), H, I, P,
                                        B.seg_start, B.wg2, B.wk2, B.wg13, B.wk13, nt2, nt13,
                                        B.wp2, B.wp13, B.g2, G, Tk, T, B.dxg, B.g1, B.dmg);
  MOE_CUDA(cudaGetLastError());
  const int rmax = static_cast<int>(B.KX - B.Tpad);
  const long long tpad = B.Tpad, sh = static_cast<long long>(Ks) * B.Tpad;

  const long long PI = static_cast<long long>(P) * I;
  if (Rall > 0) {
  // ---- grouped GEMMs over the forward's groups: pre-activations and dm = dh W2
  // mn: the weights are stored as the operand's transpose ([K rows, M
  // columns] per expert) and read MN-major
  auto row_gemm = [&](const void* wr, const void* wsh, uint64_t rows_per_expert, int K, bool mn,
                      const void* b_routed, const void* b_shared, int b_shared_rows,
                      const GroupDesc* groups, void* out0, uint64_t out0_rows, void* out1,
                      uint64_t out1_rows, int out_cols) -> moe_status {
    tc::Params p;
    memset(&p, 0, sizeof(p));
    if (mn) {
      MOE_TRY(make_map3_mn(&p.a[0], wr, static_cast<uint64_t>(E) * K, rows_per_expert));
      if (Ks) MOE_TRY(make_map3_mn(&p.a[1], wsh, static_cast<uint64_t>(Ks) * K, rows_per_expert));
      else p.a[1] = p.a[0];
      p.a_mn = 1;
      p.a_mn_per_expert = static_cast<int>(rows_per_expert);
      p.a_k_per_expert = K;
    } else {
      MOE_TRY(make_map3(&p.a[0], wr, static_cast<uint64_t>(E) * rows_per_expert, K, tc::kBM));
      if (Ks) MOE_TRY(make_map3(&p.a[1], wsh, static_cast<uint64_t>(Ks) * rows_per_expert, K, tc::kBM));
      else p.a[1] = p.a[0];
    }
    MOE_TRY(make_token_maps(p.b[1], b_shared, b_shared_rows, K));
    if (b_routed != nullptr) MOE_TRY(make_token_maps(p.b[0], b_routed, Tk, K));
    else memcpy(p.b[0], p.b[1], sizeof(p.b[0]));
    p.groups = groups;
    p.tile_prefix = B.tile_prefix;
    p.n_groups = G;
    p.n_wtiles = cdiv(static_cast<int>(rows_per_expert), tc::kBM * pair);
    p.num_k_blocks = cdiv(K, tc::kBK);
    p.out[0] = out0;
    p.out[1] = out1;
    MOE_TRY(make_out_map(&p.omap[0], out0, out0_rows, out_cols));
    MOE_TRY(make_out_map(&p.omap[1], out1, out1_rows, out_cols));
    p.out_ld = out_cols;
    p.out_cols = out_cols;
    return launch_ffn<tc::EPI_BF16>(p, bn, st);
  };
  const void* xr = Tk > 0 ? B.x_perm : nullptr;
  const void* dr = Tk > 0 ? B.d_perm : nullptr;
  if (saved == nullptr) {  // pre-activations, recomputed
    MOE_TRY(row_gemm(wt->w1, wt->sw1, I, H, false, xr, u, T, B.g1, B.a, Rall, B.a, Rall, I));
    if (swiglu)
      MOE_TRY(row_gemm(wt->w3, wt->sw3, I, H, false, xr, u, T, B.g1, B.c, Rall, B.c, Rall, I));
  }
  if (swiglu) {
    // dm = dh W2 (W2 [H, I] per expert is the operand's transpose, read
    // MN-major) with the SwiGLU derivative in the epilogue: da | dc into
    // dh1p, g act into gactp (padded row space, zero padding rows), <dm, act>
    // per routed row and 32-feature block into dg_part; a and c come in by TMA
    tc::Params p;
    memset(&p, 0, sizeof(p));
    MOE_TRY(make_map3_mn(&p.a[0], wt->w2, static_cast<uint64_t>(E) * H, I));
    if (Ks) MOE_TRY(make_map3_mn(&p.a[1], wt->sw2, static_cast<uint64_t>(Ks) * H, I));
    else p.a[1] = p.a[0];
    p.a_mn = 1;
    p.a_mn_per_expert = I;
    p.a_k_per_expert = H;
    MOE_TRY(make_token_maps(p.b[1], dh, T, H));
    if (dr != nullptr) MOE_TRY(make_token_maps(p.b[0], dr, Tk, H));
    else memcpy(p.b[0], p.b[1], sizeof(p.b[0]));
    p.groups = B.dmg;
    p.tile_prefix = B.tile_prefix;
    p.n_groups = G;
    p.n_wtiles = cdiv(I, tc::kBM * pair);
    p.num_k_blocks = cdiv(H, tc::kBK);
    p.out_cols = I;
    p.out_ld = I;
    p.out[0] = B.dh1p;
    p.out[1] = B.gactp;
    // a and c in boxes of 32 columns x 16 rows (half an epilogue chunk)
    MOE_TRY(make_out_map(&p.bwd_map[0], B.a, static_cast<uint64_t>(Rall), I, 16));
    MOE_TRY(make_out_map(&p.bwd_map[1], B.c, static_cast<uint64_t>(Rall), I, 16));
    p.bwd_gate = B.row_gate;
    p.bwd_dg = B.dg_part;
    p.bwd_routed_rows = Tk;
    p.pad_rows = kSegAlign;
    // eight epilogue warps when the contraction is short enough for the
    // epilogue to set the pace
    if (H <= kBwdEpi8MaxK) MOE_TRY(launch_ffn<tc::EPI_SWIGLU_BWD8>(p, bn, st));
    else MOE_TRY(launch_ffn<tc::EPI_SWIGLU_BWD>(p, bn, st));
  } else {
  // dm = dh W2: W2 [H, I] per expert is the operand's transpose
  MOE_TRY(row_gemm(wt->w2, wt->sw2, I, H, true, dr, dh, T, B.g1, B.dm, Rall, B.dm, Rall, I));

  // ---- ReLU derivative and gate-scaled activation into the padded row
  // space, <dm, act> per routed row and 64-feature block
  {
    auto act_bwd = [&](dim3 grid, long long row_base, int rows_total, const int32_t* seg,
                       long long col0) -> moe_status {
      relu_backward_kernel<<<grid, 256, 0, st>>>(B.a, B.dm, B.row_gate, Tk, I, row_base,
                                                 rows_total, seg, B.offsets, E, B.dh1p,
                                                 B.gactp, col0, B.dg_part);
      MOE_CUDA(cudaGetLastError());
      return MOE_OK;
    };
    for (int j = 0; j < Ks; ++j)
      MOE_TRY(act_bwd(dim3(static_cast<unsigned>(tpad / 64), I / 64), Tk + static_cast<long long>(j) * T,
                      T, nullptr, j * tpad));
    if (Tk > 0)
      MOE_TRY(act_bwd(dim3(static_cast<unsigned>(cdiv(rmax, 64)), I / 64), 0, 0, B.seg_start, sh));
  }
  }  // ReLU

  }  // Rall > 0
  // ---- gate gradient and the router's share of du and of the centroids
  {
    const int blocks = route_blocks(T);
    const int npl = cdiv(E, 32);
    const int gate = s->gate == MOE_GATE_SOFTMAX ? 0 : 1;
#define MOE_GATE_BWD(N)                                                                 \
  gate_backward_kernel<N><<<blocks, 256, 0, st>>>(B.logits, B.idx, B.w, B.slot_row, B.dg_part, \
                                                  swiglu ? I / 32 : I / 64, T, E, k, gate,  \
                                                  Epad, B.dz)
    if (npl <= 1) MOE_GATE_BWD(1);
    else if (npl <= 2) MOE_GATE_BWD(2);
    else if (npl <= 4) MOE_GATE_BWD(4);
    else if (npl <= 8) MOE_GATE_BWD(8);
    else if (npl <= 16) MOE_GATE_BWD(16);
    else MOE_GATE_BWD(32);
#undef MOE_GATE_BWD
    MOE_CUDA(cudaGetLastError());
    // du += dz · centroids: the centroids [E, H] are the operand's transpose
    // (read MN-major), dz is the token operand, K = E (padded to Epad)
    tc::Params p;
    memset(&p, 0, sizeof(p));
    MOE_TRY(make_map3_mn(&p.a[0], wt->centroids, E, H));
    p.a[1] = p.a[0];
    p.a_mn = 1;
    p.a_mn_per_expert = H;
    p.a_k_per_expert = E;
    MOE_TRY(make_token_maps(p.b[0], B.dz, T, Epad));
    memcpy(p.b[1], p.b[0], sizeof(p.b[0]));
    p.dense_count = T;
    p.n_wtiles = cdiv(H, 256);
    p.num_k_blocks = Epad / tc::kBK;
    p.out[0] = p.out[1] = B.du_router;
    p.out_ld = H;
    p.out_cols = H;
    p.f32_tma = 1;
    MOE_TRY(make_out_map_f32(&p.omap32[0], B.du_router, T, H));
    p.omap32[1] = p.omap32[0];
    MOE_TRY((launch_tc<tc::EPI_F32, 256, 2>(p, INT_MAX, st)));
    // d_centroids = dzᵀ u: dz [T, Epad] read MN-major (M = experts), u [T, H]
    // read MN-major (N = H; K = T, rows past T zero-filled); stored
    // transposed into [E, H]
    tc::Params q;
    memset(&q, 0, sizeof(q));
    MOE_TRY(make_map3_mn(&q.a[0], B.dz, T, Epad));
    q.a[1] = q.a[0];
    q.a_mn = 1;
    q.a_mn_per_expert = Epad;
    q.a_k_per_expert = T;
    MOE_TRY(make_map3_mn(&q.b[0][0], u, T, H));
    q.b[1][0] = q.b[0][0];
    q.b_mn = 1;
    q.dense_count = H;
    q.n_wtiles = cdiv(Epad, 256);
    q.num_k_blocks = static_cast<int>(B.Tpad / tc::kBK);
    q.k_splits = B.dc_splits;
    q.k_split_blocks = B.dc_split_blocks;
    q.split_stride = static_cast<long long>(E) * H;
    q.out[0] = q.out[1] = B.dc_part;
    q.out_ld = H;
    q.out_cols = E;
    q.out_tr = 1;
    MOE_TRY((launch_tc<tc::EPI_F32, 256, 2>(q, INT_MAX, st)));
    // the ranges' partial sums, added in range order
    const long long n4 = static_cast<long long>(E) * H / 4;
    const int sp_blocks = static_cast<int>(
        std::min<long long>(one_wave_blocks(sum_partials_kernel, 256), (n4 + 255) / 256));
    if (sp_blocks <= 0) return cuda_fail(cudaErrorInvalidConfiguration);
    sum_partials_kernel<<<sp_blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(B.dc_part),
                                                   B.dc_splits, n4,
                                                   reinterpret_cast<float4*>(gr->d_centroids));
    MOE_CUDA(cudaGetLastError());
  }

  // ---- dx = dh1 [W1; W3] per expert row, then du
  if (Rall > 0) {
    // dx = [da | dc] [W1; W3]: W1 and W3 [I, H] per expert are the operand's
    // transpose, read MN-major, W1's k-chunks first
    tc::Params p;
    memset(&p, 0, sizeof(p));
    p.a_mn_per_expert = H;
    p.a_k_per_expert = I;
    if (swiglu) {
      p.a_mn = 2;
      p.a_stack_chunks = I / tc::kBK;
      MOE_TRY(make_map4_mn_pair(&p.a[0], wt->w1, wt->w3, static_cast<uint64_t>(E) * I, H,
                                &p.a_stack_swap[0]));
      if (Ks)
        MOE_TRY(make_map4_mn_pair(&p.a[1], wt->sw1, wt->sw3, static_cast<uint64_t>(Ks) * I, H,
                                  &p.a_stack_swap[1]));
      else {
        p.a[1] = p.a[0];
        p.a_stack_swap[1] = p.a_stack_swap[0];
      }
    } else {
      p.a_mn = 1;
      MOE_TRY(make_map3_mn(&p.a[0], wt->w1, static_cast<uint64_t>(E) * I, H));
      if (Ks) MOE_TRY(make_map3_mn(&p.a[1], wt->sw1, static_cast<uint64_t>(Ks) * I, H));
      else p.a[1] = p.a[0];
    }
    MOE_TRY(make_token_maps(p.b[0], B.dh1p, B.KA, PI));
    memcpy(p.b[1], p.b[0], sizeof(p.b[0]));
    p.groups = B.dxg;
    p.tile_prefix = B.tile_prefix;
    p.n_groups = G;
    p.n_wtiles = cdiv(H, tc::kBM * pair);
    p.num_k_blocks = static_cast<int>(PI / tc::kBK);
    void* o0 = Tk ? static_cast<void*>(B.dx_perm) : static_cast<void*>(B.dx_sh);
    void* o1 = Ks ? static_cast<void*>(B.dx_sh) : static_cast<void*>(B.dx_perm);
    p.out[0] = o0;
    p.out[1] = o1;
    MOE_TRY(make_out_map(&p.omap[0], o0, Tk ? Tk : static_cast<uint64_t>(Ks) * T, H));
    MOE_TRY(make_out_map(&p.omap[1], o1, Ks ? static_cast<uint64_t>(Ks) * T : Tk, H));
    p.out_ld = H;
    p.out_cols = H;
    MOE_TRY(launch_ffn<tc::EPI_BF16>(p, bn, st));
  }
  const int gc_blocks = one_wave_blocks(grad_combine_kernel, 256);
  if (gc_blocks <= 0) return cuda_fail(cudaErrorInvalidConfiguration);
  grad_combine_kernel<<<gc_blocks, 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(dh), B.dx_perm, B.dx_sh, B.slot_row, B.du_router, T, H,
      k, Ks, static_cast<__nv_bfloat16*>(du));
  MOE_CUDA(cudaGetLastError());

  // ---- weight gradients: contractions over each expert's own rows; the
  // row-major operands (dh and x rows) are read MN-major where they are.
  // The shared experts' groups come first and contract over Tpad rows, the
  // routed ones over about T·k/E: the two-class tile order (long tiles
  // dealt first, the clusters that drew one more of them taking fewer of the
  // rest) keeps every cluster's work about even.
  auto wgrad_order = [&](tc::Params& p, int tiles_per_group, int long_groups) -> moe_status {
    if (long_groups == 0) return MOE_OK;
    int grid = 0;
    MOE_TRY((tc_grid<tc::EPI_F32, 256, 2>(&grid)));
    const int clusters = std::max(1, grid / 2);
    const int nh = long_groups * tiles_per_group;
    const int nl = (p.n_groups - long_groups) * tiles_per_group;
    const int r = nh % clusters;
    // a tile's cost in k-chunks, plus about four for its epilogue
    const double c_long = static_cast<double>(B.Tpad) / tc::kBK + 4.0;
    const double c_short = (E > 0 ? static_cast<double>(Tk) / E : 0.0) / tc::kBK + 1.0 + 4.0;
    const int D = r ? static_cast<int>(std::lround(c_long / c_short)) : 0;
    p.sched_heavy = nh;
    p.sched_qb = std::max(0, cdiv(std::max(0, nl - D * (clusters - r)), clusters));
    return MOE_OK;
  };
  {  // dW2[e][h][i] = Σ_r dh_r[h] · (g act)_r[i]
    tc::Params p;
    memset(&p, 0, sizeof(p));
    MOE_TRY(make_map3_mn(&p.a[0], B.gactp, B.KA, I));
    p.a[1] = p.a[0];
    p.a_mn = 1;
    p.a_k_rows = 1;
    p.a_mn_per_expert = I;   // every group's M range starts at 0: no per-expert offset
    p.a_k_per_expert = 0;
    MOE_TRY(make_map3_mn(&p.b[1][0], dh, T, H));
    if (Tk > 0) MOE_TRY(make_map3_mn(&p.b[0][0], B.d_perm, Tk, H));
    else p.b[0][0] = p.b[1][0];
    p.b_mn = 1;
    p.b_k_rows = 1;
    p.groups = B.wg2;
    p.tile_prefix = B.wp2;
    p.krange = B.wk2;
    p.n_groups = E + Ks;
    p.n_wtiles = cdiv(I, 256);
    p.out[0] = gr->dw2;
    p.out[1] = Ks ? gr->dsw2 : gr->dw2;
    p.out_ld = I;
    p.out_cols = I;
    p.f32_tma = 1;
    MOE_TRY(make_out_map_f32(&p.omap32[0], p.out[0], static_cast<uint64_t>(E) * H, I));
    MOE_TRY(make_out_map_f32(&p.omap32[1], p.out[1],
                             static_cast<uint64_t>(Ks ? Ks : E) * H, I));
    MOE_TRY(wgrad_order(p, p.n_wtiles * nt2, Ks));
    MOE_TRY((launch_tc<tc::EPI_F32, 256, 2>(p, INT_MAX, st)));
  }
  {  // dW1[e][i][h] = Σ_r da_r[i] · x_r[h], dW3 likewise with dc
    tc::Params p;
    memset(&p, 0, sizeof(p));
    MOE_TRY(make_map3_mn(&p.a[1], u, T, H));
    if (Tk > 0) MOE_TRY(make_map3_mn(&p.a[0], B.x_perm, Tk, H));
    else p.a[0] = p.a[1];
    p.a_mn = 1;
    p.a_k_rows = 1;
    p.a_mn_per_expert = H;   // every group's M range starts at 0: expert 0, no k offset
    p.a_k_per_expert = 0;
    MOE_TRY(make_map3_mn(&p.b[0][0], B.dh1p, B.KA, PI));
    p.b[1][0] = p.b[0][0];
    p.b_mn = 1;
    p.b_k_rows = 1;
    p.groups = B.wg13;
    p.tile_prefix = B.wp13;
    p.krange = B.wk13;
    p.n_groups = (E + Ks) * P;
    p.n_wtiles = cdiv(H, 256);
    p.out[0] = gr->dw1;
    p.out[1] = swiglu ? gr->dw3 : gr->dw1;
    p.out[2] = Ks ? gr->dsw1 : gr->dw1;
    p.out[3] = (Ks && swiglu) ? gr->dsw3 : gr->dw1;
    p.out_ld = H;
    p.out_cols = H;
    p.f32_tma = 1;
    for (int o = 0; o < 4; ++o) {
      const bool sh = o >= 2 && Ks;  // out[2], out[3] are the shared stacks when Ks > 0
      MOE_TRY(make_out_map_f32(&p.omap32[o], p.out[o],
                               static_cast<uint64_t>(sh ? Ks : E) * I, H));
    }
    MOE_TRY(wgrad_order(p, p.n_wtiles * nt13, Ks * P));
    MOE_TRY((launch_tc<tc::EPI_F32, 256, 2>(p, INT_MAX, st)));
  }
  return MOE_OK;
}

MOE_API moe_status moe_layer_backward(const moe_shape* s, const moe_weights* weights,
                                      const void* u, const void* dh, void* du,
                                      const moe_weight_grads* grads, const void* saved,
                                      size_t saved_bytes, void* ws, size_t ws_bytes,
                                      moe_stream_t stream) {
  return layer_backward(s, weights, u, dh, du, grads, saved, saved_bytes, ws, ws_bytes,
                        cs(stream));
}
