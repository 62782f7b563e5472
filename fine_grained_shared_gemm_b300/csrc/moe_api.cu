// C-ABI entry points of the MoE layer forward (declared in include/moe.h).
//
// Host side only: argument checks, scratch carving, TMA tensor maps and the
// launches of the kernels in the headers included below.  Nothing here
// allocates device memory; every launch goes to the caller's stream.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <string.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <mutex>

#include "moe.h"

#include "backward.cuh"
#include "balance.cuh"
#include "combine.cuh"
#include "common.cuh"
#include "dispatch.cuh"
#include "expert_parallel.cuh"
#include "route.cuh"
#include "simt_gemm.cuh"
#include "tc_gemm.cuh"

using namespace moe;

namespace {

thread_local int t_last_cuda_error = 0;

moe_status cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return MOE_ERR_CUDA;
}

#define MOE_CUDA(call)                                \
  do {                                                \
    cudaError_t e_ = (call);                          \
    if (e_ != cudaSuccess) return cuda_fail(e_);      \
  } while (0)

#define MOE_TRY(call)                                 \
  do {                                                \
    moe_status s_ = (call);                           \
    if (s_ != MOE_OK) return s_;                      \
  } while (0)

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
inline int cdiv(int a, int b) { return (a + b - 1) / b; }
inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t elt_bytes(const moe_shape* s) { return s->dtype == MOE_DTYPE_F32 ? 4 : 2; }
inline cudaStream_t cs(moe_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

moe_status check_shape(const moe_shape* s) {
  if (s == nullptr) return MOE_ERR_INVALID_ARG;
  if (s->T < 0 || s->H <= 0 || s->n_routed < 1 || s->n_shared < 0 || s->top_k < 0 ||
      s->inter <= 0 || s->top_k > s->n_routed)
    return MOE_ERR_INVALID_ARG;
  if (s->gate != MOE_GATE_SOFTMAX && s->gate != MOE_GATE_SIGMOID_BIAS) return MOE_ERR_INVALID_ARG;
  if (s->act != MOE_ACT_RELU && s->act != MOE_ACT_SWIGLU) return MOE_ERR_INVALID_ARG;
  if (s->dtype != MOE_DTYPE_F32 && s->dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
  if (s->n_routed + s->n_shared > 1024 || s->top_k > 32) return MOE_ERR_UNSUPPORTED;
  if (s->n_groups < 0 || s->topk_groups < 0) return MOE_ERR_INVALID_ARG;
  if (s->n_groups > 0) {
    if (s->n_groups > 32) return MOE_ERR_UNSUPPORTED;
    if (s->n_routed % s->n_groups != 0 || s->topk_groups < 1 || s->topk_groups > s->n_groups ||
        s->topk_groups * (s->n_routed / s->n_groups) < s->top_k)
      return MOE_ERR_INVALID_ARG;
  } else if (s->topk_groups != 0) {
    return MOE_ERR_INVALID_ARG;
  }
  if (s->H % 8 != 0 || s->inter % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (s->dtype == MOE_DTYPE_BF16) {
    if (s->H % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (s->inter % (s->act == MOE_ACT_SWIGLU ? 64 : 128) != 0) return MOE_ERR_UNSUPPORTED;
  }
  const long long rows = static_cast<long long>(s->T) * (s->top_k + s->n_shared);
  if (rows > INT_MAX / 2) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(s->n_routed + s->n_shared) * s->inter > INT_MAX / 2 ||
      static_cast<long long>(s->n_routed + s->n_shared) * s->H > INT_MAX / 2)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

// ---------------------------------------------------------------- TMA maps

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

moe_status encode(CUtensorMap* m, int rank, const void* base, const cuuint64_t* dims,
                  const cuuint64_t* strides, const cuuint32_t* box,
                  CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B,
                  CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return cuda_fail(cudaErrorNotSupported);
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(m, dtype, rank, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : cuda_fail(cudaErrorInvalidValue);
}

// bf16 [rows, cols] row-major (cols % 64 == 0) viewed as (64 columns, rows,
// cols / 64 chunks): a box of box_rows rows x tc::kKPS chunks lands the
// chunks one after the other, each box_rows x 128 bytes, 128-byte swizzled.
// Chunks past the end are zero-filled.
moe_status make_map3(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                     uint32_t box_rows) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(tc::kBK), rows, cols / tc::kBK};
  const cuuint64_t strides[2] = {cols * 2, tc::kBK * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(tc::kBK), box_rows, tc::kKPS};
  return encode(m, 3, base, dims, strides, box);
}

// A weight stack bf16 [rows, cols] row-major read MN-major (the operand is its
// transpose): (64 columns, rows, cols / 64 column blocks), box 64 columns x
// kKPS·64 rows x 2 column blocks, landing [block][row][64] (two slabs).
moe_status make_map3_mn(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(tc::kBK), rows, cols / tc::kBK};
  const cuuint64_t strides[2] = {cols * 2, tc::kBK * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(tc::kBK), tc::kKPS * tc::kBK, 2};
  return encode(m, 3, base, dims, strides, box);
}

// Two stacks w1, w3 (bf16 [rows, cols] each) read MN-major one after the
// other along k: (64 columns, rows, 2 stacks, cols / 64 blocks), the stack
// dimension stepping between the two allocations (< 2^40 bytes apart).
// *swap: the lower-addressed allocation (the map's first stack) is w3.
moe_status make_map4_mn_pair(CUtensorMap* m, const void* w1, const void* w3, uint64_t rows,
                             uint64_t cols, int* swap) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(w1), b = reinterpret_cast<uintptr_t>(w3);
  *swap = b < a;
  const uintptr_t gap = b < a ? a - b : b - a;
  if (gap == 0 || gap >= (static_cast<uintptr_t>(1) << 40)) return MOE_ERR_UNSUPPORTED;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(tc::kBK), rows, 2, cols / tc::kBK};
  const cuuint64_t strides[3] = {cols * 2, static_cast<cuuint64_t>(gap), tc::kBK * 2};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(tc::kBK), tc::kKPS * tc::kBK, 1, 2};
  return encode(m, 4, b < a ? w3 : w1, dims, strides, box);
}

// SwiGLU gate and up stacks w1, w3 (both bf16 [rows, cols], rows % 64 == 0)
// as one 5-D tensor (64 columns, 64 rows, {first, second} stack, 64-row
// blocks, cols / 64 chunks) whose third dimension steps between the two
// allocations.  One box lands, for each of tc::kKPS chunks, 64 rows of the
// lower-addressed stack then the same 64 rows of the other: *up_first says
// whether that is W3.  The two allocations must be less than 2^40 bytes apart.
moe_status make_map5_gate_up(CUtensorMap* m, const void* w1, const void* w3, uint64_t rows,
                             uint64_t cols, int* up_first) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(w1), b = reinterpret_cast<uintptr_t>(w3);
  *up_first = b < a;
  const uintptr_t gap = b < a ? a - b : b - a;
  if (gap == 0 || gap >= (static_cast<uintptr_t>(1) << 40)) return MOE_ERR_UNSUPPORTED;
  const cuuint64_t dims[5] = {static_cast<cuuint64_t>(tc::kBK), 64, 2, rows / 64, cols / tc::kBK};
  const cuuint64_t strides[4] = {cols * 2, static_cast<cuuint64_t>(gap), 64 * cols * 2,
                                 tc::kBK * 2};
  const cuuint32_t box[5] = {static_cast<cuuint32_t>(tc::kBK), 64, 2, 1, tc::kKPS};
  return encode(m, 5, b < a ? w3 : w1, dims, strides, box);
}

// bf16 output [rows, cols] row-major for the epilogue's bulk stores: box of
// 32 columns x box_rows rows, plain row-major tile in shared memory.
moe_status make_out_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                        uint32_t box_rows = 32) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {32, box_rows};
  return encode(m, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// fp32 output [rows, cols] row-major for the epilogue's bulk stores: box of
// 32 columns x 32 rows.
moe_status make_out_map_f32(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 4};
  const cuuint32_t box[2] = {32, 32};
  return encode(m, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
}

// Token-source maps for every box height.
moe_status make_token_maps(CUtensorMap* maps, const void* base, uint64_t rows, uint64_t cols) {
  for (int i = 0; i < tc::kNumBoxes; ++i) MOE_TRY(make_map3(&maps[i], base, rows, cols, 16u << i));
  return MOE_OK;
}


// The persistent grid of the grouped GEMM: one CTA per SM, or for PAIR == 2
// as many two-CTA clusters as fit on the device at once.  The dynamic
// shared-memory limit and the grid are set up once per device.
template <int EPI, int BN, int PAIR>
cudaLaunchConfig_t tc_config(cudaLaunchAttribute* attr, cudaStream_t st) {
  using C = tc::EpiConfig<EPI, BN, PAIR>;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = PAIR;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(tc::num_threads<EPI>(), 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = PAIR == 2 ? 1 : 0;
  return cfg;
}

template <int EPI, int BN, int PAIR>
moe_status tc_grid(int* grid) {
  using C = tc::EpiConfig<EPI, BN, PAIR>;
  auto kern = tc::grouped_gemm_kernel<EPI, BN, PAIR>;
  static int grid_for[64] = {0};
  int dev = 0;
  MOE_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
  if (grid_for[dev] == 0) {
    MOE_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  C::kSmemBytes));
    int g = num_sms();
    if (PAIR == 2) {
      cudaLaunchAttribute attr[1];
      cudaLaunchConfig_t cfg = tc_config<EPI, BN, PAIR>(attr, nullptr);
      int clusters = 0;
      cfg.gridDim = dim3(static_cast<unsigned>(g - g % 2), 1, 1);
      MOE_CUDA(cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg));
      if (clusters < 1) return cuda_fail(cudaErrorInvalidConfiguration);
      g = 2 * clusters;
    }
    grid_for[dev] = g;
  }
  *grid = grid_for[dev];
  return MOE_OK;
}

// Launches the grouped GEMM persistently on its grid (at most max_ctas CTAs).
template <int EPI, int BN, int PAIR>
moe_status launch_tc(const tc::Params& p, int max_ctas, cudaStream_t st) {
  int grid = 0;
  MOE_TRY((tc_grid<EPI, BN, PAIR>(&grid)));
  grid = std::min(grid, std::max(max_ctas, PAIR));
  grid -= grid % PAIR;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = tc_config<EPI, BN, PAIR>(attr, st);
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  MOE_CUDA(cudaLaunchKernelEx(&cfg, tc::grouped_gemm_kernel<EPI, BN, PAIR>, p));
  return MOE_OK;
}

// Expert GEMMs: 256-token tiles on CTA pairs, 64-token tiles on single CTAs.
template <int EPI>
moe_status launch_ffn(const tc::Params& p, int bn, cudaStream_t st) {
  return bn == 256 ? launch_tc<EPI, 256, 2>(p, INT_MAX, st) : launch_tc<EPI, 64, 1>(p, INT_MAX, st);
}

// ---------------------------------------------------------------- workspace

struct DispatchWs {
  int32_t* chunk_hist;
  int32_t* chunk_base;
};

size_t dispatch_ws_bytes(const moe_shape* s) {
  const size_t n = static_cast<size_t>(cdiv(s->T, kDispatchChunk)) * s->n_routed * 4;
  return 2 * align256(n);
}

DispatchWs carve_dispatch(void* ws, const moe_shape* s) {
  const size_t n = static_cast<size_t>(cdiv(s->T, kDispatchChunk)) * s->n_routed * 4;
  char* p = static_cast<char*>(ws);
  return DispatchWs{reinterpret_cast<int32_t*>(p), reinterpret_cast<int32_t*>(p + align256(n))};
}

struct FfnWs {
  GroupDesc* g1;
  GroupDesc* g2;
  int* tile_prefix;
  void* act;
};

// Rows of the routed experts' input: T·k for a layer, or the rows an
// expert-parallel rank received (moe_expert_ffn_rows).
size_t routed_rows_of(const moe_shape* s, long long routed_rows) {
  return routed_rows >= 0 ? static_cast<size_t>(routed_rows)
                          : static_cast<size_t>(s->T) * s->top_k;
}

size_t act_rows(const moe_shape* s, long long routed_rows = -1) {
  return routed_rows_of(s, routed_rows) + static_cast<size_t>(s->T) * s->n_shared;
}

// Shared experts are planned as pieces of kSharedPiece tokens (a multiple of
// every token-tile height) spread between the routed experts; the number of
// pieces keeps the group count within the grouped GEMM's 1024.
constexpr int kSharedPiece = 512;

int shared_pieces(const moe_shape* s) {
  if (s->n_shared == 0 || s->T == 0) return 0;
  const int cap = (1024 - s->n_routed) / s->n_shared;  // >= 1: n_routed + n_shared <= 1024
  return std::max(1, std::min(cdiv(s->T, kSharedPiece), cap));
}

int shared_piece_rows(const moe_shape* s) {
  const int p = shared_pieces(s);
  return p == 0 ? 0 : cdiv(cdiv(s->T, p), kSharedPiece) * kSharedPiece;
}

size_t ffn_groups(const moe_shape* s) {
  return static_cast<size_t>(s->n_routed) + static_cast<size_t>(s->n_shared) * shared_pieces(s);
}

size_t ffn_ws_bytes(const moe_shape* s, long long routed_rows = -1) {
  const size_t G = ffn_groups(s);
  return 2 * align256(G * sizeof(GroupDesc)) + align256((G + 1) * 4) +
         align256(act_rows(s, routed_rows) * s->inter * elt_bytes(s));
}

FfnWs carve_ffn(void* ws, const moe_shape* s) {
  const size_t G = ffn_groups(s);
  char* p = static_cast<char*>(ws);
  FfnWs w;
  w.g1 = reinterpret_cast<GroupDesc*>(p);
  p += align256(G * sizeof(GroupDesc));
  w.g2 = reinterpret_cast<GroupDesc*>(p);
  p += align256(G * sizeof(GroupDesc));
  w.tile_prefix = reinterpret_cast<int*>(p);
  p += align256((G + 1) * 4);
  w.act = p;
  return w;
}

// Router logits of a batch with few (128-expert x 64-token) tiles: the
// contraction over H is cut into ranges of whole pipeline stages so that
// about kRouterCtas CTAs stream it, each range's partial logits written apart
// and added in order after (decode: 3 tiles over H = 7168 take 28 ranges of
// four k-blocks).  Large batches have enough tiles and stay whole.  Fixed
// constants, not the device's SM count, so the workspace size is the same
// on every device.
constexpr int kRouterCtas = 128;
constexpr int kRouterMaxSplits = 32;
int router_splits(const moe_shape* s, int* blocks_per_range) {
  *blocks_per_range = 0;
  if (s->dtype != MOE_DTYPE_BF16 || s->T <= 0) return 1;
  const int tiles = cdiv(s->n_routed, tc::kBM) * cdiv(s->T, 64);
  const int nkb = cdiv(s->H, tc::kBK);
  const int want = std::min({kRouterMaxSplits, kRouterCtas / tiles, nkb / tc::kKPS});
  if (want < 2) return 1;
  const int per = tc::kKPS * cdiv(nkb, want * tc::kKPS);
  const int S = cdiv(nkb, per);
  if (S < 2) return 1;
  *blocks_per_range = per;
  return S;
}

size_t router_ws_bytes(const moe_shape* s) {
  int per = 0;
  const int S = router_splits(s, &per);
  return S > 1 ? static_cast<size_t>(S) * s->T * s->n_routed * 4 : 0;
}

struct LayerWs {
  float* logits;
  float* logit_part;  // the router's partial logits [S, T, E] (nullptr: not split)
  int32_t* idx;
  float* w;
  int32_t* offsets;
  int32_t* row_token;
  int32_t* slot_row;
  void* u_perm;
  void* y_perm;
  void* y_shared;
  void* dispatch_ws;
  void* ffn_ws;
  size_t total;
};

LayerWs carve_layer(void* ws, const moe_shape* s) {
  const size_t T = s->T, E = s->n_routed, k = s->top_k, Ks = s->n_shared, H = s->H;
  const size_t e = elt_bytes(s);
  char* base = static_cast<char*>(ws);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = base + off;
    off += align256(bytes);
    return static_cast<void*>(p);
  };
  LayerWs L;
  L.logits = static_cast<float*>(take(T * E * 4));
  const size_t part_bytes = router_ws_bytes(s);
  L.logit_part = part_bytes ? static_cast<float*>(take(part_bytes)) : nullptr;
  L.idx = static_cast<int32_t*>(take(T * k * 4));
  L.w = static_cast<float*>(take(T * k * 4));
  L.offsets = static_cast<int32_t*>(take((E + 1) * 4));
  L.row_token = static_cast<int32_t*>(take(T * k * 4));
  L.slot_row = static_cast<int32_t*>(take(T * k * 4));
  L.u_perm = take(T * k * H * e);
  L.y_perm = take(T * k * H * e);
  L.y_shared = take(Ks * T * H * e);
  L.dispatch_ws = take(dispatch_ws_bytes(s));
  L.ffn_ws = take(ffn_ws_bytes(s));
  L.total = off;
  return L;
}

// ---------------------------------------------------------------- steps

int route_blocks(int T) { return std::max(1, std::min(cdiv(T, 8), num_sms() * 8)); }

// Row work of the scatter and the combine: a warp takes one (token, segment)
// item at a time.  A batch of fewer tokens than about 32 warps per SM gets
// several segments per token row, each of whole 32-vector passes (decode:
// 64 tokens of 896 vectors become 64 x 28 items); larger batches keep one
// segment per token.  `blocks` covers the items with 8-warp blocks, at most
// `max_blocks_per_sm` a SM (a grid-stride loop takes the rest).
struct RowSplit {
  int nseg, seg_vecs, blocks;
};
RowSplit row_split(int T, int nvec, int max_blocks_per_sm) {
  RowSplit r{1, nvec, 1};
  const int per = T > 0 ? num_sms() * 32 / T : 1;
  if (per > 1 && nvec > 32) {
    r.seg_vecs = 32 * cdiv(nvec, 32 * per);
    r.nseg = cdiv(nvec, r.seg_vecs);
  }
  const long long items = static_cast<long long>(T) * r.nseg;
  r.blocks = static_cast<int>(std::max<long long>(
      1, std::min<long long>(cdiv(items, 8LL), static_cast<long long>(num_sms()) * max_blocks_per_sm)));
  return r;
}

// Blocks of `threads` that are resident on the device at once (one wave) for
// a kernel without dynamic shared memory; cached per kernel and device.
template <typename K>
int one_wave_blocks(K kernel, int threads) {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) !=
            cudaSuccess || per_sm <= 0)
      return 0;
    cached[dev] = per_sm * num_sms();
  }
  return cached[dev];
}

// part: scratch for the router_splits ranges' partial logits, or nullptr to
// run the contraction whole.
moe_status do_router_logits(const moe_shape* s, const void* u, const void* cent,
                            const float* off, float* logits, float* part, cudaStream_t st) {
  const int T = s->T, E = s->n_routed, H = s->H;
  if (T == 0) return MOE_OK;
  if (s->dtype == MOE_DTYPE_F32) {
    SimtParams p{};
    p.a[0] = p.a[1] = static_cast<const float*>(cent);
    p.b[0] = p.b[1] = static_cast<const float*>(u);
    p.out[0] = p.out[1] = logits;
    p.groups = nullptr;
    p.dense_count = T;
    p.K = H;
    p.n_cols = E;
    p.out_ld = E;
    p.col_offset = off;
    dim3 grid(cdiv(E, kSimtTile), cdiv(T, kSimtTile), 1);
    simt_gemm_kernel<SIMT_LOGITS><<<grid, 256, 0, st>>>(p);
    MOE_CUDA(cudaGetLastError());
    return MOE_OK;
  }
  tc::Params p;
  memset(&p, 0, sizeof(p));
  MOE_TRY(make_map3(&p.a[0], cent, E, H, tc::kBM));
  p.a[1] = p.a[0];
  MOE_TRY(make_token_maps(p.b[0], u, T, H));
  memcpy(p.b[1], p.b[0], sizeof(p.b[0]));
  p.groups = nullptr;
  p.tile_prefix = nullptr;
  p.dense_count = T;
  p.n_wtiles = cdiv(E, tc::kBM);
  p.num_k_blocks = cdiv(H, tc::kBK);
  p.out[0] = p.out[1] = logits;
  p.out_ld = E;
  p.out_cols = E;
  p.col_offset = off;
  const int bn = (T > 64 && p.n_wtiles * cdiv(T, 256) >= num_sms()) ? 256 : 64;
  const int tiles = p.n_wtiles * cdiv(T, bn);
  int per = 0;
  const int S = part != nullptr && bn == 64 ? router_splits(s, &per) : 1;
  if (S > 1) {
    // the ranges' partial logits, without the offset; then their sum
    p.k_splits = S;
    p.k_split_blocks = per;
    p.split_stride = static_cast<long long>(T) * E;
    p.out[0] = p.out[1] = part;
    p.col_offset = nullptr;
    MOE_TRY((launch_tc<tc::EPI_F32, 64, 1>(p, tiles * S, st)));
    const long long n = static_cast<long long>(T) * E;
    const int blocks = static_cast<int>(std::min<long long>((n + 255) / 256, num_sms() * 4LL));
    sum_logit_partials_kernel<<<blocks, 256, 0, st>>>(part, S, n, E, off, logits);
    MOE_CUDA(cudaGetLastError());
    return MOE_OK;
  }
  return bn == 256 ? launch_tc<tc::EPI_F32, 256, 1>(p, tiles, st)
                   : launch_tc<tc::EPI_F32, 64, 1>(p, tiles, st);
}

moe_status do_route(const moe_shape* s, const float* logits, const float* bias, int32_t* idx,
                    float* w, float* gap, cudaStream_t st) {
  const int T = s->T, E = s->n_routed;
  if (T == 0) return MOE_OK;
  const int blocks = route_blocks(T);
  const int npl = cdiv(E, 32);
  const int gate = s->gate == MOE_GATE_SOFTMAX ? 0 : 1;
#define MOE_ROUTE(N)                                                                     \
  route_kernel<N><<<blocks, 256, 0, st>>>(logits, bias, T, E, s->top_k, gate, s->n_groups, \
                                          s->topk_groups, idx, w, gap)
  if (npl <= 1) MOE_ROUTE(1);
  else if (npl <= 2) MOE_ROUTE(2);
  else if (npl <= 4) MOE_ROUTE(4);
  else if (npl <= 8) MOE_ROUTE(8);
  else if (npl <= 16) MOE_ROUTE(16);
  else MOE_ROUTE(32);
#undef MOE_ROUTE
  MOE_CUDA(cudaGetLastError());
  return MOE_OK;
}

moe_status do_dispatch(const moe_shape* s, const int32_t* idx, const void* u, int32_t* offsets,
                       int32_t* row_token, int32_t* slot_row, void* u_perm, void* ws,
                       cudaStream_t st) {
  const int T = s->T, E = s->n_routed, k = s->top_k;
  const int n_chunks = cdiv(T, kDispatchChunk);
  DispatchWs d = carve_dispatch(ws, s);
  if (n_chunks > 0 && k > 0)
    dispatch_count<<<n_chunks, 256, E * 4, st>>>(idx, T, k, E, d.chunk_hist);
  else if (n_chunks > 0)
    MOE_CUDA(cudaMemsetAsync(d.chunk_hist, 0, static_cast<size_t>(n_chunks) * E * 4, st));
  MOE_CUDA(cudaGetLastError());
  dispatch_scan<<<1, 1024, 0, st>>>(d.chunk_hist, n_chunks, E, d.chunk_base, offsets);
  MOE_CUDA(cudaGetLastError());
  if (n_chunks == 0 || k == 0) return MOE_OK;
  dispatch_scatter<<<n_chunks, kDispatchWarps * 32, kDispatchWarps * E * 4, st>>>(
      idx, T, k, E, d.chunk_base, row_token, slot_row);
  MOE_CUDA(cudaGetLastError());
  const int esize = s->dtype == MOE_DTYPE_F32 ? 4 : 2;
  const RowSplit rs = row_split(T, s->H * esize / 16, 16);
  if (s->dtype == MOE_DTYPE_F32)
    scatter_token_rows<float><<<rs.blocks, 256, 0, st>>>(static_cast<const float*>(u), T, k,
                                                         slot_row, s->H, rs.nseg, rs.seg_vecs,
                                                         static_cast<float*>(u_perm));
  else
    scatter_token_rows<__nv_bfloat16><<<rs.blocks, 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(u), T, k, slot_row, s->H, rs.nseg, rs.seg_vecs,
        static_cast<__nv_bfloat16*>(u_perm));
  MOE_CUDA(cudaGetLastError());
  return MOE_OK;
}

// Token tile height for the tensor-core expert GEMMs: wide tiles when experts
// get many rows, narrow (deeper pipeline) when they get a handful.
int ffn_bn(const moe_shape* s, long long routed_rows = -1) {
  const long long rr = static_cast<long long>(routed_rows_of(s, routed_rows));
  const long long avg = rr / s->n_routed;
  return (avg > 48 || (s->n_shared > 0 && rr == 0 && s->T > 64)) ? 256 : 64;
}

// save_a / save_c (bf16 layers, may be null): GEMM1 also stores the
// pre-activations a = x W1ᵀ and (SwiGLU) c = x W3ᵀ, [act_rows, I] each, rows
// laid out like the activation (routed rows, then each shared expert's T).
moe_status do_expert_ffn(const moe_shape* s, const moe_weights* wt, const void* u,
                         const void* u_perm, const int32_t* offsets, void* y_perm,
                         void* y_shared, void* ws, cudaStream_t st, void* save_a = nullptr,
                         void* save_c = nullptr, long long routed_rows = -1) {
  const int T = s->T, E = s->n_routed, Ks = s->n_shared, H = s->H, I = s->inter;
  const int G = static_cast<int>(ffn_groups(s));
  const int Tk = static_cast<int>(routed_rows_of(s, routed_rows));  // routed input rows
  const int rows_act = static_cast<int>(act_rows(s, routed_rows));
  if (rows_act == 0) return MOE_OK;
  // the largest group: a routed expert takes at most one row per token of a
  // layer, or any number of the rows a rank received
  const int max_group = std::max(T, routed_rows >= 0 ? Tk : 0);
  FfnWs f = carve_ffn(ws, s);  // act is carved last, so the row count does not move it
  const bool f32 = s->dtype == MOE_DTYPE_F32;
  const int bn = f32 ? kSimtTile : ffn_bn(s, routed_rows);
  // weights read by about two token tiles or fewer stream from HBM: mix
  // heavily and lightly loaded experts through the launch
  const int by_load = (!f32 && static_cast<long long>(Tk) <= 2LL * bn * E) ? 1 : 0;
  ffn_plan_kernel<<<1, cdiv(G, 32) * 32, 0, st>>>(offsets, E, Ks, T, Tk, I, H, bn,
                                                   shared_pieces(s), shared_piece_rows(s),
                                                   by_load, f.g1, f.g2, f.tile_prefix);
  MOE_CUDA(cudaGetLastError());
  const bool swiglu = s->act == MOE_ACT_SWIGLU;

  if (f32) {
    SimtParams p{};
    p.a[0] = static_cast<const float*>(wt->w1);
    p.a[1] = static_cast<const float*>(Ks ? wt->sw1 : wt->w1);
    p.a3[0] = static_cast<const float*>(swiglu ? wt->w3 : nullptr);
    p.a3[1] = static_cast<const float*>(swiglu ? (Ks ? wt->sw3 : wt->w3) : nullptr);
    p.b[0] = static_cast<const float*>(Tk ? u_perm : u);
    p.b[1] = static_cast<const float*>(u);
    p.out[0] = p.out[1] = static_cast<float*>(f.act);
    p.groups = f.g1;
    p.K = H;
    p.n_cols = I;
    p.out_ld = I;
    dim3 g1(cdiv(I, kSimtTile), cdiv(max_group, kSimtTile), G);
    if (swiglu) simt_gemm_kernel<SIMT_SWIGLU><<<g1, 256, 0, st>>>(p);
    else simt_gemm_kernel<SIMT_RELU><<<g1, 256, 0, st>>>(p);
    MOE_CUDA(cudaGetLastError());
    SimtParams q{};
    q.a[0] = static_cast<const float*>(wt->w2);
    q.a[1] = static_cast<const float*>(Ks ? wt->sw2 : wt->w2);
    q.b[0] = q.b[1] = static_cast<const float*>(f.act);
    q.out[0] = static_cast<float*>(Tk ? y_perm : y_shared);
    q.out[1] = static_cast<float*>(Ks ? y_shared : y_perm);
    q.groups = f.g2;
    q.K = I;
    q.n_cols = H;
    q.out_ld = H;
    dim3 g2(cdiv(H, kSimtTile), cdiv(max_group, kSimtTile), G);
    simt_gemm_kernel<SIMT_PLAIN><<<g2, 256, 0, st>>>(q);
    MOE_CUDA(cudaGetLastError());
    return MOE_OK;
  }

  // ---- GEMM1: gate/up projection with the activation fused in the epilogue
  tc::Params p;
  memset(&p, 0, sizeof(p));
  const uint32_t a1_box = swiglu ? tc::kBM / 2 : tc::kBM;  // output columns per CTA
  if (swiglu) {
    MOE_TRY(make_map5_gate_up(&p.a[0], wt->w1, wt->w3, static_cast<uint64_t>(E) * I, H,
                              &p.up_first[0]));
    if (Ks)
      MOE_TRY(make_map5_gate_up(&p.a[1], wt->sw1, wt->sw3, static_cast<uint64_t>(Ks) * I, H,
                                &p.up_first[1]));
    else {
      p.a[1] = p.a[0];
      p.up_first[1] = p.up_first[0];
    }
  } else {
    MOE_TRY(make_map3(&p.a[0], wt->w1, static_cast<uint64_t>(E) * I, H, tc::kBM));
    if (Ks) MOE_TRY(make_map3(&p.a[1], wt->sw1, static_cast<uint64_t>(Ks) * I, H, tc::kBM));
    else p.a[1] = p.a[0];
  }
  MOE_TRY(make_token_maps(p.b[1], u, T, H));
  if (Tk) MOE_TRY(make_token_maps(p.b[0], u_perm, Tk, H));
  else memcpy(p.b[0], p.b[1], sizeof(p.b[0]));
  // wide token tiles run on CTA pairs: 256 weight rows per tile
  const int pair = bn == 256 ? 2 : 1;
  p.groups = f.g1;
  p.tile_prefix = f.tile_prefix;
  p.n_groups = G;
  p.n_wtiles = cdiv(I, static_cast<int>(a1_box) * pair);
  p.num_k_blocks = cdiv(H, tc::kBK);
  p.out[0] = p.out[1] = f.act;
  MOE_TRY(make_out_map(&p.omap[0], f.act, rows_act, I));
  p.omap[1] = p.omap[0];
  MOE_TRY(make_out_map(&p.omap16[0], f.act, rows_act, I, 16));
  p.omap16[1] = p.omap16[0];
  p.out_ld = I;
  p.out_cols = I;
  if (save_a != nullptr) {
    p.save = 1;
    p.save_out[0] = save_a;
    p.save_out[1] = swiglu ? save_c : save_a;
    MOE_TRY(make_out_map(&p.save_map[0], save_a, rows_act, I));
    MOE_TRY(make_out_map(&p.save_map[1], p.save_out[1], rows_act, I));
  }
  if (swiglu) MOE_TRY(launch_ffn<tc::EPI_SWIGLU>(p, bn, st));
  else MOE_TRY(launch_ffn<tc::EPI_RELU>(p, bn, st));

  // ---- GEMM2: down projection
  tc::Params q;
  memset(&q, 0, sizeof(q));
  MOE_TRY(make_map3(&q.a[0], wt->w2, static_cast<uint64_t>(E) * H, I, tc::kBM));
  if (Ks) MOE_TRY(make_map3(&q.a[1], wt->sw2, static_cast<uint64_t>(Ks) * H, I, tc::kBM));
  else q.a[1] = q.a[0];
  MOE_TRY(make_token_maps(q.b[0], f.act, rows_act, I));
  memcpy(q.b[1], q.b[0], sizeof(q.b[0]));
  q.groups = f.g2;
  q.tile_prefix = f.tile_prefix;
  q.n_groups = G;
  q.n_wtiles = cdiv(H, tc::kBM * pair);
  q.num_k_blocks = cdiv(I, tc::kBK);
  q.out[0] = Tk ? y_perm : y_shared;
  q.out[1] = Ks ? y_shared : y_perm;
  MOE_TRY(make_out_map(&q.omap[0], q.out[0], Tk ? Tk : static_cast<uint64_t>(Ks) * T, H));
  MOE_TRY(make_out_map(&q.omap[1], q.out[1], Ks ? static_cast<uint64_t>(Ks) * T : Tk, H));
  q.out_ld = H;
  q.out_cols = H;
  return launch_ffn<tc::EPI_BF16>(q, bn, st);
}

moe_status do_combine(const moe_shape* s, const void* u, const void* y_perm,
                      const void* y_shared, const float* w, const int32_t* slot_row, void* h,
                      cudaStream_t st) {
  const int T = s->T;
  if (T == 0) return MOE_OK;
  const bool f32 = s->dtype == MOE_DTYPE_F32;
  const RowSplit rs = row_split(T, s->H / (f32 ? 4 : 8), 8);
  if (f32)
    combine_kernel<float><<<rs.blocks, 256, 0, st>>>(
        static_cast<const float*>(u), static_cast<const float*>(y_perm),
        static_cast<const float*>(y_shared), w, slot_row, T, s->H, s->top_k, s->n_shared,
        rs.nseg, rs.seg_vecs, static_cast<float*>(h));
  else
    combine_kernel<__nv_bfloat16><<<rs.blocks, 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(u), static_cast<const __nv_bfloat16*>(y_perm),
        static_cast<const __nv_bfloat16*>(y_shared), w, slot_row, T, s->H, s->top_k,
        s->n_shared, rs.nseg, rs.seg_vecs, static_cast<__nv_bfloat16*>(h));
  MOE_CUDA(cudaGetLastError());
  return MOE_OK;
}

// Pointer checks: required pointers non-null and 16-byte aligned.
bool ok_ptr(const void* p) { return p != nullptr && al16(p); }
bool ok_opt(const void* p) { return p == nullptr || al16(p); }

moe_status check_weights_ffn(const moe_shape* s, const moe_weights* w) {
  if (w == nullptr) return MOE_ERR_INVALID_ARG;
  const bool sw = s->act == MOE_ACT_SWIGLU;
  if (!ok_ptr(w->w1) || !ok_ptr(w->w2) || (sw && !ok_ptr(w->w3))) return MOE_ERR_INVALID_ARG;
  if (s->n_shared > 0 && (!ok_ptr(w->sw1) || !ok_ptr(w->sw2) || (sw && !ok_ptr(w->sw3))))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// Host-buffer pipeline: how many token chunks, and the two copy streams
// (created once per device, non-blocking, kept until the process exits).
// A chunk keeps at least kHostChunkTokens tokens and, on average, two full
// 256-row token tiles per routed expert: smaller chunks would add partly
// filled tiles, each of which streams its expert's weights again.
constexpr int kMaxHostChunks = 8;
constexpr int kHostChunkTokens = 4096;
constexpr int kHostChunkExpertRows = 512;

int host_chunks(const moe_shape* s) {
  int n = s->T / kHostChunkTokens;
  if (s->top_k > 0)
    n = std::min<long long>(n, static_cast<long long>(s->T) * s->top_k /
                                   (static_cast<long long>(s->n_routed) * kHostChunkExpertRows));
  return std::max(1, std::min(kMaxHostChunks, n));
}

struct CopyStreams {
  cudaStream_t in, out;
};

moe_status copy_streams(CopyStreams* out) {
  static std::mutex mu;
  static CopyStreams per_dev[64];
  static bool made[64] = {false};
  int dev = 0;
  MOE_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  if (!made[dev]) {
    MOE_CUDA(cudaStreamCreateWithFlags(&per_dev[dev].in, cudaStreamNonBlocking));
    MOE_CUDA(cudaStreamCreateWithFlags(&per_dev[dev].out, cudaStreamNonBlocking));
    made[dev] = true;
  }
  *out = per_dev[dev];
  return MOE_OK;
}

// What moe_layer_forward_train keeps for moe_layer_backward.
struct SavedLayout {
  float* logits;       // [T, E]
  int32_t* idx;        // [T, k]
  float* w;            // [T, k]
  int32_t* offsets;    // [E + 1]
  int32_t* row_token;  // [T·k]
  int32_t* slot_row;   // [T·k]
  void* x_perm;        // [T·k, H]
  void* a;             // [T·(k + Ks), I]
  void* c;             // [T·(k + Ks), I] (SwiGLU)
  size_t total;
};

SavedLayout carve_saved(void* base_ptr, const moe_shape* s) {
  const size_t T = s->T, E = s->n_routed, k = s->top_k, H = s->H, I = s->inter;
  char* base = static_cast<char*>(base_ptr);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = base + off;
    off += align256(bytes);
    return static_cast<void*>(p);
  };
  SavedLayout S;
  S.logits = static_cast<float*>(take(T * E * 4));
  S.idx = static_cast<int32_t*>(take(T * k * 4));
  S.w = static_cast<float*>(take(T * k * 4));
  S.offsets = static_cast<int32_t*>(take((E + 1) * 4));
  S.row_token = static_cast<int32_t*>(take(T * k * 4));
  S.slot_row = static_cast<int32_t*>(take(T * k * 4));
  S.x_perm = take(T * k * H * 2);
  S.a = take(act_rows(s) * I * 2);
  S.c = s->act == MOE_ACT_SWIGLU ? take(act_rows(s) * I * 2) : nullptr;
  S.total = off;
  return S;
}

moe_status layer_forward(const moe_shape* s, const moe_weights* wt, const void* u, void* h,
                         const moe_route_outputs* ro, void* ws, size_t ws_bytes,
                         cudaStream_t st, void* saved = nullptr) {
  MOE_TRY(check_shape(s));
  MOE_TRY(check_weights_ffn(s, wt));
  if (!ok_ptr(wt->centroids) || !ok_opt(wt->logit_offset) || !ok_opt(wt->select_bias))
    return MOE_ERR_INVALID_ARG;
  if (s->T > 0 && (!ok_ptr(u) || !ok_ptr(h))) return MOE_ERR_INVALID_ARG;
  if (ro != nullptr && (!ok_opt(ro->logits) || !ok_opt(ro->topk_idx) || !ok_opt(ro->topk_w) ||
                        !ok_opt(ro->expert_offsets)))
    return MOE_ERR_INVALID_ARG;
  LayerWs L = carve_layer(nullptr, s);
  if (ws == nullptr || !al16(ws) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  L = carve_layer(ws, s);
  float* logits = (ro && ro->logits) ? ro->logits : L.logits;
  int32_t* idx = (ro && ro->topk_idx) ? ro->topk_idx : L.idx;
  float* w = (ro && ro->topk_w) ? ro->topk_w : L.w;
  int32_t* offsets = (ro && ro->expert_offsets) ? ro->expert_offsets : L.offsets;
  int32_t* row_token = L.row_token;
  int32_t* slot_row = L.slot_row;
  void* u_perm = L.u_perm;
  void *save_a = nullptr, *save_c = nullptr;
  if (saved != nullptr) {  // training: routing, permuted rows and pre-activations are kept
    SavedLayout S = carve_saved(saved, s);
    logits = S.logits;
    idx = S.idx;
    w = S.w;
    offsets = S.offsets;
    row_token = S.row_token;
    slot_row = S.slot_row;
    u_perm = S.x_perm;
    save_a = S.a;
    save_c = S.c;
  }
  const float* bias = s->gate == MOE_GATE_SIGMOID_BIAS ? wt->select_bias : nullptr;
  MOE_TRY(do_router_logits(s, u, wt->centroids, wt->logit_offset, logits, L.logit_part, st));
  MOE_TRY(do_route(s, logits, bias, idx, w, nullptr, st));
  MOE_TRY(do_dispatch(s, idx, u, offsets, row_token, slot_row, u_perm, L.dispatch_ws, st));
  MOE_TRY(do_expert_ffn(s, wt, u, u_perm, offsets, L.y_perm, L.y_shared, L.ffn_ws, st, save_a,
                        save_c));
  return do_combine(s, u, L.y_perm, L.y_shared, w, slot_row, h, st);
}

}  // namespace

// ==================================================================== C ABI

extern "C" {

MOE_API const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

MOE_API int moe_last_cuda_error(void) { return t_last_cuda_error; }

MOE_API moe_status moe_device_status(moe_stream_t stream, int32_t* code) {
  MOE_CUDA(cudaStreamSynchronize(cs(stream)));
  int v = 0;
  MOE_CUDA(cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)));
  if (v != 0) {
    const int zero = 0;
    MOE_CUDA(cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)));
  }
  if (code != nullptr) *code = v;
  if (v & (DEV_ERR_TIMEOUT_PRODUCER | DEV_ERR_TIMEOUT_MMA | DEV_ERR_TIMEOUT_EPILOGUE))
    return MOE_ERR_TIMEOUT;
  if (v & DEV_ERR_BAD_EXPERT) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

MOE_API moe_status moe_check_bounded_wait(uint32_t limit_us, moe_stream_t stream) {
  if (limit_us == 0 || limit_us > 1000000) return MOE_ERR_INVALID_ARG;
  tc::wait_timeout_probe_kernel<<<1, 32, 0, cs(stream)>>>(
      static_cast<uint64_t>(limit_us) * 1000ull, DEV_ERR_TIMEOUT_MMA);
  MOE_CUDA(cudaGetLastError());
  return MOE_OK;
}

MOE_API size_t moe_dispatch_workspace_size(const moe_shape* s) {
  return check_shape(s) == MOE_OK ? dispatch_ws_bytes(s) : 0;
}

MOE_API size_t moe_expert_ffn_workspace_size(const moe_shape* s) {
  return check_shape(s) == MOE_OK ? ffn_ws_bytes(s) : 0;
}

MOE_API size_t moe_layer_workspace_size(const moe_shape* s) {
  return check_shape(s) == MOE_OK ? carve_layer(nullptr, s).total : 0;
}

MOE_API size_t moe_router_logits_workspace_size(const moe_shape* s) {
  return check_shape(s) == MOE_OK ? router_ws_bytes(s) : 0;
}

MOE_API moe_status moe_router_logits(const moe_shape* s, const void* u, const void* centroids,
                                     const float* logit_offset, float* logits, void* ws,
                                     size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_shape(s));
  if (!ok_ptr(centroids) || !ok_opt(logit_offset)) return MOE_ERR_INVALID_ARG;
  if (s->T > 0 && (!ok_ptr(u) || !ok_ptr(logits))) return MOE_ERR_INVALID_ARG;
  const size_t need = router_ws_bytes(s);
  if (ws != nullptr && (!al16(ws) || ws_bytes < need)) return MOE_ERR_WORKSPACE;
  float* part = ws != nullptr && need > 0 ? static_cast<float*>(ws) : nullptr;
  return do_router_logits(s, u, centroids, logit_offset, logits, part, cs(stream));
}

MOE_API moe_status moe_route(const moe_shape* s, const float* logits, const float* select_bias,
                             int32_t* topk_idx, float* topk_w, float* kth_gap,
                             moe_stream_t stream) {
  MOE_TRY(check_shape(s));
  if (!ok_opt(select_bias) || !ok_opt(kth_gap)) return MOE_ERR_INVALID_ARG;
  if (s->T > 0 && !ok_ptr(logits)) return MOE_ERR_INVALID_ARG;
  if (s->T > 0 && s->top_k > 0 && (!ok_ptr(topk_idx) || !ok_ptr(topk_w)))
    return MOE_ERR_INVALID_ARG;
  const float* bias = s->gate == MOE_GATE_SIGMOID_BIAS ? select_bias : nullptr;
  return do_route(s, logits, bias, topk_idx, topk_w, kth_gap, cs(stream));
}

MOE_API moe_status moe_dispatch(const moe_shape* s, const int32_t* topk_idx, const void* u,
                                int32_t* expert_offsets, int32_t* row_token, int32_t* slot_row,
                                void* u_perm, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_shape(s));
  if (!ok_ptr(expert_offsets)) return MOE_ERR_INVALID_ARG;
  if (s->top_k > 0 && s->T > 0 && (!ok_ptr(topk_idx) || !ok_ptr(u) || !ok_ptr(row_token) ||
                                   !ok_ptr(slot_row) || !ok_ptr(u_perm)))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < dispatch_ws_bytes(s) || (dispatch_ws_bytes(s) > 0 && (ws == nullptr || !al16(ws))))
    return MOE_ERR_WORKSPACE;
  return do_dispatch(s, topk_idx, u, expert_offsets, row_token, slot_row, u_perm, ws,
                     cs(stream));
}

MOE_API moe_status moe_expert_ffn(const moe_shape* s, const moe_weights* weights, const void* u,
                                  const void* u_perm, const int32_t* expert_offsets,
                                  void* y_perm, void* y_shared, void* ws, size_t ws_bytes,
                                  moe_stream_t stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(check_weights_ffn(s, weights));
  if (!ok_ptr(expert_offsets)) return MOE_ERR_INVALID_ARG;
  if (s->T > 0 && !ok_ptr(u)) return MOE_ERR_INVALID_ARG;
  if (s->top_k > 0 && s->T > 0 && (!ok_ptr(u_perm) || !ok_ptr(y_perm)))
    return MOE_ERR_INVALID_ARG;
  if (s->n_shared > 0 && s->T > 0 && !ok_ptr(y_shared)) return MOE_ERR_INVALID_ARG;
  if (ws == nullptr || !al16(ws) || ws_bytes < ffn_ws_bytes(s)) return MOE_ERR_WORKSPACE;
  return do_expert_ffn(s, weights, u, u_perm, expert_offsets, y_perm, y_shared, ws, cs(stream));
}

MOE_API moe_status moe_combine(const moe_shape* s, const void* u, const void* y_perm,
                               const void* y_shared, const float* topk_w,
                               const int32_t* slot_row, void* h, moe_stream_t stream) {
  MOE_TRY(check_shape(s));
  if (s->T > 0 && (!ok_ptr(u) || !ok_ptr(h))) return MOE_ERR_INVALID_ARG;
  if (s->top_k > 0 && s->T > 0 && (!ok_ptr(y_perm) || !ok_ptr(topk_w) || !ok_ptr(slot_row)))
    return MOE_ERR_INVALID_ARG;
  if (s->n_shared > 0 && s->T > 0 && !ok_ptr(y_shared)) return MOE_ERR_INVALID_ARG;
  return do_combine(s, u, y_perm, y_shared, topk_w, slot_row, h, cs(stream));
}

MOE_API moe_status moe_update_select_bias(const moe_shape* s, const int32_t* expert_offsets,
                                          float* select_bias, float gamma, int32_t* loads,
                                          moe_stream_t stream) {
  MOE_TRY(check_shape(s));
  if (!ok_ptr(expert_offsets) || !ok_ptr(select_bias) || !ok_opt(loads))
    return MOE_ERR_INVALID_ARG;
  if (!(gamma >= 0.0f) || gamma == INFINITY) return MOE_ERR_INVALID_ARG;  // also rejects NaN
  const int E = s->n_routed;
  bias_update_kernel<<<cdiv(E, 256), 256, 0, cs(stream)>>>(
      expert_offsets, E, static_cast<long long>(s->T) * s->top_k, gamma, select_bias, loads);
  MOE_CUDA(cudaGetLastError());
  return MOE_OK;
}

MOE_API size_t moe_balance_stats_workspace_size(const moe_shape* s) {
  if (check_shape(s) != MOE_OK) return 0;
  return align256(static_cast<size_t>(cdiv(s->T, kStatChunk)) * s->n_routed * sizeof(float));
}

MOE_API moe_status moe_balance_stats(const moe_shape* s, const float* logits,
                                     const int32_t* expert_offsets, float* f, float* p, void* ws,
                                     size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_shape(s));
  if (!ok_ptr(expert_offsets) || !ok_ptr(f) || !ok_ptr(p)) return MOE_ERR_INVALID_ARG;
  if (s->T > 0 && !ok_ptr(logits)) return MOE_ERR_INVALID_ARG;
  const size_t need = moe_balance_stats_workspace_size(s);
  if (need > 0 && (ws == nullptr || !al16(ws) || ws_bytes < need)) return MOE_ERR_WORKSPACE;
  const int E = s->n_routed;
  const int n_chunks = cdiv(s->T, kStatChunk);
  float* partial = static_cast<float*>(ws);
  if (n_chunks > 0)
    balance_partial_kernel<<<n_chunks, 256, 0, cs(stream)>>>(
        logits, s->T, E, s->gate == MOE_GATE_SIGMOID_BIAS, partial);
  balance_final_kernel<<<cdiv(E, 256), 256, 0, cs(stream)>>>(partial, n_chunks, expert_offsets,
                                                             s->T, E, s->top_k, f, p);
  MOE_CUDA(cudaGetLastError());
  return MOE_OK;
}

#include "backward_api.cuh"  // the backward's host code, in place

MOE_API size_t moe_expert_ffn_rows_workspace_size(const moe_shape* s, int64_t max_rows) {
  if (check_shape(s) != MOE_OK || max_rows < 0 || max_rows > INT_MAX / 2) return 0;
  return ffn_ws_bytes(s, max_rows);
}

MOE_API moe_status moe_expert_ffn_rows(const moe_shape* s, const moe_weights* weights,
                                       int64_t n_rows, const void* u, const void* x_rows,
                                       const int32_t* expert_offsets, void* y_rows,
                                       void* y_shared, void* ws, size_t ws_bytes,
                                       moe_stream_t stream) {
  MOE_TRY(check_shape(s));
  if (n_rows < 0 || n_rows > INT_MAX / 2 ||
      static_cast<long long>(n_rows) + static_cast<long long>(s->T) * s->n_shared > INT_MAX / 2)
    return MOE_ERR_UNSUPPORTED;
  if (weights == nullptr) return MOE_ERR_INVALID_ARG;
  const bool sw = s->act == MOE_ACT_SWIGLU;
  if (!ok_ptr(weights->w1) || !ok_ptr(weights->w2) || (sw && !ok_ptr(weights->w3)))
    return MOE_ERR_INVALID_ARG;
  if (s->n_shared > 0 && s->T > 0 &&
      (!ok_ptr(weights->sw1) || !ok_ptr(weights->sw2) || (sw && !ok_ptr(weights->sw3))))
    return MOE_ERR_INVALID_ARG;
  if (!ok_ptr(expert_offsets)) return MOE_ERR_INVALID_ARG;
  if (n_rows > 0 && (!ok_ptr(x_rows) || !ok_ptr(y_rows))) return MOE_ERR_INVALID_ARG;
  if (s->n_shared > 0 && s->T > 0 && (!ok_ptr(u) || !ok_ptr(y_shared)))
    return MOE_ERR_INVALID_ARG;
  if (ws == nullptr || !al16(ws) || ws_bytes < ffn_ws_bytes(s, n_rows)) return MOE_ERR_WORKSPACE;
  return do_expert_ffn(s, weights, u, x_rows, expert_offsets, y_rows, y_shared, ws, cs(stream),
                       nullptr, nullptr, n_rows);
}

MOE_API moe_status moe_ep_regroup(const moe_shape* s, int32_t n_ranks, const int32_t* counts,
                                  int64_t n_rows, const void* src, void* dst,
                                  int32_t* expert_offsets, int32_t to_expert_major,
                                  moe_stream_t stream) {
  MOE_TRY(check_shape(s));
  if (n_ranks < 1 || static_cast<long long>(n_ranks) * s->n_routed > kRegroupThreads)
    return MOE_ERR_UNSUPPORTED;
  if (n_rows < 0 || n_rows > INT_MAX / 2) return MOE_ERR_UNSUPPORTED;
  if (!ok_ptr(counts) || !ok_opt(expert_offsets)) return MOE_ERR_INVALID_ARG;
  if (n_rows > 0 && (!ok_ptr(src) || !ok_ptr(dst))) return MOE_ERR_INVALID_ARG;
  const int blocks = std::max(1, std::min(cdiv(static_cast<int>(n_rows), kRegroupThreads / 32),
                                          2 * num_sms()));
  cudaStream_t st = cs(stream);
  const int tem = to_expert_major != 0;
  if (s->dtype == MOE_DTYPE_F32)
    ep_regroup_kernel<float><<<blocks, kRegroupThreads, 0, st>>>(
        counts, n_ranks, s->n_routed, s->H, static_cast<const float*>(src),
        static_cast<float*>(dst), expert_offsets, tem);
  else
    ep_regroup_kernel<__nv_bfloat16><<<blocks, kRegroupThreads, 0, st>>>(
        counts, n_ranks, s->n_routed, s->H, static_cast<const __nv_bfloat16*>(src),
        static_cast<__nv_bfloat16*>(dst), expert_offsets, tem);
  MOE_CUDA(cudaGetLastError());
  return MOE_OK;
}

MOE_API moe_status moe_layer_forward(const moe_shape* s, const moe_weights* weights,
                                     const void* u, void* h, const moe_route_outputs* route_out,
                                     void* ws, size_t ws_bytes, moe_stream_t stream) {
  return layer_forward(s, weights, u, h, route_out, ws, ws_bytes, cs(stream));
}

MOE_API size_t moe_layer_saved_size(const moe_shape* s) {
  if (check_shape(s) != MOE_OK || s->dtype != MOE_DTYPE_BF16) return 0;
  return carve_saved(nullptr, s).total;
}

MOE_API moe_status moe_layer_forward_train(const moe_shape* s, const moe_weights* weights,
                                           const void* u, void* h, void* saved,
                                           size_t saved_bytes, void* ws, size_t ws_bytes,
                                           moe_stream_t stream) {
  MOE_TRY(check_shape(s));
  if (s->dtype != MOE_DTYPE_BF16) return MOE_ERR_UNSUPPORTED;
  if (!ok_ptr(saved) || saved_bytes < carve_saved(nullptr, s).total) return MOE_ERR_INVALID_ARG;
  return layer_forward(s, weights, u, h, nullptr, ws, ws_bytes, cs(stream), saved);
}

MOE_API moe_status moe_layer_forward_host(const moe_shape* s, const moe_weights* weights,
                                          const void* u_host, void* h_host, void* u_dev,
                                          void* h_dev, void* ws, size_t ws_bytes,
                                          moe_stream_t stream) {
  MOE_TRY(check_shape(s));
  if (s->T > 0 && (u_host == nullptr || h_host == nullptr || !ok_ptr(u_dev) || !ok_ptr(h_dev)))
    return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_weights_ffn(s, weights));
  if (ws == nullptr || !al16(ws) || ws_bytes < carve_layer(nullptr, s).total)
    return MOE_ERR_WORKSPACE;
  cudaStream_t st = cs(stream);
  if (s->T == 0) return MOE_OK;
  const int n_chunks = host_chunks(s);
  if (n_chunks == 1) {
    const size_t bytes = static_cast<size_t>(s->T) * s->H * elt_bytes(s);
    MOE_CUDA(cudaMemcpyAsync(u_dev, u_host, bytes, cudaMemcpyHostToDevice, st));
    MOE_TRY(layer_forward(s, weights, u_dev, h_dev, nullptr, ws, ws_bytes, st));
    MOE_CUDA(cudaMemcpyAsync(h_host, h_dev, bytes, cudaMemcpyDeviceToHost, st));
    return MOE_OK;
  }
  // Token chunks in a pipeline: chunk c's host-to-device copy (stream `in`)
  // overlaps the layer on chunk c - 1 (the caller's stream) and the copy back
  // of chunk c - 2 (stream `out`).  Tokens are independent, so each chunk is
  // a layer call of its own; the workspace is reused chunk after chunk on the
  // caller's stream.
  CopyStreams cp;
  MOE_TRY(copy_streams(&cp));
  cudaEvent_t ev[3 * kMaxHostChunks];
  int n_ev = 0;
  moe_status status = MOE_OK;
  auto fail = [&](cudaError_t e) { status = cuda_fail(e); };
  for (int i = 0; i < 3 * n_chunks && status == MOE_OK; ++i) {
    const cudaError_t e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
    if (e != cudaSuccess) fail(e); else n_ev = i + 1;
  }
  // the copy streams first wait for whatever the caller queued before this call
  if (status == MOE_OK) {
    cudaError_t e = cudaEventRecord(ev[0], st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cp.in, ev[0], 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cp.out, ev[0], 0);
    if (e != cudaSuccess) fail(e);
  }
  const size_t row_bytes = static_cast<size_t>(s->H) * elt_bytes(s);
  const int per = (s->T + n_chunks - 1) / n_chunks;
  for (int c = 0; c < n_chunks && status == MOE_OK; ++c) {
    const int t0 = c * per, t1 = std::min(s->T, t0 + per);
    if (t1 <= t0) break;
    moe_shape sc = *s;
    sc.T = t1 - t0;
    const size_t off = static_cast<size_t>(t0) * row_bytes, bytes = (t1 - t0) * row_bytes;
    cudaEvent_t in_done = ev[3 * c], layer_done = ev[3 * c + 1], out_done = ev[3 * c + 2];
    cudaError_t e = cudaMemcpyAsync(static_cast<char*>(u_dev) + off,
                                    static_cast<const char*>(u_host) + off, bytes,
                                    cudaMemcpyHostToDevice, cp.in);
    if (e == cudaSuccess) e = cudaEventRecord(in_done, cp.in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, in_done, 0);
    if (e != cudaSuccess) { fail(e); break; }
    status = layer_forward(&sc, weights, static_cast<const char*>(u_dev) + off,
                           static_cast<char*>(h_dev) + off, nullptr, ws, ws_bytes, st);
    if (status != MOE_OK) break;
    e = cudaEventRecord(layer_done, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cp.out, layer_done, 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(static_cast<char*>(h_host) + off, static_cast<const char*>(h_dev) + off,
                          bytes, cudaMemcpyDeviceToHost, cp.out);
    if (e == cudaSuccess) e = cudaEventRecord(out_done, cp.out);
    // the caller's stream completes only after the last copy back
    if (e == cudaSuccess && c == n_chunks - 1) e = cudaStreamWaitEvent(st, out_done, 0);
    if (e != cudaSuccess) fail(e);
  }
  for (int i = 0; i < n_ev; ++i) cudaEventDestroy(ev[i]);  // released once they complete
  return status;
}

// Batches pipelined across calls' worth of tokens: batch b + 1's copy in
// (stream `in`) and batch b - 1's copy back (stream `out`) overlap batch b's
// layer (the caller's stream).  Two device slots of T rows each for u and
// h; a slot is refilled once the layer two batches back has read it (u) and
// its copy back has read it (h).
MOE_API moe_status moe_layer_forward_host_stream(const moe_shape* s, const moe_weights* weights,
                                                 int n_batches, const void* const* u_host,
                                                 void* const* h_host, void* u_dev, void* h_dev,
                                                 void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_shape(s));
  if (n_batches < 0) return MOE_ERR_INVALID_ARG;
  if (n_batches > 0 && s->T > 0) {
    if (u_host == nullptr || h_host == nullptr || !ok_ptr(u_dev) || !ok_ptr(h_dev))
      return MOE_ERR_INVALID_ARG;
    for (int b = 0; b < n_batches; ++b)
      if (u_host[b] == nullptr || h_host[b] == nullptr) return MOE_ERR_INVALID_ARG;
  }
  MOE_TRY(check_weights_ffn(s, weights));
  if (ws == nullptr || !al16(ws) || ws_bytes < carve_layer(nullptr, s).total)
    return MOE_ERR_WORKSPACE;
  if (n_batches == 0 || s->T == 0) return MOE_OK;
  cudaStream_t st = cs(stream);
  CopyStreams cp;
  MOE_TRY(copy_streams(&cp));
  const size_t bytes = static_cast<size_t>(s->T) * s->H * elt_bytes(s);
  // start, then per slot: copied in, layer done, copied back
  cudaEvent_t ev[7];
  int n_ev = 0;
  moe_status status = MOE_OK;
  for (int i = 0; i < 7 && status == MOE_OK; ++i) {
    const cudaError_t e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
    if (e != cudaSuccess) status = cuda_fail(e); else n_ev = i + 1;
  }
  cudaEvent_t start = ev[0];
  cudaEvent_t* in_done = ev + 1;
  cudaEvent_t* layer_done = ev + 3;
  cudaEvent_t* out_done = ev + 5;
  // the copy streams first wait for whatever the caller queued before this call
  if (status == MOE_OK) {
    cudaError_t e = cudaEventRecord(start, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cp.in, start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cp.out, start, 0);
    if (e != cudaSuccess) status = cuda_fail(e);
  }
  for (int b = 0; b < n_batches && status == MOE_OK; ++b) {
    const int slot = b & 1;
    char* u_slot = static_cast<char*>(u_dev) + slot * bytes;
    char* h_slot = static_cast<char*>(h_dev) + slot * bytes;
    cudaError_t e = cudaSuccess;
    if (b >= 2) e = cudaStreamWaitEvent(cp.in, layer_done[slot], 0);   // u slot read
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(u_slot, u_host[b], bytes, cudaMemcpyHostToDevice, cp.in);
    if (e == cudaSuccess) e = cudaEventRecord(in_done[slot], cp.in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, in_done[slot], 0);
    if (e == cudaSuccess && b >= 2) e = cudaStreamWaitEvent(st, out_done[slot], 0);  // h slot read
    if (e != cudaSuccess) { status = cuda_fail(e); break; }
    status = layer_forward(s, weights, u_slot, h_slot, nullptr, ws, ws_bytes, st);
    if (status != MOE_OK) break;
    e = cudaEventRecord(layer_done[slot], st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cp.out, layer_done[slot], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h_host[b], h_slot, bytes, cudaMemcpyDeviceToHost, cp.out);
    if (e == cudaSuccess) e = cudaEventRecord(out_done[slot], cp.out);
    if (e != cudaSuccess) status = cuda_fail(e);
  }
  // the caller's stream completes only after the last copies back
  if (status == MOE_OK) {
    cudaError_t e = cudaStreamWaitEvent(st, out_done[(n_batches - 1) & 1], 0);
    if (e == cudaSuccess && n_batches >= 2)
      e = cudaStreamWaitEvent(st, out_done[n_batches & 1], 0);
    if (e != cudaSuccess) status = cuda_fail(e);
  }
  for (int i = 0; i < n_ev; ++i) cudaEventDestroy(ev[i]);  // released once they complete
  return status;
}

// ---- moe_dispatch_static: dispatch with its scratch in a fixed array of the
// library, for callers that cannot hand the library any device memory.
// 2 x 131072 int32 = 1 MiB: chunk histograms and chunk bases of dispatch.
}  // extern "C"

namespace {

constexpr size_t kStaticDispatchEntries = 131072;  // ceil(T / 256) * n_routed
static __device__ __align__(256) int32_t g_static_dispatch_scratch[2 * kStaticDispatchEntries];

// Device address of the array in the current context, looked up once per
// device and context.  Host code cannot use the symbol itself as a device
// pointer.  The lookup is repeated when the device's current context is not
// the one the cached address was taken in (after cudaDeviceReset, or a
// primary context released and created again, the module can be loaded at
// another address).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

moe_status static_dispatch_scratch(void** out) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  static CUcontext ctx_of[64] = {nullptr};
  int dev = 0;
  MOE_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  if (get_ctx == nullptr) return cuda_fail(cudaErrorNotSupported);
  CUcontext ctx = nullptr;  // stays null while no context is current yet
  if (get_ctx(&ctx) != CUDA_SUCCESS) return cuda_fail(cudaErrorNotSupported);
  std::lock_guard<std::mutex> lock(mu);
  if (ctx == nullptr || addr[dev] == nullptr || ctx_of[dev] != ctx) {
    void* p = nullptr;
    // the runtime makes the device's primary context current here if needed
    MOE_CUDA(cudaGetSymbolAddress(&p, g_static_dispatch_scratch));
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cuda_fail(cudaErrorNotSupported);
    addr[dev] = p;
    ctx_of[dev] = ctx;
  }
  *out = addr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" {

MOE_API moe_status moe_dispatch_static(const moe_shape* s, const int32_t* topk_idx,
                                       const void* u, int32_t* expert_offsets,
                                       int32_t* row_token, int32_t* slot_row, void* u_perm,
                                       moe_stream_t stream) {
  MOE_TRY(check_shape(s));
  if (!ok_ptr(expert_offsets)) return MOE_ERR_INVALID_ARG;
  if (s->top_k > 0 && s->T > 0 && (!ok_ptr(topk_idx) || !ok_ptr(u) || !ok_ptr(row_token) ||
                                   !ok_ptr(slot_row) || !ok_ptr(u_perm)))
    return MOE_ERR_INVALID_ARG;
  const size_t entries = static_cast<size_t>(cdiv(s->T, kDispatchChunk)) * s->n_routed;
  if (entries > kStaticDispatchEntries) return MOE_ERR_UNSUPPORTED;
  // Both scratch arrays are fully written by the count and scan kernels (or
  // the memset for top_k == 0) before they are read: nothing needs clearing.
  void* scratch = nullptr;
  MOE_TRY(static_dispatch_scratch(&scratch));
  return do_dispatch(s, topk_idx, u, expert_offsets, row_token, slot_row, u_perm, scratch,
                     cs(stream));
}

}  // extern "C"
