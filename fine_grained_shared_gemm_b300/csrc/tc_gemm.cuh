// Grouped bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA)
// for the expert FFNs and the router logits of the MoE layer.
//
// Orientation ("swap-AB"): the weight rows are the MMA's M side and the token
// rows are its N side.  The ragged number of tokens each expert receives then
// only sets N, which the tensor core takes in steps of 16 (32 for a CTA
// pair), so a partly filled expert costs little extra work; decode-sized
// groups of one or two tokens run at N = 16 while the weights stream at full
// width.
//
//   D[j, c] = Σ_k W[j, k] · X[c, k]      (j: weight row, c: token of the group)
//
// Both operands are K-major in global memory (nn.Linear weights [out, in] and
// token rows [T, H]), land in shared memory through TMA with the 128-byte
// swizzle, and the fp32 accumulator lives in tensor memory (TMEM), double
// buffered so the epilogue of one tile overlaps the MMAs of the next.
//
// PAIR = 1: one CTA per tile of 128 weight rows x up to BN tokens.
// PAIR = 2: a cluster of two CTAs on two SMs shares one tile of 256 weight
//   rows x up to BN tokens through tcgen05.mma.cta_group::2.  Each CTA loads
//   its own 128 weight rows and HALF of the token rows; the tensor cores of
//   the pair exchange the token halves, so each SM pulls 16 KB of tokens per
//   k-block instead of 32 KB and the pipeline holds six stages instead of
//   four.  Each CTA's TMEM receives its own 128 rows of D.  The CTA of rank 0
//   (the leader) issues the MMAs; both CTAs' copies complete on the leader's
//   "full" barriers, and the leader's commits arrive on both CTAs' barriers.
//
// Roles (192 threads, one CTA per SM, persistent over tiles):
//   warp 0      TMA producer (one thread)
//   warp 1      TMEM allocation and (leader only) MMA issue (one thread)
//   warps 2..5  epilogue: TMEM -> registers (activation fused in) -> bf16
//               tile in shared memory -> TMA bulk store; fp32 outputs (router
//               logits, weight gradients) go straight from registers, one
//               128-byte row segment per warp store
//
// Every role decodes the same tile sequence from the per-group tile prefix,
// which is staged in shared memory.
//
// A pipeline stage holds two k-blocks (K = 128) and is filled by exactly two
// TMA copies: one for the weight tile and one for the token tile.  Each SM
// takes in at most ~50 bytes per clock through TMA, and a copy carries a fixed
// cost on top of its bytes, so few, large copies are what keep the tensor
// core fed.  The copies use tensor maps with a k-chunk dimension (stride
// 128 bytes) so that one box lands both k-blocks, one after the other, each
// in the 128-byte-swizzled K-major layout the MMA reads:
//   weights  3-D map (64 columns, rows, K/64 chunks), box 64 x 128 x 2;
//   SwiGLU   5-D map (64 columns, 64 rows, {W1, W3}, 64-row blocks, chunks)
//            whose third dimension steps from W1 to W3 (stride w3 - w1), so
//            one box lands [64 gate rows; 64 up rows] for both k-blocks;
//   tokens   3-D map, box 64 x R x 2 with R the next power of two >= the
//            rows the tile's MMA reads (extra rows are loaded, never used).
// A group's tokens are cut into full tiles of BN rows and one tail tile.  A
// chunk past the end of K is zero-filled by TMA and adds nothing.
//
// Every wait is bounded (kWaitLimitNs); on expiry the kernel sets a bit of the
// device error word, lets every role leave its loop, waits for its own copies
// and MMAs in flight, frees TMEM and returns.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace moe {
namespace tc {

constexpr int kBK = 64;            // contraction elements per k-block: one 128-byte swizzle row
constexpr int kKPS = 2;            // k-blocks per pipeline stage
constexpr int kBM = 128;           // weight rows per CTA per tile (MMA M per CTA)
constexpr int kUmmaK = 16;         // K of one tcgen05.mma for 16-bit inputs
constexpr int kABytes = kBM * kBK * 2;
constexpr int kNumBoxes = 5;       // token-tile TMA boxes of 16, 32, 64, 128, 256 rows
// Epilogue scratch per epilogue warp: two 2 KB staging tiles for bulk
// stores (32 x 32 bf16, or one 32 x 32 fp32 tile over both) and the SwiGLU
// hand-off area (16 x 33 floats).  With 7 KB a warp the 256-token pair tile
// still keeps three pipeline stages.
constexpr int kEpiWarpBytes = 7168;
// The SwiGLU-derivative epilogues keep 3.5 KB a warp: 16 rows of a chunk's a
// and c inputs, and 8 staged rows of its three outputs.  That leaves room for
// three pipeline stages beside eight epilogue warps.
constexpr int kBwdInBytes = 2 * 16 * 32 * 2;     // a and c, 16 rows x 32 features
constexpr int kBwdStageBytes = 3 * 8 * 32 * 2;   // da, dc, g act: 8 rows x 32 features
constexpr int kHandoffOffset = 4096;
constexpr int kSmemLimit = 232448; // dynamic shared memory per block, sm_100 family

// EPI_SWIGLU_BWD8 is EPI_SWIGLU_BWD with eight epilogue warps: for short
// contractions, where the derivative epilogue rather than the operand stream
// sets the pace.
enum Epi : int {
  EPI_SWIGLU = 0, EPI_RELU = 1, EPI_BF16 = 2, EPI_F32 = 3, EPI_SWIGLU_BWD = 4,
  EPI_SWIGLU_BWD8 = 5
};

__host__ __device__ constexpr bool is_swiglu_bwd(int epi) {
  return epi == EPI_SWIGLU_BWD || epi == EPI_SWIGLU_BWD8;
}

// Epilogue warps of a launch: four, one per TMEM lane quarter, or eight
// (two per quarter, taking alternate 32-row chunks).  Warp 0 loads, warp 1
// issues the MMAs, the rest are the epilogue.
template <int EPI>
__host__ __device__ constexpr int epi_warps() { return EPI == EPI_SWIGLU_BWD8 ? 8 : 4; }
template <int EPI>
__host__ __device__ constexpr int num_threads() { return 64 + 32 * epi_warps<EPI>(); }
// bytes of shared scratch per epilogue warp
template <int EPI>
__host__ __device__ constexpr int epi_warp_bytes() {
  return is_swiglu_bwd(EPI) ? kBwdInBytes + kBwdStageBytes : kEpiWarpBytes;
}

struct Params {
  CUtensorMap a[2];              // weight stacks (routed, shared): 3-D, or 5-D for SwiGLU
  // Weight operand layout.  0: K-major (the maps above are K-major).  1 or 2:
  // MN-major — the weights are read in their stored layout as the transpose
  // of the operand: expert e's operand element (m, k) lives at row
  // e · a_k_per_expert + k, column m of a row-major stack, and the map is
  // (64 columns, rows, column blocks of 64) [1], or for two stacks read one
  // after the other along k (W1 then W3) (64 columns, rows, 2 stacks, column
  // blocks) [2] with a_stack_chunks k-chunks per stack (a_stack_swap: the
  // map's first stack is the second one in k order).
  int a_mn;
  int a_mn_per_expert;           // operand rows (M) per expert: a_row0 = e · this
  int a_k_per_expert;
  int a_stack_chunks;
  int a_stack_swap[2];           // per weight stack (routed, shared)
  // With a_mn == 1, a_k_rows: the weight operand's k runs over rows of its
  // stored matrix starting at row krange.x (a row, not a k-chunk), so a
  // group's contraction can start at any row.
  int a_k_rows;
  // Token operand MN-major (b_mn): the token side is read in its stored
  // row-major layout as the transpose of the operand — operand element
  // (n, k) at row k, column n — through maps (64 columns, rows, column
  // blocks of 64) with a box of 64 columns x kKPS·64 rows x 2 blocks; a tile
  // is BN columns wide, or BN / 2 when it holds at most that many valid
  // columns and each CTA's half is still whole 64-column blocks (columns
  // past the matrix are zero-filled, only the valid ones are stored).
  // b_k_rows: k starts at row krange.y.
  int b_mn;
  int b_k_rows;
  CUtensorMap b[2][kNumBoxes];   // token sources x box heights: 3-D
  const GroupDesc* groups;       // [n_groups], or null for one dense group
  const int* tile_prefix;        // [n_groups + 1] prefix sum of token tiles
  int n_groups;                  // <= kMaxGroups
  int dense_count;               // token rows of the dense group
  int n_wtiles;                  // weight tiles (of 128 * PAIR rows) per group
  int num_k_blocks;              // ceil(K / kBK)
  // Optional per-group contraction range (null: every group runs k-chunks
  // [0, num_k_blocks) of both operands).  {x, y, z} = first k-chunk of the
  // weight operand, first k-chunk of the token operand, k-chunks (a multiple
  // of kKPS; 0 makes the tile's output zeros).  Used by the weight-gradient
  // GEMMs, whose contraction runs over each expert's own token rows.
  const int4* krange;
  // Dense group only (no krange): the contraction is cut into k_splits
  // ranges of k_split_blocks k-chunks (a multiple of kKPS; the last range
  // takes the rest).  Tile t computes range t / (n_wtiles · token tiles)
  // and writes it split_stride elements after the previous range's output
  // (plain or transposed fp32 stores, no f32_tma): partial sums that a
  // later pass adds in range order.
  int k_splits;
  int k_split_blocks;
  long long split_stride;
  // Tile order.  sched_heavy == 0: every cluster (CTA pair, or CTA) c of P
  // takes tiles c, c + P, c + 2P, ...  sched_heavy = nh > 0: tiles [0, nh)
  // are long ones (contractions several times the rest's), dealt round
  // robin first; the other tiles follow round robin too, but the nh mod P
  // clusters that drew one more long tile stop after sched_qb rounds while
  // the others go on, so every cluster ends with about the same work.
  int sched_heavy;
  int sched_qb;
  void* out[4];
  int out_ld;                    // output row pitch in elements
  int out_cols;                  // valid output columns
  int out_tr;                    // EPI_F32: store the transpose (out[col * out_ld + row])
  const float* col_offset;       // EPI_F32: per-column addend, may be null
  int up_first[2];               // SwiGLU, per stack: the 5-D map lands the up rows first
  CUtensorMap omap[2];           // bf16 outputs out[0], out[1]: 2-D, box 32 columns x 32 rows
  CUtensorMap omap16[2];         // the same outputs, box 32 columns x 16 rows (SwiGLU)
  // EPI_F32 with f32_tma: fp32 outputs out[0..3] as 2-D maps, box 32 x 32;
  // full 32-row chunks leave as bulk tensor stores
  int f32_tma;
  CUtensorMap omap32[4];
  // EPI_SWIGLU with save: also store the gate (save_out[0]) and up
  // (save_out[1]) pre-activations in bf16, same rows and columns as out
  int save;
  void* save_out[2];
  CUtensorMap save_map[2];
  // EPI_SWIGLU_BWD / EPI_SWIGLU_BWD8: the accumulator is dm = dh W2 for the tile's rows (the
  // output row space of the groups: out_row0 = the rows' index into the
  // pre-activations a, c [rows, out_cols], read through bwd_map[0] and
  // bwd_map[1], boxes of 32 columns x 32 rows; routed rows
  // [0, bwd_routed_rows) first).  Per row r and feature f, with g the routed
  // row's gate weight (1 for a shared row) and act = SiLU(a) ⊙ c:
  //   out[0] (dh1, [padded rows, 2·out_cols]):  da = g dm ⊙ c ⊙ SiLU'(a)
  //     at column f, dc = g dm ⊙ SiLU(a) at column out_cols + f;
  //   out[1] (g act, [padded rows, out_cols]):  g act at column f;
  //   bwd_dg[r · (out_cols / 32) + f / 32] = Σ over f's 32-feature block of
  //     dm ⊙ act (routed rows only).
  // The outputs sit in a padded row space: a group's rows start at its
  // GroupDesc.pad, and its rows past count up to the next multiple of
  // pad_rows are written as zeros.
  CUtensorMap bwd_map[2];
  const float* bwd_gate;
  float* bwd_dg;
  int bwd_routed_rows;
  int pad_rows;
};

constexpr int kMaxGroups = 1024;

template <int BN, int PAIR, int EPI_WARPS = 4, int EPI_WARP_BYTES = kEpiWarpBytes>
struct Config {
  static_assert(PAIR == 1 || PAIR == 2, "a tile is shared by one or two CTAs");
  static constexpr int kBRows = BN / PAIR;              // token rows one CTA holds
  static constexpr int kBBytes = kBRows * kBK * 2;      // one k-block of tokens
  static constexpr int kStageBytes = kKPS * (kABytes + kBBytes);
  static constexpr int kBarBytes = 512;                 // barriers, TMEM slot, descriptors
  static constexpr int kPrefixBytes = ((kMaxGroups + 4) * 4 + 127) / 128 * 128;
  static constexpr int kEpiBytes = EPI_WARPS * EPI_WARP_BYTES;
  static constexpr int kFit =
      (kSmemLimit - 1024 - kBarBytes - kPrefixBytes - kEpiBytes) / kStageBytes;
  static constexpr int kStages = kFit > 8 ? 8 : kFit;
  static constexpr int kSmemBytes =
      1024 + kStages * kStageBytes + kBarBytes + kPrefixBytes + kEpiBytes;
  static constexpr int kStep = 16 * PAIR;               // MMA N granularity
  static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;  // double-buffered accumulator
  static_assert(kStages >= 2, "pipeline too shallow");
  static_assert(kSmemBytes <= kSmemLimit, "shared memory over the sm_100-family limit");
  static_assert(BN % kStep == 0 && kBRows <= 256, "token tile");
};

// The configuration of one epilogue mode: the kernel and the host's launch
// (its dynamic shared memory) both take it from here.
template <int EPI, int BN, int PAIR>
using EpiConfig = Config<BN, PAIR, epi_warps<EPI>(), epi_warp_bytes<EPI>()>;

// ------------------------------------------------------------------ PTX

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in the CTA of the given rank.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Arrive on a barrier given by its shared::cluster address (own CTA or peer).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

template <bool kClusterScope>
__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  if (kClusterScope)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  return ok;
}

// Waits for the phase of the given parity to complete; false after the limit.
template <bool kClusterScope = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait<kClusterScope>(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 128; ++i)
      if (mbar_try_wait<kClusterScope>(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// Self-test of the bounded wait: one thread waits, with the GEMM's wait loop
// and the given limit, on a barrier phase that nothing completes; when the
// limit expires it sets `bits` in the device error word and returns.
__global__ void __launch_bounds__(32) wait_timeout_probe_kernel(uint64_t limit_ns, int bits) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_barrier_init();
  if (!mbar_wait(b, 0, limit_ns)) raise_device_error(bits);
}

// Tiled TMA loads into this CTA's shared memory, with an L2 cache policy
// (createpolicy).  With PAIR == 2 the completion is signalled on `bar`, a
// shared::cluster address that may be the peer CTA's barrier.
template <int PAIR>
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y, int z, uint64_t policy) {
  if (PAIR == 1)
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "l"(policy)
        : "memory");
  else
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile"
        ".mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "l"(policy)
        : "memory");
}

// A 2-D box pulled into L2 ahead of its load.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

// A 2-D box into this CTA's own shared memory, completion on its own barrier.
__device__ __forceinline__ void tma_load_2d_local(uint32_t dst, const CUtensorMap* map,
                                                  uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

template <int PAIR>
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2, int c3, uint64_t policy) {
  if (PAIR == 1)
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "l"(policy)
        : "memory");
  else
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile"
        ".mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "l"(policy)
        : "memory");
}

template <int PAIR>
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2, int c3, int c4,
                                            uint64_t policy) {
  if (PAIR == 1)
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(c4), "l"(policy)
        : "memory");
  else
    asm volatile(
        "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.tile"
        ".mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(c4), "l"(policy)
        : "memory");
}

// Bulk tensor store of a 32 x 32 bf16 box from this CTA's shared memory.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Until at most N committed groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// TMEM allocation: with PAIR == 2 one warp of each CTA of the pair issues it
// and both receive the same columns.
template <int PAIR>
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  if (PAIR == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  } else {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
}

template <int PAIR>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  if (PAIR == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(ncols)
                 : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row core-matrix groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>(1) << 16) |              // leading offset (unused when swizzled)
         (static_cast<uint64_t>(1024 >> 4) << 32) |      // stride offset between 8-row groups
         (static_cast<uint64_t>(1) << 46) |              // descriptor version
         (static_cast<uint64_t>(2) << 61);               // 128-byte swizzle
}

// Shared-memory matrix descriptor: MN-major operand, 128-byte swizzle.  The
// tile is stored as slabs of 64 M-elements (128 bytes) x K rows; 8-row
// groups along K are 1024 bytes apart (stride offset) and the slabs of
// consecutive 64-element M blocks are `slab` bytes apart (leading offset).
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t saddr, uint32_t slab) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>(slab >> 4) << 16) |      // leading offset: next M slab
         (static_cast<uint64_t>(1024 >> 4) << 32) |      // stride offset: next 8 K rows
         (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, each operand
// K-major or (a_mn, b_mn) MN-major.  m is the MMA's full M (256 for a CTA pair).
__device__ __forceinline__ uint32_t idesc_bf16(uint32_t m, uint32_t n, uint32_t a_mn = 0,
                                               uint32_t b_mn = 0) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (a_mn << 15) | (b_mn << 16) | ((n >> 3) << 17) |
         ((m >> 4) << 24);
}

template <int PAIR>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  if (PAIR == 1)
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on `bar` when all MMAs issued so far by this thread complete.
// PAIR == 2: on the barrier at the same offset in both CTAs of the pair.
template <int PAIR>
__device__ __forceinline__ void tc_commit_all(uint32_t bar) {
  if (PAIR == 1) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
  } else {
    const uint16_t mask = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar), "h"(mask)
        : "memory");
  }
}

// Arrive on this CTA's `bar` only.
template <int PAIR>
__device__ __forceinline__ void tc_commit_local(uint32_t bar) {
  if (PAIR == 1)
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
  else
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// 32 consecutive fp32 accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
        "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
        "=r"(v[31])
      : "r"(taddr));
  // The wait names the registers so that no use of them is scheduled before it.
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]),
        "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]),
        "+r"(v[13]), "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]),
        "+r"(v[19]), "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]), "+r"(v[24]),
        "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]), "+r"(v[30]),
        "+r"(v[31])
      :
      : "memory");
}

// tanh by the hardware approximation (one MUFU operation).
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// SiLU(x) = x · sigmoid(x), with sigmoid(x) = (1 + tanh(x / 2)) / 2:
// h + h · tanh(h) for h = x / 2.
__device__ __forceinline__ float silu_tanh(float x) {
  const float h = 0.5f * x;
  return fmaf(h, tanh_approx(h), h);
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also returns the AND of `pred` over the participants.
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// ------------------------------------------------------------------ tiles

__device__ __forceinline__ int box_index(int rows) {
  return rows <= 16 ? 0 : rows <= 32 ? 1 : rows <= 64 ? 2 : rows <= 128 ? 3 : 4;
}

// One tile as seen by one CTA (of rank `rank` in its pair).
struct Tile {
  int a_sel, a_row;      // weight stack and this CTA's first weight row
  int a_base;            // the group's first weight row (a_row0)
  int b_src, b_row;      // token source and this CTA's first token row
  int b_rows;            // token rows this CTA's half of the MMA reads (multiple of 16)
  int b_box;             // box index: the copy lands 16 << b_box >= b_rows rows
  int n_mma;             // MMA N: token rows of the whole tile, rounded up
  int out_sel, out_row;  // output buffer and the tile's first output row
  int out_col;           // this CTA's first output column
  int n_valid;           // valid token rows of the tile
  int nt;                // token tiles of the tile's group
  int ka0, kb0, nk;      // first k-chunk of each operand, k-chunks
  int split;             // contraction range of a dense split-K launch
  int prow;              // EPI_SWIGLU_BWD: the tile's first row in the padded row space
  int pad_end;           // EPI_SWIGLU_BWD: rows written (valid, then zero padding)
};

// Group of tile t (0 for a dense group).
__device__ __forceinline__ int group_of(const Params& p, const int* prefix, int t) {
  if (p.groups == nullptr) return 0;
  int lo = 0, hi = p.n_groups;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] * p.n_wtiles <= t) lo = mid; else hi = mid;
  }
  return lo;
}

// prefix: the tile prefix staged in shared memory (unused for a dense group).
template <int EPI, int BN, int PAIR>
__device__ __forceinline__ Tile decode_tile(const Params& p, const int* prefix, int t, int rank) {
  constexpr int kStep = Config<BN, PAIR>::kStep;
  const int nw = p.n_wtiles;
  GroupDesc d;
  int nt, local, lo = 0, split = 0;
  if (p.groups == nullptr) {
    d = GroupDesc{0, 0, 0, 0, 0, 0, p.dense_count, 0};
    nt = (p.dense_count + BN - 1) / BN;
    local = t;
    if (p.k_splits > 1) {
      split = t / (nw * nt);
      local = t - split * (nw * nt);
    }
  } else {
    int hi = p.n_groups;  // largest g with prefix[g] * nw <= t
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] * nw <= t) lo = mid; else hi = mid;
    }
    d = p.groups[lo];
    nt = prefix[lo + 1] - prefix[lo];
    local = t - prefix[lo] * nw;
  }
  // Token tile major within a group: the weight tiles of one token tile are
  // consecutive.  With weight-tile-major order and an even number of
  // clusters, a group's tiles of one token-tile position all went to the
  // clusters of one parity: dW1/dW3's half-width last column tiles (I =
  // 1408) left the odd clusters 17 % short of work (1100 -> 1033 us).
  const int n = local / nw, w = local - n * nw;
  const int th = BN;  // full tiles of BN rows, then the tail
  constexpr int kCols = (EPI == EPI_SWIGLU) ? kBM / 2 : kBM;  // output columns per CTA
  Tile tl;
  tl.a_sel = d.a_sel;
  tl.a_base = d.a_row0;
  tl.a_row = d.a_row0 + (w * PAIR + rank) * kCols;
  tl.n_valid = min(th, d.count - n * th);
  tl.n_mma = (tl.n_valid + kStep - 1) / kStep * kStep;
  tl.nt = nt;
  // MN-major tokens: whole 64-column blocks per CTA
  constexpr bool kHalfMN = (BN / 2 / PAIR) % 64 == 0;
  if (p.b_mn) tl.n_mma = (kHalfMN && tl.n_valid <= BN / 2) ? BN / 2 : BN;
  tl.b_rows = tl.n_mma / PAIR;
  tl.b_box = box_index(tl.b_rows);
  tl.b_src = d.b_src;
  tl.b_row = d.b_row0 + n * th + rank * tl.b_rows;
  tl.out_sel = d.out_sel;
  tl.out_row = d.out_row0 + n * th;
  tl.out_col = (w * PAIR + rank) * kCols;
  tl.split = split;
  if (is_swiglu_bwd(EPI)) {
    tl.prow = d.pad + n * th;
    tl.pad_end = n == nt - 1 ? (d.count + p.pad_rows - 1) / p.pad_rows * p.pad_rows - n * th : th;
  }
  if (p.krange != nullptr) {
    const int4 kr = __ldg(p.krange + lo);
    tl.ka0 = kr.x;
    tl.kb0 = kr.y;
    tl.nk = kr.z;
  } else if (p.k_splits > 1) {
    tl.ka0 = tl.kb0 = split * p.k_split_blocks;
    tl.nk = max(0, min(p.k_split_blocks, p.num_k_blocks - tl.ka0));
  } else {
    tl.ka0 = tl.kb0 = 0;
    tl.nk = p.num_k_blocks;
  }
  return tl;
}

// Tile of iteration i of cluster c of P (Params.sched_heavy), or -1 past the
// cluster's last.  Every role of both CTAs walks the same sequence.
__device__ __forceinline__ int sched_tile(const Params& p, int c, int P, int total, int i) {
  if (p.sched_heavy <= 0) {
    const int t = c + i * P;
    return t < total ? t : -1;
  }
  const int nh = p.sched_heavy;
  const int hc = nh > c ? (nh - 1 - c) / P + 1 : 0;  // long tiles c, c + P, ...
  if (i < hc) return c + i * P;
  const int k = i - hc, r = nh % P, qb = p.sched_qb;
  int idx;                                            // among the other tiles
  if (k < qb) idx = k * P + c;                        // rounds every cluster takes
  else if (c < r) return -1;                          // drew one more long tile
  else idx = qb * P + (k - qb) * (P - r) + (c - r);   // rounds of the other P - r
  return idx < total - nh ? nh + idx : -1;
}

// ------------------------------------------------------------------ kernel

template <int EPI, int BN, int PAIR>
__global__ void __launch_bounds__(num_threads<EPI>(), 1)
    grouped_gemm_kernel(const __grid_constant__ Params p) {
  using C = EpiConfig<EPI, BN, PAIR>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t bar0 = base + S * C::kStageBytes;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 128u + 8u * s; };
  auto tfull_bar = [&](int a) { return bar0 + 256u + 8u * a; };
  auto tempty_bar = [&](int a) { return bar0 + 272u + 8u * a; };
  const uint32_t done_bar = bar0 + 288u;
  // EPI_SWIGLU_BWD: each epilogue warp's input-tile barrier (by staging slot)
  auto ld_bar = [&](int slot) { return bar0 + 320u + 8u * slot; };
  uint8_t* bar_area = smem + S * C::kStageBytes;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_area + 296);
  int* s_prefix = reinterpret_cast<int*>(bar_area + C::kBarBytes);
  uint8_t* epi_area = bar_area + C::kBarBytes + C::kPrefixBytes;

  {
    // the layout above must fit the launch's allocation: a launch that
    // disagrees reports it and does nothing (every CTA of a cluster sees
    // the same size, so none waits on a partner that has left)
    uint32_t dyn;
    asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    if (dyn < static_cast<uint32_t>(C::kSmemBytes)) {
      if (threadIdx.x == 0) raise_device_error(DEV_ERR_SMEM_SHORT);
      return;
    }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR == 2 ? cluster_rank() : 0u;
  const int first = PAIR == 2 ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int stride = PAIR == 2 ? static_cast<int>(num_clusters_x()) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), epi_warps<EPI>() * PAIR);  // lane 0 of each epilogue warp of each CTA
    }
    mbar_init(done_bar, 1);
    if (is_swiglu_bwd(EPI))
      for (int e = 0; e < epi_warps<EPI>(); ++e) mbar_init(ld_bar(e), 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < 2; ++i) {
      prefetch_map(&p.a[i]);
    }
  }
  if (p.groups != nullptr)
    for (int i = threadIdx.x; i <= p.n_groups; i += blockDim.x) s_prefix[i] = __ldg(p.tile_prefix + i);
  if (warp == 1) tmem_alloc<PAIR>(smem_u32(tmem_slot), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  if (PAIR == 2) cluster_sync();  // the peer's barriers are initialised before any use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int tiles_per_w = (p.groups == nullptr) ? (p.dense_count + BN - 1) / BN
                                                : s_prefix[p.n_groups];
  const int total = p.n_wtiles * tiles_per_w * (p.k_splits > 1 ? p.k_splits : 1);

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, armed = 0, last_parity = 0;
      bool ok = true;
      // L2 policy: a weight tile that only one token tile reads is streamed
      // through (evict first); one that several token tiles read, and the
      // token rows (read by every weight tile of their group), stay (evict last)
      const uint64_t pol_once = l2_policy_evict_first(), pol_keep = l2_policy_evict_last();
      for (int i = 0; ok; ++i) {
        const int t = sched_tile(p, first, stride, total, i);
        if (t < 0) break;
        const Tile tl = decode_tile<EPI, BN, PAIR>(p, s_prefix, t, rank);
        const uint64_t pol_a = tl.nt > 1 ? pol_keep : pol_once;
        // token rows each CTA's copy lands per k-block (MN-major: BN / PAIR
        // columns, the same bytes)
        const int b_land = p.b_mn ? C::kBRows : 16 << tl.b_box;
        // bytes both CTAs' copies deliver to the leader's barrier per stage
        const uint32_t bytes =
            static_cast<uint32_t>(PAIR * kKPS) * (kABytes + static_cast<uint32_t>(b_land) * (kBK * 2));
        // MN-major weights: the expert, its first k row and this CTA's first
        // 64-column block
        const int a_e = p.a_mn ? tl.a_base / p.a_mn_per_expert : 0;
        const int a_k0 = a_e * p.a_k_per_expert;
        const int a_mb = p.a_mn ? (tl.a_row - tl.a_base) / 64 : 0;
        const CUtensorMap* bmap = &p.b[tl.b_src][tl.b_box];
        for (int kb = 0; kb < tl.nk; kb += kKPS) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1)) {
            raise_device_error(DEV_ERR_TIMEOUT_PRODUCER);
            ok = false;
            break;
          }
          const uint32_t sa = base + stage * C::kStageBytes;
          uint32_t fb = full_bar(stage);
          if (rank == 0) {
            mbar_arrive_expect_tx(fb, bytes);
            armed |= 1u << stage;
            last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          }
          if (PAIR == 2) fb = map_to_rank(fb, 0);
          // weights: both k-blocks in one copy (chunk kb and kb + 1)
          if (EPI == EPI_SWIGLU) {
            tma_load_5d<PAIR>(sa, &p.a[tl.a_sel], fb, 0, 0, 0, tl.a_row / (kBM / 2), tl.ka0 + kb,
                              pol_a);
          } else if (p.a_mn == 1) {
            // 128 k rows x two 64-column blocks: [block][row][64]
            const int row = p.a_k_rows ? tl.ka0 + kb * kBK : a_k0 + (tl.ka0 + kb) * kBK;
            tma_load_3d<PAIR>(sa, &p.a[tl.a_sel], fb, 0, row, a_mb, pol_a);
          } else if (p.a_mn == 2) {
            const int c = tl.ka0 + kb;  // k-chunk pairs never straddle the two stacks
            const int stack = (c >= p.a_stack_chunks) != (p.a_stack_swap[tl.a_sel] != 0) ? 1 : 0;
            const int row = a_k0 + (c >= p.a_stack_chunks ? c - p.a_stack_chunks : c) * kBK;
            tma_load_4d<PAIR>(sa, &p.a[tl.a_sel], fb, 0, row, stack, a_mb, pol_a);
          } else {
            tma_load_3d<PAIR>(sa, &p.a[tl.a_sel], fb, 0, tl.a_row, tl.ka0 + kb, pol_a);
          }
          // tokens: both k-blocks in one copy
          if (p.b_mn) {
            const int row = p.b_k_rows ? tl.kb0 + kb * kBK : (tl.kb0 + kb) * kBK;
            tma_load_3d<PAIR>(sa + kKPS * kABytes, &p.b[tl.b_src][0], fb, 0, row, tl.b_row / 64,
                              pol_keep);
          } else {
            tma_load_3d<PAIR>(sa + kKPS * kABytes, bmap, fb, 0, tl.b_row, tl.kb0 + kb, pol_keep);
          }
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
      }
      // No copy may land after the CTA exits: the leader waits for the last
      // armed phase of every stage (which also covers the peer's copies).
      if (rank == 0)
        for (int s = 0; s < S; ++s)
          if ((armed >> s) & 1u)
            if (!mbar_wait(full_bar(s), (last_parity >> s) & 1u))
              raise_device_error(DEV_ERR_TIMEOUT_PRODUCER);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // TMEM holds two accumulator slots of BN columns, taken in turn, so the
    // epilogue of one tile overlaps the next tile's MMAs.
    if (lane == 0 && rank == 0) {
      int stage = 0, a0 = 0;
      uint32_t phase = 0, acc_ph[2] = {0u, 0u};
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const int t = sched_tile(p, first, stride, total, i);
        if (t < 0) break;
        const Tile tl = decode_tile<EPI, BN, PAIR>(p, s_prefix, t, 0);
        if (!mbar_wait<PAIR == 2>(tempty_bar(a0), acc_ph[a0] ^ 1)) {
          raise_device_error(DEV_ERR_TIMEOUT_MMA);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a0 * BN);
        const uint32_t idesc =
            idesc_bf16(kBM * PAIR, static_cast<uint32_t>(tl.n_mma), p.a_mn != 0 ? 1u : 0u,
                       p.b_mn != 0 ? 1u : 0u);
        const uint32_t boff = static_cast<uint32_t>(16 << tl.b_box) * (kBK * 2);
        for (int kb = 0; kb < tl.nk; kb += kKPS) {
          if (!mbar_wait(full_bar(stage), phase)) {
            raise_device_error(DEV_ERR_TIMEOUT_MMA);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + stage * C::kStageBytes;
          // a chunk past the end of K was zero-filled: its MMAs add nothing
#pragma unroll
          for (int c = 0; c < kKPS; ++c) {
            // K-major A: k-block c is the c-th 16 KB block, a 16-element k
            // step is 32 bytes along the row.  MN-major A: two slabs of
            // kKPS * 64 rows x 128 bytes; k-block c starts 64 rows into each
            // slab, a k step is 16 rows (2 KB).
            const uint64_t da = p.a_mn ? sdesc_sw128_mn(sa + c * (kBK * 128), kKPS * kBK * 128)
                                       : sdesc_sw128(sa + c * kABytes);
            const uint32_t a_step = p.a_mn ? (kUmmaK * 128) >> 4 : 2;
            // K-major B: k-block c is boff bytes further; MN-major B: like
            // MN-major A (two slabs of kKPS·64 rows, k-block c 64 rows in)
            const uint64_t db = p.b_mn ? sdesc_sw128_mn(sa + kKPS * kABytes + c * (kBK * 128),
                                                         kKPS * kBK * 128)
                                       : sdesc_sw128(sa + kKPS * kABytes + c * boff);
            const uint32_t b_step = p.b_mn ? (kUmmaK * 128) >> 4 : 2;
#pragma unroll
            for (int k = 0; k < kBK / kUmmaK; ++k)
              tc_mma<PAIR>(d_tmem, da + a_step * k, db + b_step * k, idesc, ((kb + c) | k) != 0);
          }
          tc_commit_all<PAIR>(empty_bar(stage));  // frees the stage in both CTAs once read
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit_all<PAIR>(tfull_bar(a0));
        acc_ph[a0] ^= 1u;
        a0 ^= 1;
      }
      // All MMAs issued by this thread complete before TMEM is freed.
      tc_commit_local<PAIR>(done_bar);
      if (!mbar_wait(done_bar, 0)) raise_device_error(DEV_ERR_TIMEOUT_MMA);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;  // the TMEM lane quarter this warp may read
    // with eight epilogue warps, the second warp of a quarter takes the odd chunks
    const int ehalf = (warp - 2) >> 2;
    const int eslot = q + 4 * ehalf;  // this warp's staging area and input barrier
    constexpr int kChunkStride = 32 * (epi_warps<EPI>() / 4);
    float* buf = reinterpret_cast<float*>(epi_area + eslot * epi_warp_bytes<EPI>());
    // SwiGLU hand-off: this warp's area and its partner's
    float* hand = reinterpret_cast<float*>(epi_area + q * kEpiWarpBytes + kHandoffOffset);
    const float* other_hand =
        reinterpret_cast<const float*>(epi_area + (q ^ 2) * kEpiWarpBytes + kHandoffOffset);
    // the leader's accumulator-free barriers, as shared::cluster addresses
    const uint32_t tempty_leader0 = PAIR == 2 ? map_to_rank(tempty_bar(0), 0) : tempty_bar(0);
    const uint32_t tempty_leader1 = PAIR == 2 ? map_to_rank(tempty_bar(1), 0) : tempty_bar(1);
    int a0 = 0;
    uint32_t acc_ph[2] = {0u, 0u};
    uint32_t n_stores = 0;  // bulk stores this warp has issued (selects the staging buffer)
    // SwiGLU derivative: 16 rows of a chunk's a and c land in this warp's
    // scratch (a at [0, 1 KB), c at [1 KB, 2 KB)) on ld_bar(eslot); 8 rows of
    // the three outputs are staged at [2 KB, 3.5 KB) for 16-byte stores;
    // lane L holds the gate weight of row L of the next chunk
    uint16_t* ostg = reinterpret_cast<uint16_t*>(buf) + kBwdInBytes / 2;
    float gate_next = 1.0f;
    auto load_gate = [&](const Tile& tl, int c0) {
      const long long r = static_cast<long long>(tl.out_row) + c0 + lane;
      gate_next = (c0 + lane < tl.n_valid && r < p.bwd_routed_rows) ? __ldg(p.bwd_gate + r) : 1.0f;
    };
    uint32_t ld_ph = 0;
    bool ld_pending = false, ld_failed = false;
    auto load_inputs = [&](int col, int row) {
      if (lane == 0) {
        mbar_arrive_expect_tx(ld_bar(eslot), static_cast<uint32_t>(kBwdInBytes));
        tma_load_2d_local(smem_u32(buf), &p.bwd_map[0], ld_bar(eslot), col, row);
        tma_load_2d_local(smem_u32(buf) + kBwdInBytes / 2, &p.bwd_map[1], ld_bar(eslot), col,
                          row);
      }
      ld_pending = true;
    };
    // this warp has read accumulator slot a: tell the leader's MMA issuer
    auto release = [&](int a) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR == 2) mbar_arrive_cluster(a ? tempty_leader1 : tempty_leader0);
        else mbar_arrive(tempty_bar(a));
      }
      acc_ph[a] ^= 1u;
    };
    for (int i = 0;; ++i) {
      const int t = sched_tile(p, first, stride, total, i);
      if (t < 0) break;
      const Tile tl = decode_tile<EPI, BN, PAIR>(p, s_prefix, t, rank);
      // the first chunk's first 16 input rows are on their way while the MMAs run
      const int c_first = 32 * ehalf;  // this warp's first chunk
      const bool bwd_active = is_swiglu_bwd(EPI) && !ld_failed &&
                              tl.out_col + q * 32 < p.out_cols && c_first < tl.n_valid;
      if (bwd_active) {
        const int f0 = tl.out_col + q * 32;
        if (lane == 0)   // this warp's chunks' a and c boxes (16 rows each) into L2
          for (int c0 = c_first; c0 < tl.n_valid; c0 += kChunkStride)
            for (int r = c0; r < c0 + 32 && r < tl.n_valid; r += 16) {
              tma_prefetch_2d(&p.bwd_map[0], f0, tl.out_row + r);
              tma_prefetch_2d(&p.bwd_map[1], f0, tl.out_row + r);
            }
        load_inputs(f0, tl.out_row + c_first);
        load_gate(tl, c_first);
      }
      const bool ready = mbar_wait(tfull_bar(a0), acc_ph[a0]);
      // all four epilogue warps leave together, so no named barrier is left half-arrived
      if (!named_bar_and(1, 32 * epi_warps<EPI>(), ready)) {
        if (!ready) raise_device_error(DEV_ERR_TIMEOUT_EPILOGUE);
        break;
      }
      tc_fence_after();
      const bool cols_ok = tl.out_col < p.out_cols;  // a CTA half past the last row stores nothing
      const uint32_t tlane = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      // One chunk: the 32 accumulator columns from TMEM column `col` hold
      // the tile's token rows c0 .. c0 + 31 (those below n_valid are stored).
      // Every epilogue warp runs the same chunks (the SwiGLU hand-off below
      // synchronises them).
      auto chunk = [&](int col, int c0) {
        if (c0 >= tl.n_valid) return;
        uint32_t v[32];
        tmem_ld32(tlane + static_cast<uint32_t>(col), v);
        const int nrow = min(32, tl.n_valid - c0);  // token rows of this chunk
        // A full chunk of 32 tokens goes out as one bulk store from a bf16
        // tile in this warp's shared memory (two buffers, alternating; the
        // store issued two chunks ago must have read the buffer); a partial
        // chunk is stored from registers, so no box writes past the group.
        auto emit_to = [&](const CUtensorMap* map, void* base, auto value_of, int col_base) {
          if (!cols_ok) return;
          if (nrow == 32) {
            uint16_t* stg = reinterpret_cast<uint16_t*>(buf) + (n_stores & 1) * 1024;
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 32; ++j)
              stg[j * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(value_of(j)));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(map, smem_u32(stg), tl.out_col + col_base, tl.out_row + c0);
              bulk_commit();
            }
            ++n_stores;
          } else {
            __nv_bfloat16* o = static_cast<__nv_bfloat16*>(base) +
                               static_cast<size_t>(tl.out_row + c0) * p.out_ld + tl.out_col +
                               col_base + lane;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nrow) o[static_cast<size_t>(j) * p.out_ld] = __float2bfloat16_rn(value_of(j));
          }
        };
        auto emit = [&](auto value_of, int col_base) {
          emit_to(&p.omap[tl.out_sel], p.out[tl.out_sel], value_of, col_base);
        };
        // 16 token rows [row0, row0 + 16) of the chunk: a full half leaves as
        // one 32 x 16 bulk store, a partial one from registers
        auto emit16 = [&](auto value_of, int row0, int col_base) {
          if (!cols_ok) return;
          const int mrows = min(16, nrow - row0);
          if (mrows <= 0) return;
          if (mrows == 16) {
            uint16_t* stg = reinterpret_cast<uint16_t*>(buf) + (n_stores & 1) * 1024;
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 16; ++j)
              stg[j * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(value_of(j)));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&p.omap16[tl.out_sel], smem_u32(stg), tl.out_col + col_base,
                           tl.out_row + c0 + row0);
              bulk_commit();
            }
            ++n_stores;
          } else {
            __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out[tl.out_sel]) +
                               static_cast<size_t>(tl.out_row + c0 + row0) * p.out_ld +
                               tl.out_col + col_base + lane;
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (j < mrows) o[static_cast<size_t>(j) * p.out_ld] = __float2bfloat16_rn(value_of(j));
          }
        };
        if (EPI == EPI_SWIGLU) {
          // lanes 0..63 hold the gate rows and 64..127 the matching up rows
          // (the other way round when the map lands W3 first): warp q and
          // its partner q ^ 2 hold the gate and the up values of the same 32
          // output columns.  They split the chunk's tokens: the gate warp
          // computes tokens [0, 16) and hands the gate values of [16, 32) to
          // the up warp, which computes [16, 32) and hands over the up values
          // of [0, 16).  Each warp then stores its 16 rows.
          const bool gate_warp = (q < 2) != (p.up_first[tl.a_sel] != 0);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            hand[i * 33 + lane] = __uint_as_float(gate_warp ? v[16 + i] : v[i]);
          named_bar_sync(1, 128);
          // the partner's values into registers, so that the hand-off area
          // is free again at the second barrier
          float pv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pv[i] = other_hand[i * 33 + lane];
          named_bar_sync(1, 128);
          emit16([&](int i) {
            const float g = gate_warp ? __uint_as_float(v[i]) : pv[i];
            const float up = gate_warp ? pv[i] : __uint_as_float(v[16 + i]);
            return silu_tanh(g) * up;
          }, gate_warp ? 0 : 16, (q & 1) * 32);
          // in the training forward each warp also stores the pre-activation
          // it holds (gate or up, same output columns as its partner's) for a
          // later backward
          if (p.save)
            emit_to(&p.save_map[gate_warp ? 0 : 1], p.save_out[gate_warp ? 0 : 1],
                    [&](int j) { return __uint_as_float(v[j]); }, (q & 1) * 32);
        } else if (EPI == EPI_F32) {
          // lane = output column: for each token row j the warp writes 32
          // consecutive fp32 columns (128 bytes) of that row
          const int col = tl.out_col + q * 32 + lane;
          const bool col_ok = cols_ok && col < p.out_cols;
          const float add =
              (p.col_offset != nullptr && col_ok) ? __ldg(p.col_offset + col) : 0.0f;
          if (col_ok && p.out_tr) {
            // transposed: this lane's 32 token rows are 32 consecutive floats
            float* o = static_cast<float*>(p.out[tl.out_sel]) + tl.split * p.split_stride +
                       static_cast<size_t>(col) * p.out_ld + tl.out_row + c0;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nrow) o[j] = tl.nk == 0 ? 0.0f : __uint_as_float(v[j]) + add;
          } else if (p.f32_tma && nrow == 32 && cols_ok && tl.out_col + q * 32 < p.out_cols) {
            // one 32 x 32 box per chunk from this warp's staging tile (single
            // buffer: the previous store must have read it); columns past
            // out_cols are clipped by the tensor map
            float* stg = buf;
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 32; ++j)
              stg[j * 32 + lane] = tl.nk == 0 ? 0.0f : __uint_as_float(v[j]) + add;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&p.omap32[tl.out_sel], smem_u32(stg), tl.out_col + q * 32,
                           tl.out_row + c0);
              bulk_commit();
            }
          } else if (col_ok) {
            float* o = static_cast<float*>(p.out[tl.out_sel]) + tl.split * p.split_stride +
                       static_cast<size_t>(tl.out_row + c0) * p.out_ld + col;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nrow)
                o[static_cast<size_t>(j) * p.out_ld] =
                    tl.nk == 0 ? 0.0f : __uint_as_float(v[j]) + add;
          }
        } else {
          emit([&](int j) {
            const float x = __uint_as_float(v[j]);
            return EPI == EPI_RELU ? fmaxf(x, 0.0f) : x;
          }, q * 32);
          if (EPI == EPI_RELU && p.save)  // the pre-activation too, for a later backward
            emit_to(&p.save_map[0], p.save_out[0], [&](int j) { return __uint_as_float(v[j]); },
                    q * 32);
        }
      };
      if constexpr (is_swiglu_bwd(EPI)) {
        // This lane's feature f0 + lane, 32 token rows per chunk: dm from
        // the accumulator; a and c 16 rows at a time from the input tile (the
        // next 16 rows are requested as soon as these are read); da / dc /
        // g act staged 8 rows at a time and stored as 16-byte vectors;
        // <dm, act> summed over the warp's 32 features.  Rows past the
        // tile's valid rows (its group's padding) are zeros.
        const int f0 = tl.out_col + q * 32;
        if (cols_ok && f0 < p.out_cols) {
          const int nf = p.out_cols;
          const uint16_t* in = reinterpret_cast<const uint16_t*>(buf);
          for (int c0 = c_first; c0 < tl.pad_end; c0 += kChunkStride) {
            const int nrow = max(0, min(32, tl.n_valid - c0));
            const long long r0 = static_cast<long long>(tl.out_row) + c0;
            float dm[32];
            const float g_lane = gate_next;
            load_gate(tl, c0 + kChunkStride);  // the next chunk's, in flight during this one
            uint32_t v[32];
            if (nrow > 0) tmem_ld32(tlane + static_cast<uint32_t>(a0 * BN + c0), v);
#pragma unroll
            for (int j = 0; j < 32; ++j) dm[j] = j < nrow ? __uint_as_float(v[j]) : 0.0f;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int hrow = nrow - 16 * h;  // valid rows among this half's 16
              float av[16], cv[16];
              if (hrow > 0 && !ld_failed) {
                if (!mbar_wait(ld_bar(eslot), ld_ph)) {
                  raise_device_error(DEV_ERR_TIMEOUT_EPILOGUE);
                  ld_failed = true;
                } else {
                  ld_ph ^= 1u;
                  ld_pending = false;
                }
              }
              if (hrow > 0 && !ld_failed) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  av[j] = j < hrow ? __bfloat162float(__ushort_as_bfloat16(in[j * 32 + lane])) : 0.0f;
                  cv[j] = j < hrow ? __bfloat162float(__ushort_as_bfloat16(in[512 + j * 32 + lane]))
                                   : 0.0f;
                }
                // every lane's reads of the tile are ordered before the async
                // proxy refills it
                fence_proxy_async_smem();
                __syncwarp();
                // next: this chunk's second half, or the warp's next chunk
                const int next = h == 0 ? c0 + 16 : c0 + kChunkStride;
                if (next < tl.n_valid) load_inputs(f0, tl.out_row + next);
              } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) av[j] = cv[j] = 0.0f;
              }
              // 8 rows at a time: the three outputs into the staging tiles,
              // then out as 16-byte vectors (4 lanes per 64-byte row segment)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                  const int k = e * 8 + jj;   // row within the half
                  const int j = h * 16 + k;   // row within the chunk
                  const float g = __shfl_sync(0xffffffffu, g_lane, j);
                  // sigmoid(a) = (1 + tanh(a / 2)) / 2, as in the forward's SiLU
                  const float sg = fmaf(0.5f, tanh_approx(0.5f * av[k]), 0.5f);
                  const float si = av[k] * sg;
                  const float act = si * cv[k];
                  const float gd = g * dm[j];
                  ostg[jj * 32 + lane] = __bfloat16_as_ushort(
                      __float2bfloat16_rn(gd * cv[k] * sg * (1.0f + av[k] * (1.0f - sg))));
                  ostg[256 + jj * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(gd * si));
                  ostg[512 + jj * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(g * act));
                  dm[j] *= act;  // this lane's share of <dm, act> for row j
                }
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 3; ++i) {
                  const int vi = i * 32 + lane;        // 16-byte vector: output, row, 8 columns
                  const int o = vi >> 5, row = (vi >> 2) & 7, c8 = (vi & 3) * 8;
                  const uint4 val = *reinterpret_cast<const uint4*>(ostg + o * 256 + row * 32 + c8);
                  // outputs 0, 1: dh1's da and dc halves (pitch 2·nf); 2: g act
                  __nv_bfloat16* const base =
                      static_cast<__nv_bfloat16*>(o < 2 ? p.out[0] : p.out[1]) + (o == 1 ? nf : 0);
                  const size_t pitch = o < 2 ? 2 * static_cast<size_t>(nf) : static_cast<size_t>(nf);
                  *reinterpret_cast<uint4*>(
                      base + static_cast<size_t>(tl.prow + c0 + h * 16 + e * 8 + row) * pitch + f0 +
                      c8) = val;
                }
                __syncwarp();  // the staging tiles are read before the next rows fill them
              }
            }
            // sum over the 32 lanes, scattered so that lane j ends with row j
#pragma unroll
            for (int sh = 16; sh >= 1; sh >>= 1) {
              const bool up = (lane & sh) != 0;
#pragma unroll
              for (int i2 = 0; i2 < sh; ++i2) {
                const float send = up ? dm[i2] : dm[i2 + sh];
                const float keep = up ? dm[i2 + sh] : dm[i2];
                dm[i2] = keep + __shfl_xor_sync(0xffffffffu, send, sh);
              }
            }
            if (lane < nrow && r0 + lane < p.bwd_routed_rows)
              p.bwd_dg[static_cast<size_t>(r0 + lane) * (nf / 32) + f0 / 32] = dm[0];
          }
        }
      } else {
        // column c of the slot holds token row c of the tile (one call site
        // keeps the chunk body inlined once)
        for (int c0 = 0; c0 < tl.n_valid; c0 += 32) chunk(a0 * BN + c0, c0);
      }
      release(a0);
      a0 ^= 1;
    }
    // no input tile may land after the CTA exits
    if (is_swiglu_bwd(EPI) && ld_pending && !mbar_wait(ld_bar(eslot), ld_ph))
      raise_device_error(DEV_ERR_TIMEOUT_EPILOGUE);
    if (lane == 0) bulk_wait_all();  // every bulk store has completed before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (PAIR == 2) cluster_sync();  // neither CTA leaves while the pair may still touch it
  tc_fence_after();
  if (warp == 1) tmem_dealloc<PAIR>(tmem_base, C::kTmemCols);
}

}  // namespace tc
}  // namespace moe
