// prefill_tc.cuh -- multi-query attention over the paged cache on the 5th-
// generation tensor cores (tcgen05): the last n tokens of a sequence of L
// cached tokens query the cache, which already holds their keys and values
// (Attention.lean `causalGQA` / `slidingGQA` with S > 1): query i sits at
// position p = L - n + i and sees key l iff l <= p (and p - window < l with
// a window); scale 1; query head c*G + g reads KV head c.
//
// Work item (tile, c * kSlices + slice, b): 128 rows = kQ = 128 / G queries
// of sequence b times the G query heads of KV head c, row r being head r / kQ
// of query r % kQ; `slice` selects which kDS of the D output dims it writes
// (D = 512 is split in two so that O fits in tensor memory).  Per step of
// kPPS pages (N = 16 kPPS keys):
//   S   = Q K^T    tcgen05.mma M=128, N=16 kPPS, K=D, A = Q (K-major: in
//                  tensor memory, copied there from its 128-byte-swizzled
//                  shared-memory tile, or read from that tile), B = the
//                  step's K tile as TMA wrote it; accumulator in tensor
//                  memory, two buffers;
//   P   = softmax  warps 0-3 (and a second warpgroup for the second half of
//                  the keys), one thread per row (TMEM lane = row): masks,
//                  running max, P rounded to bf16 into tensor memory (or
//                  shared memory as K-major core matrices);
//   O  += P V      tcgen05.mma M=128, N=kDS, K=16, B = the V tile, MN-major
//                  with the 128-byte swizzle; accumulator O in tensor memory.
// Warp 4 copies Q and the K tiles by TMA; warps 5 .. 4 + kIssuers issue the
// S products, each a part of the k-steps (the whole warp runs the loop, one
// elected lane issues), and warp 5 allocates tensor memory; the next warp
// issues every P V product and the one after it copies the V tiles; with two
// softmax warpgroups the last four warps handle the second half of every
// row.  S of step j+1 is computed while the softmax of step j runs, and P V
// of step j while the softmax of step j+1 runs.
//
// Running max.  A row's reference max m moves only when a score exceeds it by
// more than kSlack = 64 log2 units, and then to kHeadroom = 48 above that
// score.  So every weight exp2(s - m) is at most 2^64, the row's largest is
// at least 2^-48, and only keys more than 78 log2 units below the row max
// (relative weight < 2^-78) flush to zero.  A row sum over at most 2^17 keys
// stays below 2^81 and O below 2^81 max|v|: inside fp32 (and P inside bf16)
// for any |v| < 2^46.  Numerator and denominator share m, so the result is
// the same softmax.  O is rescaled in tensor memory only when m moves, and a
// warp rescales if any of its 32 rows moves: it waits for the previous P V
// and round-trips its rows of O, so each rescale stalls the softmax.  A
// row's first keys (the window edge) estimate its max poorly; with scores of
// standard deviation 16 (unit-variance q and k, D = 256, scale 1) a band of
// 2^8 and no headroom made about half of the steps rescale, 2^16 with the
// headroom 9 %, and 2^64 almost none.  The rescale loads 64 columns per
// tensor-memory round trip.  Key rows outside [k_lo, k_hi] of the first and last page are
// zeroed in shared memory before P V (0 * NaN would be NaN); masked scores
// become -inf.
#pragma once

#include "common.cuh"
#include "tcgen05.cuh"

namespace pda {
namespace prefill_tc {

struct PrefillParams {
  const __nv_bfloat16* q;      // [total_q, Hq, D]
  const int32_t* block_table;  // [batch, max_blocks]
  const int32_t* seq_lens;     // [batch]
  const int32_t* cu_q;         // [batch + 1]
  void* o;                     // [total_q, Hq, D], bf16 or fp32
  int32_t* status;             // optional ATTN_DEV_* word
  int64_t num_pages;
  int32_t batch;
  int32_t max_blocks;
  int32_t window;  // > 0: sliding window; <= 0: none
  int32_t total_q;
  int32_t max_q;  // queries past max_q of a sequence are not computed (and flagged)
  int32_t out_f32;
};

// 3-D tile copy without a cache hint: every query tile of a sequence reads the
// same pages, so they should stay in L2 as long as possible.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

// 4-D tile copy: Q as {64 dims, chunk, query, head}; a box {64, 1, kQ, G}
// lands as [head][query][128 B], the tile's row order.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                            int32_t w, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_addr(bar))
      : "memory");
}

// 4-D tile store from shared memory (the same box shape as tma_load_4d), in
// the issuing thread's bulk async-group.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, const void* src, int32_t x, int32_t y, int32_t z,
                                             int32_t w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_addr(src)), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until this thread's bulk stores have read their shared memory ...
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// ... or have completed.
__device__ __forceinline__ void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

template <int kD_, int kDS_, int kG_, int kHkv_, int kStages_, int kPPS_, bool kPInTmem_, int kIssuers_ = 1,
          int kSoftmaxGroups_ = 1, int kRotate_ = 0, int kSBufs_ = 2, int kPBufs_ = 2, bool kQInTmem_ = false,
          int kVStages_ = kStages_, bool kPInS_ = false>
struct Config {
  static constexpr int kD = kD_;    // head dim (the contraction of S)
  static constexpr int kDS = kDS_;  // output dims per block
  static constexpr int kG = kG_;
  static constexpr int kHkv = kHkv_;
  static constexpr int kHq = kG * kHkv;
  // K and V tiles in two rings, each filled by its own producer warp: a K
  // tile is released when its S products are done, a V tile only when its
  // P V product is, so K runs further ahead than it could in a shared ring.
  static constexpr int kStages = kStages_;    // K tiles
  static constexpr int kVStages = kVStages_;  // V tiles
  static constexpr int kPPS = kPPS_;                 // pages per step
  static constexpr bool kPInTmem = kPInTmem_;        // P in tensor memory (else shared memory)
  static constexpr int kKeys = kPPS * kPage;         // keys per step: N of S, K of P V
  static constexpr int kSlices = kD / kDS;
  static constexpr int kRows = 128;
  static constexpr int kQ = kRows / kG;  // queries per block
  static constexpr int kKChunks = kD / 64;
  static constexpr int kVChunks = kDS / 64;
  static constexpr int kQChunkBytes = kRows * 128;  // [128 rows][64 dims]
  static constexpr int kChunkRows = kKeys * 128;     // one K chunk of a step: [kKeys rows][64 dims]
  static constexpr int kChunkBytes = kPage * 128;    // one chunk of one page: [16 rows][64 dims]
  static constexpr int kVPage = kVChunks * kChunkBytes;  // one page of V: one TMA box
  static constexpr int kKTile = kKChunks * kChunkRows;
  static constexpr int kVTile = kPPS * kVPage;
  static constexpr int kPBytes = kRows * kKeys * 2;
  // Threads issuing the S products: one MMA instruction costs its issuing
  // thread about 70 cycles whatever its size, so the D k-steps of a step are
  // split into kIssuers parts, each accumulated into its own S buffer (the
  // softmax adds them).  Warps 5 .. 4 + kIssuers issue the parts, and warp
  // 5 + kIssuers every P V product, so no S product waits behind a P.
  static constexpr int kIssuers = kIssuers_;
  // Softmax warpgroups: with two, each row's keys of a step are split in
  // halves (warps 0-3 the first, warps 7 + kIssuers .. 10 + kIssuers the
  // second), and so are its output dims.
  static constexpr int kSoftmaxGroups = kSoftmaxGroups_;
  static constexpr int kSoftmaxThreads = 128 * kSoftmaxGroups;
  // Step order: with kRotate > 0 the block of query tile t starts at step
  // (kRotate t) mod n_steps and wraps around, so that the blocks resident at
  // one time read different pages (the softmax does not depend on the order
  // of the keys).
  static constexpr int kRotate = kRotate_;
  // S and P buffers in tensor memory: S runs up to kSBufs steps ahead of the
  // softmax, P V may lag it by kPBufs - 1 steps.
  static constexpr int kSBufs = kSBufs_;
  static constexpr int kPBufs = kPBufs_;
  static constexpr int kThreads = (4 * kSoftmaxGroups + 3 + kIssuers) * 32;
  static constexpr int kPVWarp = 5 + kIssuers;     // the P V issuer
  static constexpr int kVProdWarp = 6 + kIssuers;  // the V producer; softmax warpgroups 1.. follow it
  static constexpr uint32_t kTmemCols = 512;
  // Q as the A operand of S in tensor memory (copied from its shared-memory
  // tile once per item) instead of shared memory: an S product with N = 32
  // then reads 1 KB of shared memory instead of 5 KB.
  static constexpr bool kQInTmem = kQInTmem_;
  static constexpr uint32_t kQCol = kDS;  // Q (bf16 pairs): kD / 2 columns
  static constexpr uint32_t kSCol = kDS + (kQInTmem ? kD / 2 : 0);  // S buffers: column kSCol + kKeys (kIssuers buffer + part)
  static constexpr uint32_t kPCol = kSCol + kSBufs * kIssuers * kKeys;  // P buffers (bf16 pairs), kKeys / 2 columns each
  // P written over its own S buffer (the first kKeys / 2 columns): no P
  // buffers, and an S buffer is free again once the P V product of its step
  // is done (committed by the P V issuer) instead of once S is read.
  static constexpr bool kPInS = kPInS_;
  __device__ static constexpr uint32_t p_col(int b) {
    return kPInS ? kSCol + kKeys * b : kPCol + (kKeys / 2) * b;
  }
  static constexpr uint32_t kIdescS = umma_idesc_bf16(128, kKeys, 0, 0);
  static constexpr uint32_t kIdescPV = umma_idesc_bf16(128, kDS, 0, 1);
  static_assert(kRows % kG == 0 && kD % 64 == 0 && kDS % 64 == 0 && kDS <= 256, "tile shapes");
  static_assert(!kPInS || (kPInTmem && kIssuers == 1 && kPBufs == kSBufs), "P over S: one S part per buffer");
  static_assert(kPCol + (kPInTmem && !kPInS ? kPBufs * kKeys / 2 : 0) <= kTmemCols,
                "O, Q, the S buffers and P fit in tensor memory");
  static_assert(kPInTmem || kPBufs == 2, "P in shared memory: two buffers");
  static_assert(kKeys % 16 == 0 && kKeys <= 256, "N of S");
  static_assert(kIssuers >= 1 && kIssuers <= kD / 16, "S k-steps split among the issuers");
  static_assert(kSoftmaxGroups == 1 ||
                    ((kSoftmaxGroups == 2 || kSoftmaxGroups == 4) && kPInTmem && (kKeys / kSoftmaxGroups) % 8 == 0 &&
                     (kDS / kSoftmaxGroups) % 64 == 0),
                "two softmax warpgroups: halves of whole 16-key blocks, P in tensor memory");

  struct Smem {
    alignas(1024) uint8_t q[kKChunks][kQChunkBytes];
    alignas(1024) uint8_t k[kStages][kKTile];
    alignas(1024) uint8_t v[kVStages][kVTile];
    alignas(128) uint8_t p[kPInTmem ? 1 : 2][kPInTmem ? 16 : kPBytes];
    // one 64-dim chunk of O in bf16, staged for a TMA store (with Q in tensor
    // memory, the Q tile's buffer stages all of O instead)
    alignas(1024) uint8_t ost[kQInTmem ? 16 : kRows * 128];
    alignas(8) uint64_t full[kStages];     // K tile landed (TMA)
    alignas(8) uint64_t empty[kStages];    // its S products done (one commit per issuer)
    alignas(8) uint64_t v_full[kVStages];   // V tile landed (TMA)
    alignas(8) uint64_t v_empty[kVStages];  // its P V product done (commit)
    alignas(8) uint64_t s_full[kSBufs];   // S buffer written (commit)
    alignas(8) uint64_t s_free[kSBufs];   // S buffer read (the softmax warps), or with P over S its P V done (commit)
    alignas(8) uint64_t p_full[kPBufs];   // P buffer written, O rescaled, V edges zeroed (the softmax warps)
    alignas(8) uint64_t p_empty[kPBufs];  // P V of the buffer's step done (commit)
    alignas(8) uint64_t q_ready;         // the item's Q tile landed (TMA)
    alignas(8) uint64_t q_empty;         // the item's Q tile read: its S products done, or copied to tensor memory
    alignas(8) uint64_t q_tfree[kIssuers];  // Q in tensor memory: issuer i's S products of the item done
    alignas(8) uint64_t ost_free;           // Q in tensor memory: the item's output stores have read the Q buffer
    alignas(8) uint64_t o_full;          // the item's last P V done (commit)
    alignas(8) uint64_t o_free;          // O read by the item's epilogue (the softmax warps)
    alignas(8) uint64_t mma_done;        // every MMA done (commit)
    uint32_t tmem_base;
    float half_max[2][kSoftmaxGroups][kRows];  // several warpgroups: each part-row's max, by step parity
    float half_sum[kSoftmaxGroups][kRows];     // and its share of the row sum, at the end
  };
  static constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "one CTA per SM within the 227 KB a CTA may have");
};

// Maximum and sum of v[0 .. N) by pairwise halving: log2 N dependent steps
// instead of N - 1 (N a power of two).
template <int N>
__device__ __forceinline__ float tree_max(const float* v) {
  static_assert((N & (N - 1)) == 0, "a power of two");
  float t[N];
#pragma unroll
  for (int k = 0; k < N; ++k) t[k] = v[k];
#pragma unroll
  for (int w = N / 2; w >= 1; w /= 2)
#pragma unroll
    for (int k = 0; k < w; ++k) t[k] = fmaxf(t[k], t[k + w]);
  return t[0];
}
template <int N>
__device__ __forceinline__ float tree_sum(const float* v) {
  static_assert((N & (N - 1)) == 0, "a power of two");
  float t[N];
#pragma unroll
  for (int k = 0; k < N; ++k) t[k] = v[k];
#pragma unroll
  for (int w = N / 2; w >= 1; w /= 2)
#pragma unroll
    for (int k = 0; k < w; ++k) t[k] += t[k + w];
  return t[0];
}

constexpr float kSlack = 64.f;     // log2 units
constexpr float kHeadroom = 48.f;  // a moved reference max sits this far above the row's max
constexpr int kRoundTrip = 4;     // 16-column TMEM loads per wait when O is rescaled or written

// 16 bytes global -> shared without a register round trip; src_bytes 0
// writes zeros (src is then not read).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// kN consecutive 32-bit columns of this thread's lane (kN a multiple of 8);
// complete after tmem_wait_ld.
template <int kN>
__device__ __forceinline__ void load_row(uint32_t taddr, float (&v)[kN]) {
  static_assert(kN % 8 == 0, "whole 8-column loads");
  if constexpr (kN % 16 == 0) {
#pragma unroll
    for (int b = 0; b < kN / 16; ++b) tmem_ld16(taddr + 16 * b, *reinterpret_cast<float(*)[16]>(&v[16 * b]));
  } else {
#pragma unroll
    for (int b = 0; b < kN / 8; ++b) tmem_ld8(taddr + 8 * b, *reinterpret_cast<float(*)[8]>(&v[8 * b]));
  }
}

// One work item (a query tile of one sequence, KV head and output slice) as
// every role of the CTA sees it.
struct TileItem {
  bool run;
  int c, slice, b, tile;  // KV head, output slice, sequence, query tile
  int q0, i0, nq, P0;     // first packed query row, the tile's first query, its valid queries, its first position
  int k_lo, k_hi;         // keys the tile sees (inclusive)
  int page0, n_pages, n_steps, rot;
};

template <typename C>
__device__ __forceinline__ TileItem load_tile(const PrefillParams& p, int w, int tiles, bool reporter) {
  constexpr int kQ = C::kQ, kPPS = C::kPPS;
  TileItem it{};
  it.tile = w % tiles;
  const int rest = w / tiles;
  const int y = rest % (C::kHkv * C::kSlices);
  it.b = rest / (C::kHkv * C::kSlices);
  it.c = y / C::kSlices;
  it.slice = y % C::kSlices;
  it.q0 = p.cu_q[it.b];
  const int n = p.cu_q[it.b + 1] - it.q0;
  it.i0 = it.tile * kQ;
  const int L = p.seq_lens[it.b];
  const int cap = p.max_blocks < ATTN_MAX_SEQ_LEN / kPage ? p.max_blocks * kPage : ATTN_MAX_SEQ_LEN;
  it.run = false;
  if (n < 0 || it.q0 < 0 || static_cast<int64_t>(it.q0) + n > p.total_q) {
    if (reporter) report(p.status, ATTN_DEV_BAD_SEQ_LEN);
    return it;
  }
  if (n > p.max_q && it.tile == 0 && y == 0 && reporter)
    report(p.status, ATTN_DEV_BAD_SEQ_LEN);  // more queries than the host's max_q: the rest are not computed
  const int n_run = n < p.max_q ? n : p.max_q;
  if (it.i0 >= n_run) return it;
  if (L < n || L > cap) {
    if (reporter) report(p.status, ATTN_DEV_BAD_SEQ_LEN);
    return it;
  }
  it.run = true;
  it.nq = n_run - it.i0 < kQ ? n_run - it.i0 : kQ;
  it.P0 = L - n + it.i0;
  it.k_hi = it.P0 + it.nq - 1;
  it.k_lo = p.window > 0 ? (it.P0 - p.window + 1 > 0 ? it.P0 - p.window + 1 : 0) : 0;
  it.page0 = it.k_lo / kPage;
  it.n_pages = it.k_hi / kPage - it.page0 + 1;
  it.n_steps = (it.n_pages + kPPS - 1) / kPPS;
  it.rot = C::kRotate > 0 ? static_cast<int>((static_cast<int64_t>(it.tile) * C::kRotate) % it.n_steps) : 0;
  return it;
}

// step j of the copy order covers logical step (j + rot) mod n_steps
__device__ __forceinline__ int tile_step(const TileItem& it, int j) {
  return j + it.rot < it.n_steps ? j + it.rot : j + it.rot - it.n_steps;
}

// A value every lane of the warp holds, marked as such for the compiler, so
// that MMA descriptors derived from it stay in uniform registers.
__device__ __forceinline__ int warp_uniform_int(int v) { return __shfl_sync(0xffffffffu, v, 0); }

// The grid holds one CTA per work item, or fewer (one per SM) that loop over
// the items: work item w = tile + tiles * (c * kSlices + slice + Hkv kSlices b),
// CTA g taking g, g + gridDim.x, ...  Every pipeline (stages, S and P
// buffers) runs on counters that continue from one item to the next, so the
// next item's Q and pages stream in, and its first S products run, while the
// last item's softmax and epilogue finish.  Q is one buffer, refilled once
// the item's S products are done (q_empty); O passes from an item's epilogue
// to the next item's first P V product through o_full / o_free.
template <typename C>
__global__ void __launch_bounds__(C::kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
                      const __grid_constant__ PrefillParams p) {
  constexpr int kD = C::kD, kDS = C::kDS, kG = C::kG, kHq = C::kHq, kQ = C::kQ, kStages = C::kStages;
  constexpr int kPPS = C::kPPS;
  extern __shared__ uint8_t smem_raw[];
  typename C::Smem& s =
      *reinterpret_cast<typename C::Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles = (p.max_q + kQ - 1) / kQ;
  const int n_work = tiles * C::kHkv * C::kSlices * p.batch;

  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&s.full[st], 1);
      mbar_init(&s.empty[st], C::kIssuers);
    }
    for (int st = 0; st < C::kVStages; ++st) {
      mbar_init(&s.v_full[st], 1);
      mbar_init(&s.v_empty[st], 1);
    }
    for (int i = 0; i < C::kSBufs; ++i) {
      mbar_init(&s.s_full[i], C::kIssuers);
      mbar_init(&s.s_free[i], C::kPInS ? 1 : 4 * C::kSoftmaxGroups);
    }
    for (int i = 0; i < C::kPBufs; ++i) {
      mbar_init(&s.p_full[i], 4 * C::kSoftmaxGroups);
      mbar_init(&s.p_empty[i], 1);
    }
    mbar_init(&s.q_ready, 1);
    mbar_init(&s.q_empty, C::kIssuers);
    for (int i = 0; i < C::kIssuers; ++i) mbar_init(&s.q_tfree[i], 1);
    mbar_init(&s.ost_free, 1);
    mbar_init(&s.o_full, 1);
    mbar_init(&s.o_free, 4 * C::kSoftmaxGroups);
    mbar_init(&s.mma_done, C::kIssuers + 1);
    fence_mbar_init();
  }
  if (warp == 4 && lane == 0) {
    prefetch_tensor_map(&tm_k);
    prefetch_tensor_map(&tm_v);
    prefetch_tensor_map(&tm_q);
  }
  if (warp == 5) tmem_alloc(&s.tmem_base, C::kTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = s.tmem_base;

  // q, the cache and the tables may be written by the previous kernel in the stream.
  wait_for_primary_grid();
  allow_dependent_launch();

  if (warp == 4 || warp == C::kVProdWarp) {
    // ---------------- producers: warp 4 each item's Q and its K tiles, the V producer its V tiles ----------------
    // Lane ch < D/64 copies chunk ch of Q (G heads x kQ queries in one box;
    // queries past the tile's own are copied too and masked by the softmax,
    // queries past total_q read as zeros).  Lane pg < kPPS copies page pg of
    // a step (K chunk by chunk, so that the step's pages sit contiguously in
    // each [kKeys rows][64 dims] chunk).  Pages past the range (the last
    // step) and bad page ids are copied from a fully out-of-range row: zeros.
    static_assert(32 % kPPS == 0, "a step's pages in one batch of 32 table entries");
    static_assert(C::kKChunks <= 32, "one lane per Q chunk");
    const bool kw = warp == 4;  // the K producer
    const int n_slots = kw ? kStages : C::kVStages;
    uint64_t* const fullb = kw ? s.full : s.v_full;
    uint64_t* const emptyb = kw ? s.empty : s.v_empty;
    bool ok = true;
    int gs = 0, gt = 0;  // steps and items issued
    for (int w = blockIdx.x; w < n_work && ok; w += gridDim.x) {
      const TileItem it = load_tile<C>(p, w, tiles, lane == 0 && kw);
      if (!it.run) continue;
      if (kw) {
        if (gt >= 1) {  // the previous item's Q tile read
          int wq = lane == 0 ? static_cast<int>(mbar_wait_fast(&s.q_empty, (gt - 1) & 1)) : 0;
          // with Q in tensor memory the buffer also stages the output of the
          // item before the previous one
          if (C::kQInTmem && gt >= 2 && wq) wq = lane == 0 ? static_cast<int>(mbar_wait_fast(&s.ost_free, (gt - 2) & 1)) : 0;
          ok = __shfl_sync(0xffffffffu, wq, 0) != 0;
          if (!ok) break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&s.q_ready, C::kKChunks * C::kQChunkBytes);
        __syncwarp();
        if (lane < C::kKChunks) tma_load_4d(s.q[lane], &tm_q, 0, lane, it.q0 + it.i0, it.c * kG, &s.q_ready);
      }
      ++gt;
      const int32_t* bt = p.block_table + static_cast<int64_t>(it.b) * p.max_blocks;
      // block-table entry of the page copied at position gp of the order
      const auto entry = [&](int gp) {
        const int lp = tile_step(it, gp / kPPS) * kPPS + gp % kPPS;
        return gp < it.n_steps * kPPS && lp < it.n_pages ? bt[it.page0 + lp] : -1;
      };
      // block-table entries of pages 32k + lane (in copy order), one batch ahead
      int cur = entry(lane);
      int nxt = entry(32 + lane);
      for (int i = 0; i < it.n_steps; ++i) {
        const int gp0 = i * kPPS;
        if (gp0 > 0 && (gp0 & 31) == 0) {
          cur = nxt;
          nxt = entry(gp0 + 32 + lane);
        }
        const int phys = __shfl_sync(0xffffffffu, cur, (gp0 + (lane < kPPS ? lane : 0)) & 31);
        const int stage = gs % n_slots;
        if (gs >= n_slots) {
          const int wv = lane == 0 ? static_cast<int>(mbar_wait_fast(&emptyb[stage], ((gs / n_slots) - 1) & 1)) : 0;
          ok = __shfl_sync(0xffffffffu, wv, 0) != 0;
        }
        if (!ok) break;
        if (lane == 0) mbar_arrive_expect_tx(&fullb[stage], kw ? C::kKTile : C::kVTile);
        __syncwarp();
        if (lane < kPPS) {
          const int gp = tile_step(it, i) * kPPS + lane;
          int32_t y = -kPage;
          if (gp < it.n_pages) {
            if (phys < 0 || static_cast<int64_t>(phys) >= p.num_pages)
              report(p.status, ATTN_DEV_BAD_PAGE);
            else
              y = phys * kPage;
          }
          if (kw) {
#pragma unroll
            for (int ch = 0; ch < C::kKChunks; ++ch)
              tma_load_3d(s.k[stage] + ch * C::kChunkRows + lane * (kPage * 128), &tm_k, 0, y,
                          it.c * C::kKChunks + ch, &fullb[stage]);
          } else {
            tma_load_3d(s.v[stage] + lane * C::kVPage, &tm_v, 0, y, it.c * C::kKChunks + it.slice * C::kVChunks,
                        &fullb[stage]);
          }
        }
        ++gs;
        __syncwarp();
      }
    }
    if (!ok && lane == 0) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
    if (lane == 0) {  // no copy may still be landing, nor a commit arriving, when the CTA retires
      if (kw && gt >= 1) {
        if (!mbar_wait(&s.q_ready, (gt - 1) & 1)) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
        if (ok && !mbar_wait(&s.q_empty, (gt - 1) & 1)) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
      }
      for (int st = 0; st < n_slots && st < gs; ++st) {
        const int uses = (gs - 1 - st) / n_slots + 1;
        if (!mbar_wait(&fullb[st], (uses - 1) & 1)) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
        if (ok && !mbar_wait(&emptyb[st], (uses - 1) & 1)) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
      }
    }
  } else if (warp >= 5 && warp < 5 + C::kIssuers) {
    // ---------------- S issuers (whole warps; an elected lane issues): part i of the k-steps ----------------
    // Stage and S buffer indices advance by one per step, with their phase
    // parities, and the loop bounds are broadcast from lane 0: the
    // descriptors then stay in uniform registers.  S waits only for its
    // stage and a free S buffer, never for P.
    constexpr int kPart = (kD / 16) / C::kIssuers;  // k-steps per issuer, whole 64-dim chunks
    static_assert(kPart % 4 == 0, "each issuer takes whole chunks of Q and K");
    const int part = warp - 5;
    bool ok = true;
    int gt = 0, g = 0;  // items done, steps done
    int st = 0, st_ph = 0, sb = 0, sb_ph = 0;
    const uint32_t q_base = smem_addr(s.q[0]) + (part * kPart / 4) * C::kQChunkBytes;
    for (int w = blockIdx.x; w < n_work; w += gridDim.x) {
      const TileItem it = load_tile<C>(p, w, tiles, false);
      if (!warp_uniform_int(it.run)) continue;
      const int n_steps = warp_uniform_int(it.n_steps);
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.q_ready, gt & 1));
      if constexpr (C::kQInTmem) {
        // this issuer's k-steps of Q into tensor memory, once its S products
        // of the previous item have read the columns
        if (ok && gt >= 1) ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.q_tfree[part], (gt - 1) & 1));
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < kPart; ++kk)
          tmem_cp_128x256b_warp(tmem + C::kQCol + 8 * (part * kPart + kk),
                                umma_desc(q_base + (kk >> 2) * C::kQChunkBytes + (kk & 3) * 32, 16, 1024, 2));
        umma_commit_warp(&s.q_empty);  // the shared-memory tile may take the next item's Q
      }
      for (int j = 0; j < n_steps; ++j) {
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.full[st], st_ph));
        if (ok && g >= C::kSBufs) ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.s_free[sb], sb_ph ^ 1));
        tc_fence_after_sync();
        const uint32_t k_base = smem_addr(s.k[st]) + (part * kPart / 4) * C::kChunkRows;
#pragma unroll
        for (int kk = 0; kk < kPart; ++kk) {
          const uint64_t b_desc = umma_desc(k_base + (kk >> 2) * C::kChunkRows + (kk & 3) * 32, 16, 1024, 2);
          const uint32_t d_tmem = tmem + C::kSCol + C::kKeys * (C::kIssuers * sb + part);
          if constexpr (C::kQInTmem) {
            umma_bf16_ts_warp(d_tmem, tmem + C::kQCol + 8 * (part * kPart + kk), b_desc, C::kIdescS, kk > 0 ? 1u : 0u);
          } else {
            const uint64_t a_desc = umma_desc(q_base + (kk >> 2) * C::kQChunkBytes + (kk & 3) * 32, 16, 1024, 2);
            umma_bf16_warp(d_tmem, a_desc, b_desc, C::kIdescS, kk > 0 ? 1u : 0u);
          }
        }
        umma_commit_warp(&s.s_full[sb]);
        umma_commit_warp(&s.empty[st]);  // this issuer's reads of the K tile done
        if (j == n_steps - 1) umma_commit_warp(C::kQInTmem ? &s.q_tfree[part] : &s.q_empty);  // and of the item's Q
        if (++st == kStages) st = 0, st_ph ^= 1;
        if (++sb == C::kSBufs) sb = 0, sb_ph ^= 1;
        ++g;
      }
      ++gt;
    }
    if constexpr (C::kQInTmem) {  // the last item's commit on q_tfree
      if (ok && gt >= 1) ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.q_tfree[part], (gt - 1) & 1));
    }
    if (part == 0) {  // the softmax warps' last arrivals on s_free (not waited for above)
      for (int k = g >= C::kSBufs ? g - C::kSBufs : 0; k < g; ++k)
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.s_free[k % C::kSBufs], (k / C::kSBufs) & 1));
    }
    umma_commit_warp(&s.mma_done);
    if (!__all_sync(0xffffffffu, mbar_wait_fast(&s.mma_done, 0))) ok = false;  // every product done before the memory is freed
    if (!ok && lane == 0) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
  } else if (warp == C::kPVWarp) {
    // ---------------- P V issuer (whole warp): O += P_j V_j, one product of K = 16 per page ----------------
    bool ok = true;
    int gt = 0;                      // items done
    int pst = 0, pst_ph = 0, pb = 0, pb_ph = 0;  // V tile and P buffer of the next step
    for (int w = blockIdx.x; w < n_work; w += gridDim.x) {
      const TileItem it = load_tile<C>(p, w, tiles, false);
      if (!warp_uniform_int(it.run)) continue;
      const int n_steps = warp_uniform_int(it.n_steps);
      // the item's first P V overwrites O: the previous item's epilogue must have read it
      if (ok && gt >= 1) ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.o_free, (gt - 1) & 1));
      for (int j = 0; j < n_steps; ++j) {
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.v_full[pst], pst_ph));
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.p_full[pb], pb_ph));
        tc_fence_after_sync();
        const uint32_t v_base = smem_addr(s.v[pst]);
#pragma unroll
        for (int kk = 0; kk < kPPS; ++kk) {
          const uint64_t b_desc = umma_desc(v_base + kk * C::kVPage, C::kChunkBytes, 1024, 2);
          if constexpr (C::kPInTmem) {
            umma_bf16_ts_warp(tmem, tmem + C::p_col(pb) + 8 * kk, b_desc, C::kIdescPV,
                              (j > 0 || kk > 0) ? 1u : 0u);
          } else {
            const uint64_t a_desc = umma_desc(smem_addr(s.p[pb]) + kk * 256, 128, C::kKeys * 16, 0);
            umma_bf16_warp(tmem, a_desc, b_desc, C::kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
          }
        }
        umma_commit_warp(&s.v_empty[pst]);  // the V tile read
        umma_commit_warp(C::kPInS ? &s.s_free[pb] : &s.p_empty[pb]);  // P read
        if (++pst == C::kVStages) pst = 0, pst_ph ^= 1;
        if (++pb == C::kPBufs) pb = 0, pb_ph ^= 1;
      }
      umma_commit_warp(&s.o_full);  // the item's products done
      ++gt;
    }
    // the last epilogue's arrival on o_free (not waited for above)
    if (ok && gt >= 1) ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.o_free, (gt - 1) & 1));
    umma_commit_warp(&s.mma_done);
    if (!__all_sync(0xffffffffu, mbar_wait_fast(&s.mma_done, 0))) ok = false;
    if (!ok && lane == 0) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
  } else {
    // ---------------- softmax and epilogue: one thread per row (and half) ----------------
    // With two warpgroups, thread r of group h handles keys [h kHalf, (h + 1) kHalf)
    // of each step of row r, and columns [h kDS/2, (h + 1) kDS/2) of O; the
    // two halves of a row share the row max through shared memory.
    constexpr int kGroups = C::kSoftmaxGroups;
    constexpr int kHalf = C::kKeys / kGroups;  // keys of a step per thread
    constexpr int kOCols = kDS / kGroups;      // output dims per thread
    static_assert(kOCols % (16 * kRoundTrip) == 0, "whole TMEM round trips");
    const int h = warp < 4 ? 0 : (warp - C::kVProdWarp - 1) / 4 + 1;  // softmax warpgroup (warps 0-3, then the last ones)
    const int r = 32 * (warp & 3) + lane;       // row = TMEM lane
    const int st = h * 128 + r;                 // index among the softmax threads
    const int kc0 = h * kHalf;                  // this thread's first key column of a step
    const int oc0 = h * kOCols;                 // and first output column
    const int g = r / kQ;
    const int qi = r % kQ;
    const uint32_t t_row = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    bool ok = true;
    int gs = 0, gt = 0;  // steps and items done
    for (int w = blockIdx.x; w < n_work; w += gridDim.x) {
      const TileItem it = load_tile<C>(p, w, tiles, false);
      if (!it.run) continue;
      const bool valid = qi < it.nq;
      const int head = it.c * kG + g;
      // whether this CTA has another item: its Q then passes through the Q
      // buffer before this item's output may be staged there
      bool has_next = false;
      if constexpr (C::kQInTmem) {
        for (int w2 = w + gridDim.x; w2 < n_work && !has_next; w2 += gridDim.x)
          has_next = load_tile<C>(p, w2, tiles, false).run;
      }
      const int pos = it.P0 + qi;
      const int lo_r = p.window > 0 ? pos - p.window + 1 : 0;

      float m = -INFINITY, l = 0.f;  // reference max (log2 units) and this thread's share of the row sum
      for (int j = 0; j < it.n_steps; ++j) {
        const int gj = gs + j;
        const int bs = gj % C::kSBufs;  // S buffer
        const int pb = gj % C::kPBufs;  // P buffer
        const int xb = gj & 1;          // exchange buffer of the half-row maxima
        const int step0 = (it.page0 + tile_step(it, j) * kPPS) * kPage;  // key of the step's column 0
        const int pos0 = step0 + kc0;                   // key of this thread's first column
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.s_full[bs], (gj / C::kSBufs) & 1));
        tc_fence_after_sync();
        float sv[kHalf];
        load_row<kHalf>(t_row + C::kSCol + C::kKeys * (C::kIssuers * bs) + kc0, sv);
#pragma unroll
        for (int part = 1; part < C::kIssuers; ++part) {
          float sb[kHalf];
          load_row<kHalf>(t_row + C::kSCol + C::kKeys * (C::kIssuers * bs + part) + kc0, sb);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < kHalf; ++k) sv[k] += sb[k];
        }
        tmem_wait_ld();
        tc_fence_before_sync();
        __syncwarp();
        if (!C::kPInS && lane == 0) mbar_arrive(&s.s_free[bs]);

        if (!valid || pos0 < lo_r || pos0 + kHalf - 1 > pos) {
#pragma unroll
          for (int k = 0; k < kHalf; ++k) {
            const int key = pos0 + k;
            if (!valid || key < lo_r || key > pos) sv[k] = -INFINITY;
          }
        }
        float mx = tree_max<kHalf>(sv);
        if constexpr (kGroups > 1) {
          // only the warps holding the same 32 rows exchange: one barrier per
          // set of them (ids 2-5), so a warp waits for its partners alone
          s.half_max[xb][h][r] = mx;
          named_barrier_sync(2 + (warp & 3), 32 * kGroups);
#pragma unroll
          for (int o = 1; o < kGroups; ++o) mx = fmaxf(mx, s.half_max[xb][(h + o) % kGroups][r]);
        }
        const float m_new = mx * kLog2e;
        const bool move = m_new > m + kSlack;  // false while the row has no visible key
        const bool rescale = move && m != -INFINITY;
        if (__any_sync(0xffffffffu, rescale)) {
          // O's row holds P V up to step j-1: wait for that product, then scale in place
          if (ok && j >= 1)
            ok = __all_sync(0xffffffffu, mbar_wait_fast(C::kPInS ? &s.s_free[(gj - 1) % C::kPBufs]
                                                                 : &s.p_empty[(gj - 1) % C::kPBufs],
                                                        ((gj - 1) / C::kPBufs) & 1));
          tc_fence_after_sync();
          const float f = rescale ? ex2_approx(m - (m_new + kHeadroom)) : 1.f;
#pragma unroll 1
          for (int col = oc0; col < oc0 + kOCols; col += 16 * kRoundTrip) {
            float ov[kRoundTrip][16];
#pragma unroll
            for (int u = 0; u < kRoundTrip; ++u) tmem_ld16(t_row + col + 16 * u, ov[u]);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < kRoundTrip; ++u) {
#pragma unroll
              for (int k = 0; k < 16; ++k) ov[u][k] *= f;
              tmem_st16(t_row + col + 16 * u, ov[u]);
            }
          }
          tmem_wait_st();
          l *= f;
        }
        if (move) m = m_new + kHeadroom;
        const float m_use = m == -INFINITY ? 0.f : m;
#pragma unroll
        for (int k = 0; k < kHalf; ++k) sv[k] = ex2_approx(fmaf(sv[k], kLog2e, -m_use));
        l += tree_sum<kHalf>(sv);

        // P row into buffer pb (K-major core matrices of 8 rows x 8 keys) once
        // P V of step gj - kPBufs has read it
        // (P over S: the buffer's previous P V finished before this S was computed)
        if (!C::kPInS && ok && gj >= C::kPBufs)
          ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.p_empty[pb], ((gj / C::kPBufs) - 1) & 1));
        if constexpr (C::kPInTmem) {
          // this row's keys into its lane: column p_col(pb) + k / 2 holds keys k, k + 1
          if constexpr (kHalf % 16 == 0) {
#pragma unroll
            for (int kc = 0; kc < kHalf / 16; ++kc) {
              uint32_t wv[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) wv[e] = pack_bf16x2(sv[16 * kc + 2 * e], sv[16 * kc + 2 * e + 1]);
              tmem_st8(t_row + C::p_col(pb) + kc0 / 2 + 8 * kc, wv);
            }
          } else {  // 8 keys: 4 columns
            uint32_t wv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) wv[e] = pack_bf16x2(sv[2 * e], sv[2 * e + 1]);
            tmem_st4(t_row + C::p_col(pb) + kc0 / 2, wv);
          }
          tmem_wait_st();
        } else {
          const uint32_t p_row = smem_addr(s.p[pb]) + (r >> 3) * (C::kKeys * 16) + (r & 7) * 16;
#pragma unroll
          for (int kc = 0; kc < C::kKeys / 8; ++kc)
            st_shared_v4(p_row + kc * 128,
                         make_uint4(pack_bf16x2(sv[8 * kc], sv[8 * kc + 1]), pack_bf16x2(sv[8 * kc + 2], sv[8 * kc + 3]),
                                    pack_bf16x2(sv[8 * kc + 4], sv[8 * kc + 5]),
                                    pack_bf16x2(sv[8 * kc + 6], sv[8 * kc + 7])));
        }
        // zero this step's V rows outside [k_lo, k_hi] (the first and last steps)
        const bool edge = step0 < it.k_lo || step0 + C::kKeys - 1 > it.k_hi;
        if (edge) {
          const int vs = gj % C::kVStages;  // the V tile must have landed before its rows are zeroed
          if (ok) ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.v_full[vs], (gj / C::kVStages) & 1));
          const uint32_t v_base = smem_addr(s.v[vs]);
#pragma unroll 1
          for (int e = st; e < C::kKeys * 8; e += C::kSoftmaxThreads) {
            const int kr = e >> 3;  // key row of the step
            const int key = step0 + kr;
            if (key < it.k_lo || key > it.k_hi) {
#pragma unroll
              for (int ch = 0; ch < C::kVChunks; ++ch)
                st_shared_v4(v_base + (kr >> 4) * C::kVPage + ch * C::kChunkBytes + (kr & 15) * 128 + (e & 7) * 16,
                             make_uint4(0, 0, 0, 0));
            }
          }
        }
        // shared-memory writes (P, zeroed V rows) made visible to the MMA's reads
        if (!C::kPInTmem || edge) fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.p_full[pb]);
      }

      // ---- epilogue: wait for the item's last P V, normalise, write this row's output dims ----
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.o_full, gt & 1));
      tc_fence_after_sync();
      if constexpr (kGroups > 1) {
        s.half_sum[h][r] = l;
        named_barrier_sync(1, C::kSoftmaxThreads);
        float lt = 0.f;  // the row sum in group order, the same in every group
#pragma unroll
        for (int o = 0; o < kGroups; ++o) lt += s.half_sum[o][r];
        l = lt;
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if (!p.out_f32 && it.nq == kQ) {
        // A full tile in bf16: O goes out one 64-dim chunk at a time, staged in
        // shared memory (swizzled like Q) and written by one TMA store per
        // chunk, G heads x kQ queries in one box.  A thread's own row is 8 KB
        // from its neighbours' in global memory, so per-thread stores made 32
        // transactions of every warp instruction.  (A partial tile takes the
        // per-thread stores below: a box would reach the next sequence's rows.)
        constexpr int kOutChunks = kDS / 64;
        constexpr int kOwnChunks = kOutChunks / kGroups;
        if constexpr (C::kQInTmem) {
          // every chunk in its own 16 KB of the Q buffer, once the next item's
          // Q has been copied out of it
          static_assert(kOutChunks <= C::kKChunks, "O fits the Q buffer");
          if (ok && has_next) ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.q_empty, (gt + 1) & 1));
#pragma unroll 1
          for (int cc = h * kOwnChunks; cc < (h + 1) * kOwnChunks; ++cc) {
            float ov[4][16];
#pragma unroll
            for (int u = 0; u < 4; ++u) tmem_ld16(t_row + 64 * cc + 16 * u, ov[u]);
            tmem_wait_ld();
            const uint32_t row = smem_addr(s.q[cc]) + r * 128;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float* v = &ov[u >> 1][8 * (u & 1)];
              st_shared_v4(row + ((u ^ (r & 7)) << 4),
                           make_uint4(pack_bf16x2(v[0] * inv, v[1] * inv), pack_bf16x2(v[2] * inv, v[3] * inv),
                                      pack_bf16x2(v[4] * inv, v[5] * inv), pack_bf16x2(v[6] * inv, v[7] * inv)));
            }
          }
          fence_proxy_async_smem();
          named_barrier_sync(1, C::kSoftmaxThreads);
          if (st == 0) {
            for (int cc = 0; cc < kOutChunks; ++cc)
              tma_store_4d(&tm_o, s.q[cc], 0, it.slice * kOutChunks + cc, it.q0 + it.i0, it.c * kG);
            tma_store_wait_read();
          }
        } else {
#pragma unroll 1
        for (int cc = 0; cc < kOutChunks; ++cc) {
          if (cc / kOwnChunks == h) {
            float ov[4][16];
#pragma unroll
            for (int u = 0; u < 4; ++u) tmem_ld16(t_row + 64 * cc + 16 * u, ov[u]);
            tmem_wait_ld();
            const uint32_t row = smem_addr(s.ost) + r * 128;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float* v = &ov[u >> 1][8 * (u & 1)];
              st_shared_v4(row + ((u ^ (r & 7)) << 4),
                           make_uint4(pack_bf16x2(v[0] * inv, v[1] * inv), pack_bf16x2(v[2] * inv, v[3] * inv),
                                      pack_bf16x2(v[4] * inv, v[5] * inv), pack_bf16x2(v[6] * inv, v[7] * inv)));
            }
            fence_proxy_async_smem();
          }
          named_barrier_sync(1, C::kSoftmaxThreads);
          if (st == 0) {
            tma_store_4d(&tm_o, s.ost, 0, it.slice * kOutChunks + cc, it.q0 + it.i0, it.c * kG);
            tma_store_wait_read();
          }
          named_barrier_sync(1, C::kSoftmaxThreads);  // the staging buffer read: the next chunk may overwrite it
        }
        }
      } else {
      const size_t o_off = (static_cast<size_t>(it.q0 + it.i0 + qi) * kHq + head) * kD + it.slice * kDS;
#pragma unroll 1
      for (int col0 = oc0; col0 < oc0 + kOCols; col0 += 16 * kRoundTrip) {
        float ovs[kRoundTrip][16];
#pragma unroll
        for (int u = 0; u < kRoundTrip; ++u) tmem_ld16(t_row + col0 + 16 * u, ovs[u]);
        tmem_wait_ld();
        if (!valid) continue;
#pragma unroll
        for (int u = 0; u < kRoundTrip; ++u) {
          const float* ov = ovs[u];
          const int col = col0 + 16 * u;
          if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + o_off + col);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              dst[k] = make_float4(ov[4 * k] * inv, ov[4 * k + 1] * inv, ov[4 * k + 2] * inv, ov[4 * k + 3] * inv);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + o_off + col);
            dst[0] = make_uint4(pack_bf16x2(ov[0] * inv, ov[1] * inv), pack_bf16x2(ov[2] * inv, ov[3] * inv),
                                pack_bf16x2(ov[4] * inv, ov[5] * inv), pack_bf16x2(ov[6] * inv, ov[7] * inv));
            dst[1] = make_uint4(pack_bf16x2(ov[8] * inv, ov[9] * inv), pack_bf16x2(ov[10] * inv, ov[11] * inv),
                                pack_bf16x2(ov[12] * inv, ov[13] * inv), pack_bf16x2(ov[14] * inv, ov[15] * inv));
          }
        }
      }
      }
      if constexpr (kGroups > 1) named_barrier_sync(1, C::kSoftmaxThreads);  // half_sum read before its next write
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.o_free);  // the next item's first P V may overwrite O
      if (C::kQInTmem && st == 0) mbar_arrive(&s.ost_free);  // (its stores, if any, have read the Q buffer)
      gs += it.n_steps;
      ++gt;
    }
    // the last P V products' commits (not all waited for above)
    for (int gj = gs >= C::kPBufs ? gs - C::kPBufs : 0; gj < gs; ++gj)
      if (ok)
        ok = __all_sync(0xffffffffu, mbar_wait_fast(C::kPInS ? &s.s_free[gj % C::kPBufs] : &s.p_empty[gj % C::kPBufs],
                                                    (gj / C::kPBufs) & 1));
    if (!ok && lane == 0) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
    if (st == 0) tma_store_wait_all();  // the output stores complete before the CTA retires
  }

  // ---------------- teardown: free the tensor memory ----------------
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Gemma-4-12B shapes.  Sliding: 64 queries x 2 heads per work item, D = 256,
// 4-page steps (N = 64), K and V tiles in rings of 2 x 32 KB each, Q in
// tensor memory, two S buffers with P written over them (O 256 + Q 128 +
// S 2 x 64 columns), one S issuer and a P V issuer, two softmax warpgroups.
// Global: 8 queries x 16 heads per block, D = 512 split into two blocks of
// 256 output dims (both compute S), 2-page steps in 2 stages of 48 KB, two S
// issuers, one softmax warpgroup; every block of a KV head reads the same
// pages, so tile t starts 7 t steps into its range (the blocks resident at
// one time then read different pages: 8 % faster than all in step).
using SlidingConfig =
    Config<ATTN_SLIDING_D, ATTN_SLIDING_D, ATTN_SLIDING_HQ / ATTN_SLIDING_HKV, ATTN_SLIDING_HKV, 2, 4, true, 1, 2, 0,
           2, 2, true, 2, true>;
using GlobalConfig = Config<ATTN_GLOBAL_D, 256, ATTN_GLOBAL_HQ / ATTN_GLOBAL_HKV, ATTN_GLOBAL_HKV, 2, 2, true, 2, 1, 7>;

}  // namespace prefill_tc
}  // namespace pda
