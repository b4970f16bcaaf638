// prefill_pair.cuh -- multi-query attention over the paged cache (the same
// operation as prefill_tc.cuh: Attention.lean `causalGQA` / `slidingGQA`
// with S > 1) on pairs of CTAs sharing every tensor-core product
// (tcgen05 cta_group::2).
//
// A cluster of two CTAs takes two adjacent query tiles of one sequence and KV
// head: CTA rank r holds tile 2t + r, 128 rows (kQ = 128 / G queries times
// the G query heads), and its Q in shared memory.  The pair walks the union
// of its two tiles' key ranges in steps of kPPS pages (16 kPPS keys, kPPS =
// 2 or 4):
//   S   = Q K^T   one M = 256, N = 16 kPPS MMA per 16 dims of D, issued by
//                 rank 0: A = each CTA's own Q rows, B = the step's keys,
//                 CTA r holding pages r kPPS/2 .. (r+1) kPPS/2 - 1 of the
//                 step, chunk-major ([chunk][kPPS/2 x 16 rows][128 B]); D =
//                 each CTA's own S rows in its tensor memory;
//   P   = softmax as in prefill_tc.cuh, each CTA on its own rows;
//   O  += P V     M = 256, N = kDS, K = 16 per page: A = P in each CTA's
//                 tensor memory, B = V with CTA r holding output dims
//                 [r kDS/2, (r+1) kDS/2) of every page of the step.
// So each SM copies half of every K and V tile, and one instruction does
// the work of two.
//
// Handshakes.  K and V tiles sit in two rings with a producer warp each; a
// K tile is free again when its S products are done, a V tile when its P V
// product is.  Each CTA's copies complete on its own `k_full` / `v_full`
// barriers; rank 1's idle issuing warp forwards each landed K tile to rank
// 0's `k_peer`.  The softmax warps of each CTA arrive on their own CTA's
// `s_free`, `p_full` and `q_ready`, and two warps of rank 1 forward each
// completed phase to rank 0's (which count one arrival more), the p_full
// forward only once rank 1's V tile of the step has landed: an arrival with
// release at cluster scope cost a softmax warp about 400 cycles, twice per
// step, so no softmax warp makes one.  Rank 0 commits every product to both
// CTAs' barriers (`s_full`, `p_empty`, `k_empty`, `v_empty`, `mma_done`,
// multicast).  Every arrival a CTA receives is waited for before the final
// cluster barrier, so none can land after a CTA has left; every wait is
// bounded.
#pragma once

#include "prefill_tc.cuh"

namespace pda {
namespace prefill_pair {

using prefill_tc::PrefillParams;

template <int kD_, int kDS_, int kG_, int kHkv_, int kStages_, int kSoftmaxGroups_, int kRotate_, int kSBufs_ = 2,
          int kPBufs_ = 2, int kSIssuers_ = 1, int kPPS_ = 2>
struct PairConfig {
  static constexpr int kD = kD_;    // head dim (the contraction of S)
  static constexpr int kDS = kDS_;  // output dims per pair (each CTA holds V for half of them)
  static constexpr int kG = kG_;
  static constexpr int kHkv = kHkv_;
  static constexpr int kHq = kG * kHkv;
  static constexpr int kStages = kStages_;
  // Pages per step: 2 (one page of K per CTA) or 4 (two per CTA).  S has
  // N = 16 kPPS, and each CTA supplies the B rows of its kKPages pages.
  static constexpr int kPPS = kPPS_;
  static constexpr int kKPages = kPPS / 2;       // pages of K per CTA per step
  static constexpr int kKeys = kPPS * kPage;     // N of S, K of P V
  static constexpr int kSlices = kD / kDS;
  static constexpr int kRows = 128;               // rows per CTA
  static constexpr int kQ = kRows / kG;           // queries per CTA
  static constexpr int kKChunks = kD / 64;
  static constexpr int kVChunksHalf = kDS / 128;  // 64-dim chunks of V per CTA
  static constexpr int kQChunkBytes = kRows * 128;
  static constexpr int kPageChunk = kPage * 128;  // one 64-dim chunk of one page: [16 rows][128 B]
  // This CTA's K of a step, chunk-major: [chunk][kKPages * 16 rows][128 B],
  // so that the B operand of S has its 8-row groups 1 KB apart.  One page
  // per CTA is one TMA box of all chunks; two pages take one 2 KB box per
  // page and chunk (a box lands densely, so two pages cannot interleave).
  static constexpr int kKChunkBytes = kKPages * kPageChunk;
  static constexpr int kKTile = kKChunks * kKChunkBytes;
  static constexpr int kKBoxChunks = kKPages == 1 ? kKChunks : 1;  // 64-dim chunks per K box
  static constexpr int kVPage = kVChunksHalf * kPageChunk;
  static constexpr int kVTile = kPPS * kVPage;
  static constexpr int kSoftmaxGroups = kSoftmaxGroups_;
  static constexpr int kSoftmaxThreads = 128 * kSoftmaxGroups;
  static constexpr int kSoftmaxWarps = 4 * kSoftmaxGroups;
  // + the K producer (warp 4), two more warps and the V producer in each
  // CTA.  Rank 0: warp 5 issues the S products, warp kFwdSWarp the P V
  // products (separate threads, so that S runs ahead of the softmax whatever
  // P waits for).  Rank 1: warp 5 forwards its landed K tiles, kFwdSWarp
  // its s_free and q_ready phases, kFwdPWarp its p_full phases (each once
  // its V tile of the step has landed too) to rank 0.
  static constexpr int kThreads = (kSoftmaxWarps + 5) * 32;
  static constexpr int kFwdSWarp = kSoftmaxWarps + 2;
  static constexpr int kFwdPWarp = kSoftmaxWarps + 3;
  static constexpr int kVProdWarp = kSoftmaxWarps + 4;
  static constexpr int kRotate = kRotate_;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kSBufs = kSBufs_;                  // S buffers: S runs up to kSBufs steps ahead
  // Warps of rank 0 issuing S (1 or 2): with two, warp kFwdPWarp (idle on
  // rank 0 otherwise) issues the second half of the D k-steps into its own
  // part of each S buffer, and the softmax adds the two parts.
  static constexpr int kSIssuers = kSIssuers_;
  static constexpr uint32_t kSCol = kDS;                  // kSBufs S buffers of kSIssuers x kKeys columns
  static constexpr int kPBufs = kPBufs_;                  // P buffers: P V may lag the softmax by kPBufs - 1 steps
  static constexpr uint32_t kPCol = kSCol + kSBufs * kSIssuers * kKeys;  // P buffers (bf16 pairs), kKeys / 2 columns each
  static_assert((kSIssuers == 1 || kSIssuers == 2) && ((kD / 16) / kSIssuers) % 4 == 0,
                "each S issuer takes whole 64-dim chunks of Q and K");
  static constexpr uint32_t kIdescS = umma_idesc_bf16(256, kKeys, 0, 0);
  static constexpr uint32_t kIdescPV = umma_idesc_bf16(256, kDS, 0, 1);
  static_assert(kRows % kG == 0 && kD % 64 == 0 && kDS % 128 == 0 && kDS <= 256, "tile shapes");
  static_assert(kPPS == 2 || kPPS == 4, "two or four pages per step");
  static_assert(kPCol + kPBufs * kKeys / 2 <= kTmemCols, "O, the S buffers and the P buffers fit in tensor memory");
  static_assert(kSoftmaxGroups == 1 || (kSoftmaxGroups == 2 && (kKeys / 2) % 16 == 0 && kDS % 32 == 0),
                "two softmax warpgroups: halves of whole 16-key blocks");

  struct Smem {
    alignas(1024) uint8_t q[kKChunks][kQChunkBytes];
    alignas(1024) uint8_t k[kStages][kKTile];
    alignas(1024) uint8_t v[kStages][kVTile];
    // K and V tiles in two rings, each filled by its own producer warp: a K
    // tile is released when its S products are done, a V tile when its P V
    // product is, so that K is copied a step earlier than a shared stage
    // would allow.
    alignas(8) uint64_t k_full[kStages];   // this CTA's K tile landed (TMA)
    alignas(8) uint64_t k_peer[kStages];   // rank 0: rank 1's K tile landed (forwarded)
    alignas(8) uint64_t k_empty[kStages];  // S products of the tile done (commits, both CTAs)
    alignas(8) uint64_t v_full[kStages];   // this CTA's V tile landed (TMA)
    alignas(8) uint64_t v_empty[kStages];  // P V of the tile done (commit, both CTAs)
    alignas(8) uint64_t s_full[kSBufs];      // S buffer written (commit, both CTAs)
    alignas(8) uint64_t s_free[kSBufs];      // S buffer read by this CTA's softmax warps (rank 0: and rank 1's)
    alignas(8) uint64_t p_full[kPBufs];      // P written, O rescaled, V edges zeroed (rank 0: both CTAs)
    alignas(8) uint64_t p_empty[kPBufs];     // P V of the buffer's step done (commit, both CTAs)
    alignas(8) uint64_t q_ready;             // Q tile written (rank 0: both CTAs)
    alignas(8) uint64_t mma_done;            // every product done (one commit per issuer, both CTAs)
    uint32_t tmem_base;
    float half_max[2][kSoftmaxGroups][kRows];
    float half_sum[kSoftmaxGroups][kRows];
  };
  static constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "one CTA per SM within the 227 KB a CTA may have");
};

template <typename C>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(C::kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ PrefillParams p) {
  using prefill_tc::kSlack;
  using prefill_tc::kHeadroom;
  using prefill_tc::kRoundTrip;
  constexpr int kD = C::kD, kDS = C::kDS, kG = C::kG, kHq = C::kHq, kQ = C::kQ, kStages = C::kStages;
  constexpr int kPPS = C::kPPS;
  extern __shared__ uint8_t smem_raw[];
  typename C::Smem& s =
      *reinterpret_cast<typename C::Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const uint32_t rank = cluster_ctarank();  // 0 issues the products
  const int tile = blockIdx.x;              // this CTA's query tile
  const int pair = blockIdx.x >> 1;
  const int c = blockIdx.y / C::kSlices;
  const int slice = blockIdx.y % C::kSlices;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // this CTA's softmax warps, and at rank 0 one forwarded arrival for rank 1's
  const int kArrivals = C::kSoftmaxWarps + (rank == 0 ? 1 : 0);

  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&s.k_full[st], 1);
      mbar_init(&s.k_peer[st], 1);
      mbar_init(&s.k_empty[st], C::kSIssuers);  // the S issuers
      mbar_init(&s.v_full[st], 1);
      mbar_init(&s.v_empty[st], 1);  // the P V issuer
    }
    for (int i = 0; i < C::kSBufs; ++i) {
      mbar_init(&s.s_full[i], C::kSIssuers);
      mbar_init(&s.s_free[i], kArrivals);
    }
    for (int i = 0; i < C::kPBufs; ++i) {
      mbar_init(&s.p_full[i], kArrivals);
      mbar_init(&s.p_empty[i], 1);
    }
    mbar_init(&s.q_ready, kArrivals);
    mbar_init(&s.mma_done, C::kSIssuers + 1);
    fence_mbar_init();
  }
  if (warp == 4 && lane == 0) {
    prefetch_tensor_map(&tm_k);
    prefetch_tensor_map(&tm_v);
  }
  if (warp == 5) tmem_alloc_pair(&s.tmem_base, C::kTmemCols);
  tc_fence_before_sync();
  cluster_sync_all();  // both CTAs' barriers initialised and tensor memory allocated
  tc_fence_after_sync();
  const uint32_t tmem = s.tmem_base;
  // rank 0's copy of a barrier (for arrivals from either CTA)
  const auto at_rank0 = [](uint64_t* bar) { return mapa_shared(smem_addr(bar), 0); };

  // q, the cache and the tables may be written by the previous kernel in the stream.
  wait_for_primary_grid();
  allow_dependent_launch();

  // ---- the pair's queries and the keys they can see (uniform over the pair) ----
  const int q0 = p.cu_q[b];
  const int n = p.cu_q[b + 1] - q0;
  const int i0p = pair * 2 * kQ;  // the pair's first query
  const int i0 = tile * kQ;       // this CTA's first query
  const int L = p.seq_lens[b];
  const int cap = p.max_blocks < ATTN_MAX_SEQ_LEN / kPage ? p.max_blocks * kPage : ATTN_MAX_SEQ_LEN;
  bool run = true;
  if (n < 0 || q0 < 0 || static_cast<int64_t>(q0) + n > p.total_q) {
    if (threadIdx.x == 0 && rank == 0) report(p.status, ATTN_DEV_BAD_SEQ_LEN);
    run = false;
  } else {
    if (n > p.max_q && pair == 0 && blockIdx.y == 0 && threadIdx.x == 0 && rank == 0)
      report(p.status, ATTN_DEV_BAD_SEQ_LEN);  // more queries than the host's max_q: the rest are not computed
    if (i0p >= (n < p.max_q ? n : p.max_q)) {
      run = false;
    } else if (L < n || L > cap) {
      if (threadIdx.x == 0 && rank == 0) report(p.status, ATTN_DEV_BAD_SEQ_LEN);
      run = false;
    }
  }

  if (run) {
    const int n_run = n < p.max_q ? n : p.max_q;                  // queries computed
    const int nqp = n_run - i0p < 2 * kQ ? n_run - i0p : 2 * kQ;  // valid queries of the pair
    const int nq = n_run - i0 < 0 ? 0 : (n_run - i0 < kQ ? n_run - i0 : kQ);  // of this CTA
    const int P0p = L - n + i0p;   // position of the pair's first query
    const int P0 = L - n + i0;     // of this CTA's first query
    const int k_hi = P0p + nqp - 1;  // last key the pair sees (inclusive)
    const int k_lo = p.window > 0 ? (P0p - p.window + 1 > 0 ? P0p - p.window + 1 : 0) : 0;
    const int page0 = k_lo / kPage;
    const int n_pages = k_hi / kPage - page0 + 1;
    const int n_steps = (n_pages + kPPS - 1) / kPPS;
    const int rot = C::kRotate > 0 ? static_cast<int>((static_cast<int64_t>(pair) * C::kRotate) % n_steps) : 0;
    const auto logical_step = [&](int j) { return j + rot < n_steps ? j + rot : j + rot - n_steps; };
    const auto logical_page = [&](int gp) { return logical_step(gp / kPPS) * kPPS + gp % kPPS; };

    if (warp == 4 || warp == C::kVProdWarp) {
      // ---------------- producers: this CTA's half of every step, K (warp 4) and V ----------------
      // V: lane pg < kPPS copies this CTA's output dims of V for page pg of
      // the step.  K: lanes kKPages rank .. kKPages (rank + 1) - 1 copy all of
      // K of their page (the CTA's B rows of S).  Pages past the range and
      // bad page ids are copied from a fully out-of-range row: zeros.
      const bool is_k = warp == 4;
      uint64_t* const full = is_k ? s.k_full : s.v_full;
      uint64_t* const empty = is_k ? s.k_empty : s.v_empty;
      const int32_t* bt = p.block_table + static_cast<int64_t>(b) * p.max_blocks;
      bool ok = true;
      int issued = 0;
      const auto entry = [&](int gp) {
        const int lp = logical_page(gp);
        return gp < n_steps * kPPS && lp < n_pages ? bt[page0 + lp] : -1;
      };
      int cur = entry(lane);
      int nxt = entry(32 + lane);
      const int v_z = c * C::kKChunks + slice * (kDS / 64) + static_cast<int>(rank) * C::kVChunksHalf;
      for (int i = 0; i < n_steps; ++i) {
        const int gp0 = i * kPPS;
        if (gp0 > 0 && (gp0 & 31) == 0) {
          cur = nxt;
          nxt = entry(gp0 + 32 + lane);
        }
        const int phys = __shfl_sync(0xffffffffu, cur, (gp0 + (lane < kPPS ? lane : 0)) & 31);
        const int stage = i % kStages;
        if (i >= kStages) {
          const int w = lane == 0 ? static_cast<int>(mbar_wait_fast(&empty[stage], ((i / kStages) - 1) & 1)) : 0;
          ok = __shfl_sync(0xffffffffu, w, 0) != 0;
        }
        if (!ok) {
          if (lane == 0) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&full[stage], is_k ? C::kKTile : C::kVTile);
        __syncwarp();
        if (lane < kPPS) {
          const int gp = logical_page(gp0 + lane);
          int32_t y = -kPage;
          if (gp < n_pages) {
            if (phys < 0 || static_cast<int64_t>(phys) >= p.num_pages)
              report(p.status, ATTN_DEV_BAD_PAGE);
            else
              y = phys * kPage;
          }
          if (!is_k) {
            prefill_tc::tma_load_3d(s.v[stage] + lane * C::kVPage, &tm_v, 0, y, v_z, &full[stage]);
          } else if (lane / C::kKPages == static_cast<int>(rank)) {
            if constexpr (C::kKPages == 1) {
              prefill_tc::tma_load_3d(s.k[stage], &tm_k, 0, y, c * C::kKChunks, &full[stage]);
            } else {
              const int pc = lane % C::kKPages;  // the page's place among this CTA's keys
#pragma unroll
              for (int ch = 0; ch < C::kKChunks; ++ch)
                prefill_tc::tma_load_3d(s.k[stage] + ch * C::kKChunkBytes + pc * C::kPageChunk, &tm_k, 0, y,
                                        c * C::kKChunks + ch, &full[stage]);
            }
          }
        }
        ++issued;
        __syncwarp();
      }
      if (lane == 0) {  // no copy may still be landing, nor a commit arriving, when the CTA retires
        for (int st = 0; st < kStages && st < issued; ++st) {
          const int uses = (issued - 1 - st) / kStages + 1;
          if (!mbar_wait(&full[st], (uses - 1) & 1)) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
          if (ok && !mbar_wait(&empty[st], (uses - 1) & 1)) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
        }
      }
    } else if ((warp == 5 || (C::kSIssuers == 2 && warp == C::kFwdPWarp)) && rank == 0) {
      // ---------------- rank 0: the pair's S products (whole warp, an elected lane issues) ----------------
      constexpr int kPart = (kD / 16) / C::kSIssuers;  // k-steps per S issuer
      const int part = warp == 5 ? 0 : 1;
      bool ok = __all_sync(0xffffffffu, mbar_wait_cluster(&s.q_ready, 0));
      const uint32_t q_base = smem_addr(s.q[0]) + (part * kPart / 4) * C::kQChunkBytes;
      for (int j = 0; j < n_steps; ++j) {
        const int st = j % kStages;
        const int bs = j % C::kSBufs;
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.k_full[st], (j / kStages) & 1));
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_cluster(&s.k_peer[st], (j / kStages) & 1));
        if (ok && j >= C::kSBufs)
          ok = __all_sync(0xffffffffu, mbar_wait_cluster(&s.s_free[bs], ((j / C::kSBufs) - 1) & 1));
        tc_fence_after_sync();
        const uint32_t k_base = smem_addr(s.k[st]) + (part * kPart / 4) * C::kKChunkBytes;
#pragma unroll
        for (int kk = 0; kk < kPart; ++kk) {
          const uint64_t a_desc = umma_desc(q_base + (kk >> 2) * C::kQChunkBytes + (kk & 3) * 32, 16, 1024, 2);
          const uint64_t b_desc = umma_desc(k_base + (kk >> 2) * C::kKChunkBytes + (kk & 3) * 32, 16, 1024, 2);
          umma_bf16_pair_warp(tmem + C::kSCol + C::kKeys * (C::kSIssuers * bs + part), a_desc, b_desc, C::kIdescS,
                              kk > 0 ? 1u : 0u);
        }
        umma_commit_pair_warp(&s.s_full[bs]);
        umma_commit_pair_warp(&s.k_empty[st]);  // the K tile read
      }
      // the softmax warps' last arrivals on s_free (they are not waited for above)
      for (int j = n_steps >= C::kSBufs ? n_steps - C::kSBufs : 0; j < n_steps; ++j)
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_cluster(&s.s_free[j % C::kSBufs], (j / C::kSBufs) & 1));
      umma_commit_pair_warp(&s.mma_done);
      if (!__all_sync(0xffffffffu, mbar_wait_fast(&s.mma_done, 0))) ok = false;
      if (!ok && lane == 0) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
    } else if (warp == C::kFwdSWarp && rank == 0) {
      // ---------------- rank 0: the pair's P V products, one of K = 16 per page ----------------
      // P(j) is complete in both CTAs once p_full completes; rank 1 forwards
      // its arrival only after its own V tile of step j has landed, and this
      // CTA's V tile is waited for here.
      bool ok = true;
      for (int j = 0; j < n_steps; ++j) {
        const int bp = j % C::kPBufs;
        const int st = j % kStages;
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_cluster(&s.p_full[bp], (j / C::kPBufs) & 1));
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.v_full[st], (j / kStages) & 1));
        tc_fence_after_sync();
        const uint32_t v_base = smem_addr(s.v[st]);
#pragma unroll
        for (int kk = 0; kk < kPPS; ++kk) {
          const uint64_t b_desc = umma_desc(v_base + kk * C::kVPage, C::kPageChunk, 1024, 2);
          umma_bf16_ts_pair_warp(tmem, tmem + C::kPCol + (C::kKeys / 2) * bp + 8 * kk, b_desc, C::kIdescPV,
                                 (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit_pair_warp(&s.v_empty[st]);  // the V tile read
        umma_commit_pair_warp(&s.p_empty[bp]);
      }
      umma_commit_pair_warp(&s.mma_done);
      if (!__all_sync(0xffffffffu, mbar_wait_fast(&s.mma_done, 0))) ok = false;
      if (!ok && lane == 0) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
    } else if (warp == 5) {
      // ---------------- rank 1: tell rank 0 when each K tile of this CTA has landed ----------------
      bool ok = true;
      const uint32_t k_peer0 = at_rank0(&s.k_peer[0]);
      for (int j = 0; j < n_steps; ++j) {
        const int st = j % kStages;
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.k_full[st], (j / kStages) & 1));
        if (lane == 0) mbar_arrive_cluster_relaxed(k_peer0 + 8 * st);
      }
      if (!__all_sync(0xffffffffu, mbar_wait_fast(&s.mma_done, 0))) ok = false;  // rank 0's last product
      if (!ok && lane == 0) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
    } else if (warp == C::kFwdSWarp || warp == C::kFwdPWarp) {
      // ---------------- rank 1: forward its softmax warps' arrivals to rank 0 ----------------
      if (rank == 1) {
        bool ok = true;
        const bool fwd_s = warp == C::kFwdSWarp;
        if (fwd_s) {
          ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.q_ready, 0));
          if (lane == 0) mbar_arrive_cluster(at_rank0(&s.q_ready));
        }
        const uint32_t dst0 = at_rank0(fwd_s ? &s.s_free[0] : &s.p_full[0]);
        const int nbuf = fwd_s ? C::kSBufs : C::kPBufs;
        for (int j = 0; j < n_steps; ++j) {
          const int bs = j % nbuf;
          if (ok) ok = __all_sync(0xffffffffu, mbar_wait_fast(fwd_s ? &s.s_free[bs] : &s.p_full[bs], (j / nbuf) & 1));
          // p_full(j) also tells rank 0 that this CTA's V tile of step j has
          // landed (P V reads it); the tile is refilled only after P V(j)
          if (!fwd_s && ok)
            ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.v_full[j % kStages], (j / kStages) & 1));
          if (lane == 0) {
            // s_free relays finished tensor-memory loads and p_full finished
            // tensor-memory stores (tcgen05.wait::ld / ::st): no data to
            // publish, except the V rows that the first and last steps zero
            // in shared memory
            const int step0 = (page0 + logical_step(j) * kPPS) * kPage;
            if (!fwd_s && (step0 < k_lo || step0 + C::kKeys - 1 > k_hi))
              mbar_arrive_cluster(dst0 + 8 * bs);
            else
              mbar_arrive_cluster_relaxed(dst0 + 8 * bs);
          }
        }
        if (!ok && lane == 0) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
      }
    } else {
      // ---------------- softmax and epilogue: one thread per row (and half) of this CTA ----------------
      constexpr int kGroups = C::kSoftmaxGroups;
      constexpr int kHalf = C::kKeys / kGroups;  // keys of a step per thread
      constexpr int kOCols = kDS / kGroups;      // output dims per thread
      static_assert(kOCols % (16 * kRoundTrip) == 0, "whole TMEM round trips");
      const int h = warp >= 4 ? 1 : 0;            // softmax warpgroup (warps 0-3, then 6-9)
      const int r = 32 * (warp & 3) + lane;       // row = TMEM lane
      const int st = h * 128 + r;                 // index among the softmax threads
      const int kc0 = h * kHalf;
      const int oc0 = h * kOCols;
      const int g = r / kQ;
      const int qi = r % kQ;
      const bool valid = qi < nq;
      const int head = c * kG + g;
      const int pos = P0 + qi;
      const int lo_r = p.window > 0 ? pos - p.window + 1 : 0;
      const uint32_t t_row = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);

      // Q row into shared memory: K-major, 128-byte swizzle, chunks of 64 dims
      {
        const uint8_t* src_row = reinterpret_cast<const uint8_t*>(
            p.q + (static_cast<size_t>(valid ? q0 + i0 + qi : 0) * kHq + head) * kD);
        const uint32_t q_base = smem_addr(s.q[0]);
        constexpr int kUnits = kD / 8 / kGroups;
#pragma unroll 8
        for (int u = h * kUnits; u < (h + 1) * kUnits; ++u)
          prefill_tc::cp_async_16(q_base + (u >> 3) * C::kQChunkBytes + r * 128 + (((u & 7) ^ (r & 7)) << 4),
                                  src_row + 16 * u, valid ? 16u : 0u);
        prefill_tc::cp_async_wait_all();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.q_ready);
      }

      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < n_steps; ++j) {
        const int bs = j & 1;              // exchange buffer of the row maxima
        const int pb = j % C::kPBufs;      // P buffer
        const int sb = j % C::kSBufs;      // S buffer
        const int step0 = (page0 + logical_step(j) * kPPS) * kPage;  // key of the step's column 0
        const int pos0 = step0 + kc0;
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.s_full[sb], (j / C::kSBufs) & 1));
        tc_fence_after_sync();
        float sv[kHalf];
#pragma unroll
        for (int blk = 0; blk < kHalf / 16; ++blk)
          tmem_ld16(t_row + C::kSCol + C::kKeys * (C::kSIssuers * sb) + kc0 + 16 * blk,
                    *reinterpret_cast<float(*)[16]>(&sv[16 * blk]));
        if constexpr (C::kSIssuers == 2) {
          float sb2[kHalf];
#pragma unroll
          for (int blk = 0; blk < kHalf / 16; ++blk)
            tmem_ld16(t_row + C::kSCol + C::kKeys * (C::kSIssuers * sb + 1) + kc0 + 16 * blk,
                      *reinterpret_cast<float(*)[16]>(&sb2[16 * blk]));
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < kHalf; ++k) sv[k] += sb2[k];
        }
        tmem_wait_ld();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.s_free[sb]);

        if (!valid || pos0 < lo_r || pos0 + kHalf - 1 > pos) {
#pragma unroll
          for (int k = 0; k < kHalf; ++k) {
            const int key = pos0 + k;
            if (!valid || key < lo_r || key > pos) sv[k] = -INFINITY;
          }
        }
        float mx = sv[0];
#pragma unroll
        for (int k = 1; k < kHalf; ++k) mx = fmaxf(mx, sv[k]);
        if constexpr (kGroups == 2) {
          s.half_max[bs][h][r] = mx;
          named_barrier_sync(1, C::kSoftmaxThreads);
          mx = fmaxf(mx, s.half_max[bs][1 - h][r]);
        }
        const float m_new = mx * kLog2e;
        const bool move = m_new > m + kSlack;
        const bool rescale = move && m != -INFINITY;
        if (__any_sync(0xffffffffu, rescale)) {
          if (ok && j >= 1)
            ok = __all_sync(0xffffffffu,
                            mbar_wait_fast(&s.p_empty[(j - 1) % C::kPBufs], ((j - 1) / C::kPBufs) & 1));
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
        float ls = 0.f;
#pragma unroll
        for (int k = 0; k < kHalf; ++k) {
          sv[k] = ex2_approx(fmaf(sv[k], kLog2e, -m_use));
          ls += sv[k];
        }
        l += ls;

        // P row into buffer pb once P V of step j - kPBufs has read it
        if (ok && j >= C::kPBufs)
          ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.p_empty[pb], ((j / C::kPBufs) - 1) & 1));
#pragma unroll
        for (int kc = 0; kc < kHalf / 16; ++kc) {
          uint32_t w[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(sv[16 * kc + 2 * e], sv[16 * kc + 2 * e + 1]);
          tmem_st8(t_row + C::kPCol + (C::kKeys / 2) * pb + kc0 / 2 + 8 * kc, w);
        }
        tmem_wait_st();
        // zero this CTA's V rows outside [k_lo, k_hi] (the first and last
        // steps) once its V tile has landed
        if (step0 < k_lo || step0 + C::kKeys - 1 > k_hi) {
          if (ok) ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.v_full[j % kStages], (j / kStages) & 1));
          const uint32_t v_base = smem_addr(s.v[j % kStages]);
#pragma unroll 1
          for (int it = st; it < C::kKeys * 8; it += C::kSoftmaxThreads) {
            const int kr = it >> 3;  // key row of the step
            const int key = step0 + kr;
            if (key < k_lo || key > k_hi) {
#pragma unroll
              for (int ch = 0; ch < C::kVChunksHalf; ++ch)
                st_shared_v4(v_base + (kr >> 4) * C::kVPage + ch * C::kPageChunk + (kr & 15) * 128 + (it & 7) * 16,
                             make_uint4(0, 0, 0, 0));
            }
          }
          fence_proxy_async_smem();
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.p_full[pb]);
      }

      // ---- epilogue: wait for the last P V products, normalise, write this row's output dims ----
      for (int j = n_steps >= C::kPBufs ? n_steps - C::kPBufs : 0; j < n_steps; ++j)
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_fast(&s.p_empty[j % C::kPBufs], (j / C::kPBufs) & 1));
      if (!ok && lane == 0) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
      tc_fence_after_sync();
      if constexpr (kGroups == 2) {
        s.half_sum[h][r] = l;
        named_barrier_sync(1, C::kSoftmaxThreads);
        l += s.half_sum[1 - h][r];
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const size_t o_off = (static_cast<size_t>(q0 + i0 + qi) * kHq + head) * kD + slice * kDS;
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
  }

  // ---------------- teardown: both CTAs done, then free the pair's tensor memory ----------------
  tc_fence_before_sync();
  cluster_sync_all();
  if (warp == 5) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
}

// Gemma-4-12B shapes.  Sliding: each CTA 64 queries x 2 heads, D = 256, its
// stage 8 KB of K (one page) and 8 KB of V (128 dims of two pages), 8
// stages, two softmax warpgroups.  Global: each CTA 8 queries x 16 heads, D
// = 512 split into two slices of 256 output dims (both compute S), 4-page
// steps (N = 64), K and V rings of 2 tiles (32 KB and 16 KB per CTA), one
// softmax warpgroup, the step order rotated by pair, one S issuer, two S
// buffers of 64 columns and three P buffers of 32 (O 256 + 128 + 96 of the
// 512 tensor-memory columns).  On a 4096-token chunk of a 32768-token
// context: 1023-1026 TFLOP/s, against 1018-1020 with two P buffers and
// 789-791 with 2-page steps (two S issuers, 4 stages) on one box.
using SlidingPairConfig =
    PairConfig<ATTN_SLIDING_D, ATTN_SLIDING_D, ATTN_SLIDING_HQ / ATTN_SLIDING_HKV, ATTN_SLIDING_HKV, 8, 2, 0>;
using GlobalPairConfig =
    PairConfig<ATTN_GLOBAL_D, 256, ATTN_GLOBAL_HQ / ATTN_GLOBAL_HKV, ATTN_GLOBAL_HKV, 2, 1, 7, 2, 3, 1, 4>;

}  // namespace prefill_pair
}  // namespace pda
