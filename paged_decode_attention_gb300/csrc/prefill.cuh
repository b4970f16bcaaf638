// prefill.cuh -- multi-query attention over the paged cache: the last n tokens
// of a sequence of L cached tokens query the cache, which already holds their
// keys and values (Attention.lean `causalGQA` / `slidingGQA` with S > 1):
//
//   query i of the sequence sits at position p = L - n + i and sees key l
//   iff l <= p (and p - window < l with a window); scale 1; query head
//   c*G + g reads KV head c.
//
// Block (tile, c, b): queries [tile*kQT, tile*kQT + kQT) of sequence b, KV
// head c.  Its rows (query, head) form row-groups of 16, the M of the
// m16n8k16 tensor-core products:
//   * global layers (G = 16): a row-group is the 16 heads of one query;
//   * sliding layers (G = 2): a row-group is 8 queries x 2 heads, row r being
//     head r / 8 of query r % 8, so the two rows a lane holds (r and r + 8)
//     belong to one query and share its mask.
// Each row-group has kD / 128 warps, each owning 128 of the D dims: a warp
// computes its partial S = q k^T over its dims for the page's 16 keys, the
// partials are summed through shared memory in a fixed order, every warp of
// the group runs the same online softmax (running max in log2 units), and
// accumulates P V for its own 128 output dims.
//
// Warp kConsumerWarps (producer) streams the pages holding keys
// [k_lo, k_hi], the union of the block's visible ranges, one 3-D TMA copy
// per pool per page: the page's 16 rows of this KV head's D dims land as
// D / 64 tiles of [16 rows][64 dims] with the 128-byte swizzle, the layout
// the ldmatrix reads below expect.  Key rows outside [k_lo, k_hi] of the
// first and last page (other positions, or slots past L) are zeroed in shared
// memory before the P V product, since 0 * NaN would be NaN; masked logits
// are selected to -inf.
#pragma once

#include "common.cuh"

namespace pda {
namespace prefill {

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
  int32_t out_f32;
};

template <int kD_, int kG_, int kHkv_, int kRowGroups_, int kStages_>
struct Config {
  static constexpr int kD = kD_;
  static constexpr int kG = kG_;
  static constexpr int kHkv = kHkv_;
  static constexpr int kHq = kG * kHkv;
  static constexpr int kRowGroups = kRowGroups_;
  static constexpr int kStages = kStages_;
  static constexpr int kDimWarps = kD / 128;            // warps per row-group
  static constexpr int kConsumerWarps = kRowGroups * kDimWarps;
  static constexpr int kThreads = (kConsumerWarps + 1) * 32;
  static constexpr int kQPG = 16 / kG;                  // queries per row-group
  static constexpr int kQT = kRowGroups * kQPG;         // queries per block
  static constexpr int kChunks = kD / 64;               // [16][64] tiles per page
  static constexpr int kChunkBytes = kPage * 64 * 2;    // 2 KB
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static_assert(16 % kG == 0 && kD % 128 == 0, "row-groups of 16 rows, warps of 128 dims");
  static_assert(kConsumerWarps + 1 <= 16 && kRowGroups + 2 <= 16, "named barrier ids");

  struct Smem {
    alignas(1024) uint8_t k[kStages][kTileBytes];
    alignas(1024) uint8_t v[kStages][kTileBytes];
    alignas(16) float4 xs[2][kRowGroups][kDimWarps][2][32];  // partial-S exchange, double-buffered
    alignas(8) uint64_t full[kStages];
    alignas(8) uint64_t empty[kStages];
  };
  static constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // + alignment slack
};

// byte offset of 16-byte unit `unit` of row `row` in a 128B-swizzled [16][64] tile
__device__ __forceinline__ uint32_t swz(int row, int unit) { return row * 128 + ((unit ^ (row & 7)) << 4); }

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

template <typename C>
__global__ void __launch_bounds__(C::kThreads)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ PrefillParams p) {
  constexpr int kD = C::kD, kG = C::kG, kHq = C::kHq, kQPG = C::kQPG, kQT = C::kQT;
  constexpr int kStages = C::kStages, kDimWarps = C::kDimWarps, kConsumerWarps = C::kConsumerWarps;
  constexpr int kChunkBytes = C::kChunkBytes;
  extern __shared__ uint8_t smem_raw[];
  typename C::Smem& s =
      *reinterpret_cast<typename C::Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tile = blockIdx.x;
  const int c = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&s.full[st], 1);
      mbar_init(&s.empty[st], kConsumerWarps);
    }
    fence_mbar_init();
  }
  if (warp == kConsumerWarps && lane == 0) {
    prefetch_tensor_map(&tm_k);
    prefetch_tensor_map(&tm_v);
  }
  __syncthreads();
  // q, the cache and the tables may be written by the previous kernel in the stream.
  wait_for_primary_grid();
  allow_dependent_launch();

  // ---- this block's queries and the keys they can see (uniform) ----
  const int q0 = p.cu_q[b];
  const int n = p.cu_q[b + 1] - q0;
  const int i0 = tile * kQT;
  if (n < 0 || q0 < 0 || static_cast<int64_t>(q0) + n > p.total_q) {
    if (threadIdx.x == 0) report(p.status, ATTN_DEV_BAD_SEQ_LEN);
    return;
  }
  if (tile + 1 == static_cast<int>(gridDim.x) && i0 + kQT < n && threadIdx.x == 0)
    report(p.status, ATTN_DEV_BAD_SEQ_LEN);  // more queries than the host's max_q: the rest are not computed
  if (i0 >= n) return;
  const int L = p.seq_lens[b];
  const int cap = p.max_blocks < ATTN_MAX_SEQ_LEN / kPage ? p.max_blocks * kPage : ATTN_MAX_SEQ_LEN;
  if (L < n || L > cap) {
    if (threadIdx.x == 0) report(p.status, ATTN_DEV_BAD_SEQ_LEN);
    return;
  }
  const int P0 = L - n + i0;                       // position of the block's first query
  const int nq = n - i0 < kQT ? n - i0 : kQT;      // valid queries in the block
  const int k_hi = P0 + nq - 1;                    // last visible key (inclusive)
  const int k_lo = p.window > 0 ? (P0 - p.window + 1 > 0 ? P0 - p.window + 1 : 0) : 0;
  const int page0 = k_lo / kPage;
  const int n_pages = k_hi / kPage - page0 + 1;

  if (warp == kConsumerWarps) {
    // ---------------- producer ----------------
    const int32_t* bt = p.block_table + static_cast<int64_t>(b) * p.max_blocks;
    int nxt = lane < n_pages ? bt[page0 + lane] : 0;
    int cur = 0;
    bool ok = true;
    int issued = 0;
    for (int i = 0; i < n_pages; ++i) {
      if ((i & 31) == 0) {
        cur = nxt;
        nxt = i + 32 + lane < n_pages ? bt[page0 + i + 32 + lane] : 0;
      }
      const int phys = __shfl_sync(0xffffffffu, cur, i & 31);
      const int stage = i % kStages;
      if (i >= kStages) {
        const int w = lane == 0 ? static_cast<int>(mbar_wait(&s.empty[stage], ((i / kStages) - 1) & 1)) : 0;
        ok = __shfl_sync(0xffffffffu, w, 0) != 0;
      }
      if (!ok) {
        if (lane == 0) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
        break;
      }
      if (lane == 0) {
        int32_t y;
        if (phys < 0 || static_cast<int64_t>(phys) >= p.num_pages) {
          report(p.status, ATTN_DEV_BAD_PAGE);
          y = -kPage;  // fully out of range: the copy fills zeros
        } else {
          y = phys * kPage;
        }
        mbar_arrive_expect_tx(&s.full[stage], 2 * C::kTileBytes);
        tma_load_3d(s.k[stage], &tm_k, 0, y, c * C::kChunks, &s.full[stage]);
        tma_load_3d(s.v[stage], &tm_v, 0, y, c * C::kChunks, &s.full[stage]);
      }
      ++issued;
      __syncwarp();
    }
    if (lane == 0) {
      for (int st = 0; st < kStages && st < issued; ++st) {
        const int uses = (issued - 1 - st) / kStages + 1;
        if (!mbar_wait(&s.full[st], (uses - 1) & 1)) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
      }
    }
    return;
  }

  // ---------------- consumers ----------------
  const int rg = warp / kDimWarps;  // row-group
  const int dw = warp % kDimWarps;  // which 128 dims
  const int g = lane >> 2;          // fragment rows g and g + 8
  const int tq = lane & 3;
  const int mi = lane >> 3;         // ldmatrix: which 8x8 matrix this lane addresses
  const int lr = lane & 7;

  // rows g and g + 8 of the group: (query, head) and the query's position
  int qi[2], head[2], pos[2];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int r = g + 8 * rr;
    qi[rr] = rg * kQPG + r % kQPG;  // query index within the block
    head[rr] = c * kG + r / kQPG;
    pos[rr] = qi[rr] < nq ? P0 + qi[rr] : -1;  // -1: no such query, nothing visible
  }
  // positions range of the group's valid queries, for the page-level mask test
  const int grp_first = rg * kQPG < nq ? P0 + rg * kQPG : -1;
  const int grp_last = P0 + (rg * kQPG + kQPG - 1 < nq ? rg * kQPG + kQPG - 1 : nq - 1);
  const int grp_lo = p.window > 0 ? grp_last - p.window + 1 : 0;  // every query of the group sees [grp_lo, grp_first]

  // q as m16n8k16 A fragments over this warp's 128 dims (8 k-steps of 16)
  uint32_t qa[8][4];
  {
    const uint32_t* qr[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
      qr[rr] = qi[rr] < nq
                   ? reinterpret_cast<const uint32_t*>(p.q + (static_cast<size_t>(q0 + i0 + qi[rr]) * kHq + head[rr]) * kD)
                   : nullptr;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int d = dw * 128 + ks * 16 + 2 * tq;
      qa[ks][0] = qr[0] ? __ldg(qr[0] + d / 2) : 0u;
      qa[ks][1] = qr[1] ? __ldg(qr[1] + d / 2) : 0u;
      qa[ks][2] = qr[0] ? __ldg(qr[0] + (d + 8) / 2) : 0u;
      qa[ks][3] = qr[1] ? __ldg(qr[1] + (d + 8) / 2) : 0u;
    }
  }

  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float acc[16][4];
#pragma unroll
  for (int nn = 0; nn < 16; ++nn)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nn][e] = 0.f;
  bool ok = true;

  for (int i = 0; i < n_pages; ++i) {
    const int stage = i % kStages;
    if (ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(&s.full[stage], (i / kStages) & 1));
      if (!ok && lane == 0) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
    }
    const int pos0 = (page0 + i) * kPage;
    const uint32_t kst = smem_addr(s.k[stage]);
    const uint32_t vst = smem_addr(s.v[stage]);

    // ---- partial S over this warp's dims: two n-tiles of 8 keys; even and
    //      odd k-steps accumulate separately, K fragments read two ahead ----
    float se[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float so[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      auto k_frag = [&](int ks, uint32_t (&bb)[4]) {
        const int ch = 2 * dw + (ks >> 2);
        const int row = ((mi >> 1) << 3) + lr;
        const int unit = 2 * (ks & 3) + (mi & 1);
        ldmatrix_x4(kst + ch * kChunkBytes + swz(row, unit), bb[0], bb[1], bb[2], bb[3]);
      };
      uint32_t kb[3][4];
      k_frag(0, kb[0]);
      k_frag(1, kb[1]);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        if (ks + 2 < 8) k_frag(ks + 2, kb[(ks + 2) % 3]);
        const uint32_t (&bb)[4] = kb[ks % 3];
        float (&s0)[4] = (ks & 1) ? so[0] : se[0];
        float (&s1)[4] = (ks & 1) ? so[1] : se[1];
        mma_bf16_16816(s0, qa[ks], bb[0], bb[1]);
        mma_bf16_16816(s1, qa[ks], bb[2], bb[3]);
      }
    }

    // ---- sum the group's partials in a fixed order ----
    const int buf = i & 1;
    s.xs[buf][rg][dw][0][lane] =
        make_float4(se[0][0] + so[0][0], se[0][1] + so[0][1], se[0][2] + so[0][2], se[0][3] + so[0][3]);
    s.xs[buf][rg][dw][1][lane] =
        make_float4(se[1][0] + so[1][0], se[1][1] + so[1][1], se[1][2] + so[1][2], se[1][3] + so[1][3]);
    named_barrier_sync(1 + rg, kDimWarps * 32);
    float sc[2][4];
    {
      float4 a0 = s.xs[buf][rg][0][0][lane], a1 = s.xs[buf][rg][0][1][lane];
#pragma unroll
      for (int w = 1; w < kDimWarps; ++w) {
        const float4 c0 = s.xs[buf][rg][w][0][lane], c1 = s.xs[buf][rg][w][1][lane];
        a0.x += c0.x; a0.y += c0.y; a0.z += c0.z; a0.w += c0.w;
        a1.x += c1.x; a1.y += c1.y; a1.z += c1.z; a1.w += c1.w;
      }
      sc[0][0] = a0.x; sc[0][1] = a0.y; sc[0][2] = a0.z; sc[0][3] = a0.w;
      sc[1][0] = a1.x; sc[1][1] = a1.y; sc[1][2] = a1.z; sc[1][3] = a1.w;
    }

    // ---- masks: sc[nt][e] is row g + 8*(e>>1), key pos0 + 8*nt + 2*tq + (e&1) ----
    if (grp_first < 0 || pos0 < grp_lo || pos0 + kPage - 1 > grp_first) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = pos0 + 8 * nt + 2 * tq + (e & 1);
          const int pr = pos[e >> 1];
          const bool vis = key <= pr && (p.window <= 0 || key > pr - p.window);
          if (!vis) sc[nt][e] = -INFINITY;
        }
    }

    // ---- online softmax (log2 units), exact running max ----
    float mx[2];
    mx[0] = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
    mx[1] = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
    float scale[2] = {1.f, 1.f};
    if (__any_sync(0xffffffffu, mx[0] * kLog2e > m[0] || mx[1] * kLog2e > m[1])) {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
        mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
        const float m_new = fmaxf(m[rr], mx[rr] * kLog2e);
        scale[rr] = m_new == m[rr] ? 1.f : ex2_approx(m[rr] - m_new);  // 0 on a row's first visible key
        m[rr] = m_new;
      }
    }
    float m_use[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) m_use[rr] = m[rr] == -INFINITY ? 0.f : m[rr];
    float pr[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) pr[nt][e] = ex2_approx(fmaf(sc[nt][e], kLog2e, -m_use[e >> 1]));
    l[0] = l[0] * scale[0] + ((pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]));
    l[1] = l[1] * scale[1] + ((pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]));
    if (__any_sync(0xffffffffu, scale[0] != 1.f || scale[1] != 1.f)) {
#pragma unroll
      for (int nn = 0; nn < 16; ++nn) {
        acc[nn][0] *= scale[0];
        acc[nn][1] *= scale[0];
        acc[nn][2] *= scale[1];
        acc[nn][3] *= scale[1];
      }
    }
    const uint32_t pa[4] = {pack_bf16x2(pr[0][0], pr[0][1]), pack_bf16x2(pr[0][2], pr[0][3]),
                            pack_bf16x2(pr[1][0], pr[1][1]), pack_bf16x2(pr[1][2], pr[1][3])};

    // ---- zero the V rows outside [k_lo, k_hi] of the first and last page:
    //      row-group 0 writes, every consumer waits before reading V ----
    if (pos0 < k_lo || pos0 + kPage - 1 > k_hi) {
      if (rg == 0) {
#pragma unroll 1
        for (int rr = 0; rr < kPage; ++rr) {
          const int key = pos0 + rr;
          if ((key < k_lo || key > k_hi) && lane < 16) {
            const int ch = 2 * dw + (lane >> 3);
            st_shared_v4(vst + ch * kChunkBytes + rr * 128 + (lane & 7) * 16, make_uint4(0, 0, 0, 0));
          }
        }
        fence_proxy_async_smem();  // before TMA rewrites this stage
      }
      named_barrier_sync(1 + C::kRowGroups, kConsumerWarps * 32);
    }

    // ---- O += P V over this warp's 128 dims, V fragments read two ahead ----
    {
      auto v_frag = [&](int np, uint32_t (&bb)[4]) {
        const int ch = 2 * dw + (np >> 2);
        const int row = ((mi & 1) << 3) + lr;
        const int unit = 2 * (np & 3) + (mi >> 1);
        ldmatrix_x4_trans(vst + ch * kChunkBytes + swz(row, unit), bb[0], bb[1], bb[2], bb[3]);
      };
      uint32_t vb[3][4];
      v_frag(0, vb[0]);
      v_frag(1, vb[1]);
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        if (np + 2 < 8) v_frag(np + 2, vb[(np + 2) % 3]);
        const uint32_t (&bb)[4] = vb[np % 3];
        mma_bf16_16816(acc[2 * np], pa, bb[0], bb[1]);
        mma_bf16_16816(acc[2 * np + 1], pa, bb[2], bb[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.empty[stage]);
  }

  // ---- normalise and write this warp's 128 dims of rows g and g + 8 ----
  float lt[2];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    lt[rr] = l[rr] + __shfl_xor_sync(0xffffffffu, l[rr], 1);
    lt[rr] += __shfl_xor_sync(0xffffffffu, lt[rr], 2);
  }
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    if (qi[rr] >= nq) continue;
    const float inv = lt[rr] > 0.f ? 1.f / lt[rr] : 0.f;
    const size_t row = static_cast<size_t>(q0 + i0 + qi[rr]) * kHq + head[rr];
#pragma unroll
    for (int nn = 0; nn < 16; ++nn) {
      const int d = dw * 128 + 8 * nn + 2 * tq;
      const float a = acc[nn][2 * rr] * inv, bv = acc[nn][2 * rr + 1] * inv;
      if (p.out_f32) {
        *reinterpret_cast<float2*>(static_cast<float*>(p.o) + row * kD + d) = make_float2(a, bv);
      } else {
        *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(p.o) + row * kD + d) = pack_bf16x2(a, bv);
      }
    }
  }
}

// Gemma-4-12B shapes: sliding layers 16/8 heads of 256 (5 row-groups = 40
// queries per block), global layers 16/1 heads of 512 (2 row-groups = 2
// queries per block).  Both at one block per SM (168 registers per thread).
using SlidingConfig = Config<ATTN_SLIDING_D, ATTN_SLIDING_HQ / ATTN_SLIDING_HKV, ATTN_SLIDING_HKV, 5, 6>;
using GlobalConfig = Config<ATTN_GLOBAL_D, ATTN_GLOBAL_HQ / ATTN_GLOBAL_HKV, ATTN_GLOBAL_HKV, 2, 4>;

}  // namespace prefill
}  // namespace pda
