// global.cuh -- decode kernel for the Gemma-4-12B global layers (decodeGQA:
// 16 query heads over 1 KV head, D = 512, G = 16, scale 1).
//
// With G = 16 every K/V byte feeds 16 query heads (16 flop per byte), more
// than the CUDA cores sustain at HBM speed, so both contractions run on
// tensor cores (bf16 in, fp32 accumulate):
//   S[h, l]  = sum_d q[h, d] K[l, d]     A = q (16 x 512), B = K^T per page
//   O[h, d] += sum_l P[h, l] V[l, d]     A = P (16 x 16),  B = V per page
//
// Grid (grid_x): block g streams its span of the flattened visible pages
// (balanced schedule, common.cuh):
//   * warp 4 (producer) issues, per page, 8 TMA tensor copies for K and 8
//     for V: boxes of 16 rows x 64 dims (2 KB) of the pool viewed as
//     [num_pages*16 rows, 512], written with the 128-byte swizzle so that the
//     ldmatrix reads below are free of bank conflicts;
//   * warps 0..3 (consumers) each own 128 of the 512 dims: a warp computes
//     its partial S over its dims, the four partials are summed through
//     shared memory in a fixed order (so every warp holds the bitwise-same
//     S), each warp runs the same online softmax, and accumulates P*V for its
//     own 128 output dims; since all warps share (max, sum), each writes its
//     slice of o (or of the partial) with no further merge.
// Masking selects: logits of rows outside [lo, L) become -inf, and V rows
// outside [lo, L) of a partial page are overwritten with zeros in shared
// memory before the P*V product (0 * NaN would be NaN).
#pragma once

#include "common.cuh"

namespace pda {
namespace global {

constexpr int kHq = ATTN_GLOBAL_HQ;  // 16
constexpr int kD = ATTN_GLOBAL_D;    // 512
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kDimsPerWarp = kD / kConsumerWarps;  // 128
constexpr int kChunk = 64;                          // dims per TMA box (128-byte rows)
constexpr int kChunks = kD / kChunk;                // 8
constexpr int kChunkBytes = kPage * kChunk * 2;     // 2 KB
constexpr int kPageBytes = kPage * kD * 2;          // 16 KB
constexpr int kStages = 3;
constexpr int kBlocksPerSm = 2;
constexpr int kMinPages = 4;
constexpr int kWarmPages = 2;  // pages per block pulled into L2 before the wait (32 KB each)
constexpr int kAhead = 2;  // ldmatrix fragments read ahead of their MMAs

static_assert(kHq == 16, "the m16n8k16 tiling uses the 16 query heads as the M dimension");

struct Smem {
  alignas(1024) uint8_t k[kStages][kPageBytes];  // kChunks tiles of [16 rows][64 dims], swizzled
  alignas(1024) uint8_t v[kStages][kPageBytes];
  alignas(16) float4 xs[2][kConsumerWarps][2][32];  // partial-S exchange, double-buffered
  SeqTable table;
  alignas(8) uint64_t full[kStages];
  alignas(8) uint64_t empty[kStages];
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // + alignment slack

// byte offset of 16-byte unit `unit` of row `row` in a 128B-swizzled [16][64] tile
__device__ __forceinline__ uint32_t swz(int row, int unit) {
  return row * 128 + ((unit ^ (row & 7)) << 4);
}

__global__ void __launch_bounds__(kThreads)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int gb = blockIdx.x;
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
  // With a programmatic launch this prologue overlaps the previous kernel in
  // the stream, whose writes (q, the cache, the tables, the workspace it
  // reads) are complete and visible only once griddepcontrol.wait returns.
  // Until then the block writes nothing outside its shared memory: it builds
  // the schedule from hint reads and pulls its first pages into L2.
  build_seq_table_hint(p, s.table, gb);  // ends with __syncthreads
  if (warp == kConsumerWarps) {
    warm_first_pages(p, s.table, kWarmPages, [&](int32_t y) {
      // a page is 16 contiguous rows of D elements in each pool
      bulk_prefetch_l2(p.k_pool + static_cast<size_t>(y) * kD, kPageBytes);
      bulk_prefetch_l2(p.v_pool + static_cast<size_t>(y) * kD, kPageBytes);
    });
  } else {
    warm_q(p, s.table, kHq * kD, 0, kHq * kD * 2, kConsumerWarps * 32);
  }
  wait_for_primary_grid();
  allow_dependent_launch();
  // The producer reads its first block-table entries while warp 0 confirms
  // the table; it reads them again if the table had to be rebuilt.
  int first = warp == kConsumerWarps ? page_entry(p, s.table, s.table.span, lane, false) : 0;
  confirm_seq_table(p, s.table, gb);  // ends with __syncthreads
  const SeqTable& t = s.table;
  const Span sp = t.span;
  const int n_pages = sp.end - sp.begin;
  if (n_pages <= 0) return;

  if (warp == kConsumerWarps) {
    // ---------------- producer ----------------
    const uint64_t policy = l2_policy_evict_first();
    if (t.rebuilt) first = page_entry(p, t, sp, lane, true);
    produce_pages<kStages, 2 * kPageBytes>(p, t, sp, s.full, s.empty, first, [&](int stage, int32_t y) {
      // one copy per pool: the page's 16 rows as kChunks tiles of [16][64]
      tma_load_3d_hint(s.k[stage], &tm_k, 0, y, 0, &s.full[stage], policy);
      tma_load_3d_hint(s.v[stage], &tm_v, 0, y, 0, &s.full[stage], policy);
    });
    return;
  }

  // ---------------- consumers ----------------
  const int g = lane >> 2;  // fragment row: query heads g and g + 8
  const int tq = lane & 3;  // fragment column pair
  const int dim0 = warp * kDimsPerWarp;
  const int mi = lane >> 3;  // ldmatrix: which 8x8 matrix this lane addresses
  const int lr = lane & 7;

  PageCursor cur;
  cur.start(p, t, sp);

  // q as m16n8k16 A fragments over this warp's 128 dims (8 k-steps of 16)
  uint32_t qa[8][4];
  auto load_q = [&]() {
    const uint32_t* q_g = reinterpret_cast<const uint32_t*>(p.q + (static_cast<size_t>(cur.b) * kHq + g) * kD);
    const uint32_t* q_g8 = q_g + 8 * kD / 2;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int d = dim0 + ks * 16 + 2 * tq;
      qa[ks][0] = __ldg(q_g + d / 2);
      qa[ks][1] = __ldg(q_g8 + d / 2);
      qa[ks][2] = __ldg(q_g + (d + 8) / 2);
      qa[ks][3] = __ldg(q_g8 + (d + 8) / 2);
    }
  };
  // Pull q of the span's next sequence into L2 while this one runs, so its
  // reload at the sequence boundary is an L2 hit (16 KB = 128 lines of 128
  // bytes; the 128 consumer threads take one line each).
  auto prefetch_next_q = [&]() {
    const int nb = next_seq_in_span(p, t, sp, cur.b);
    if (nb >= 0)
      prefetch_l2(reinterpret_cast<const uint8_t*>(p.q + static_cast<size_t>(nb) * kHq * kD) + threadIdx.x * 128);
  };
  load_q();
  prefetch_next_q();

  float m[2], l[2];  // rows g, g+8: running max (log2 units), this thread's share of the sum
  float acc[16][4];  // 16 n-tiles of 8 dims
  auto reset = [&]() {
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
#pragma unroll
    for (int n = 0; n < 16; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
  };
  reset();
  bool ok = true;

  for (int i = 0; i < n_pages; ++i) {
    const int f = sp.begin + i;
    if (f >= t.prefix[cur.b + 1]) {
      cur.advance(p, t, sp, f);
      load_q();
      prefetch_next_q();
    }
    const int stage = i % kStages;
    if (ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(&s.full[stage], (i / kStages) & 1));
      if (!ok && lane == 0) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
    }
    const int pos0 = cur.pos0(t, f);
    const uint32_t kst = smem_addr(s.k[stage]);
    const uint32_t vst = smem_addr(s.v[stage]);

    // ---- partial S over this warp's dims: two n-tiles of 8 positions; even
    //      and odd k-steps accumulate separately (two chains of 4 MMAs) ----
    //      The K fragments are read kAhead k-steps before their MMAs.
    float se[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float so[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      auto k_frag = [&](int ks, uint32_t (&b)[4]) {
        const int ch = 2 * warp + (ks >> 2);
        const int row = ((mi >> 1) << 3) + lr;
        const int unit = 2 * (ks & 3) + (mi & 1);
        ldmatrix_x4(kst + ch * kChunkBytes + swz(row, unit), b[0], b[1], b[2], b[3]);
      };
      uint32_t kb[kAhead + 1][4];
#pragma unroll
      for (int ks = 0; ks < kAhead; ++ks) k_frag(ks, kb[ks]);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        if (ks + kAhead < 8) k_frag(ks + kAhead, kb[(ks + kAhead) % (kAhead + 1)]);
        const uint32_t (&b)[4] = kb[ks % (kAhead + 1)];
        float (&s0)[4] = (ks & 1) ? so[0] : se[0];
        float (&s1)[4] = (ks & 1) ? so[1] : se[1];
        mma_bf16_16816(s0, qa[ks], b[0], b[1]);
        mma_bf16_16816(s1, qa[ks], b[2], b[3]);
      }
    }

    // ---- sum the four partials in a fixed order ----
    const int buf = i & 1;
    s.xs[buf][warp][0][lane] =
        make_float4(se[0][0] + so[0][0], se[0][1] + so[0][1], se[0][2] + so[0][2], se[0][3] + so[0][3]);
    s.xs[buf][warp][1][lane] =
        make_float4(se[1][0] + so[1][0], se[1][1] + so[1][1], se[1][2] + so[1][2], se[1][3] + so[1][3]);
    named_barrier_sync(1, kConsumerWarps * 32);
    float sc[2][4];
    {
      float4 a0 = s.xs[buf][0][0][lane], a1 = s.xs[buf][0][1][lane];
#pragma unroll
      for (int w = 1; w < kConsumerWarps; ++w) {
        const float4 c0 = s.xs[buf][w][0][lane], c1 = s.xs[buf][w][1][lane];
        a0.x += c0.x; a0.y += c0.y; a0.z += c0.z; a0.w += c0.w;
        a1.x += c1.x; a1.y += c1.y; a1.z += c1.z; a1.w += c1.w;
      }
      sc[0][0] = a0.x; sc[0][1] = a0.y; sc[0][2] = a0.z; sc[0][3] = a0.w;
      sc[1][0] = a1.x; sc[1][1] = a1.y; sc[1][2] = a1.z; sc[1][3] = a1.w;
    }

    // ---- masked online softmax (log2 units) ----
    // sc[nt][e]: head g + 8*(e>>1), position pos0 + 8*nt + 2*tq + (e&1).
    // Positions outside [lo, L) get -inf (pages inside the range skip the
    // test); the factor log2(e) is applied inside the exponent.
    if (pos0 < cur.lo || pos0 + kPage > cur.L) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int pos = pos0 + 8 * nt + 2 * tq + (e & 1);
          if (pos < cur.lo || pos >= cur.L) sc[nt][e] = -INFINITY;
        }
    }
    float mx[2];
    mx[0] = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
    mx[1] = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
    // The running max of a row changes only when some score exceeds it, which
    // after a sequence's first pages is rare: one vote decides whether the
    // row maxima over the four lanes that share a row are needed at all.
    // Tracking the exact max keeps the largest weight at exactly 1, so the
    // dominant term of P carries no bf16 rounding.
    float scale[2] = {1.f, 1.f};
    if (__any_sync(0xffffffffu, mx[0] * kLog2e > m[0] || mx[1] * kLog2e > m[1])) {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
        mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
        const float m_new = fmaxf(m[rr], mx[rr] * kLog2e);
        scale[rr] = m_new == m[rr] ? 1.f : ex2_approx(m[rr] - m_new);  // 0 on the first visible page
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
    // rescale only when some row's running max moved (multiplying by 1 is exact)
    if (__any_sync(0xffffffffu, scale[0] != 1.f || scale[1] != 1.f)) {
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        acc[n][0] *= scale[0];
        acc[n][1] *= scale[0];
        acc[n][2] *= scale[1];
        acc[n][3] *= scale[1];
      }
    }
    // P as the A fragment of one k16 step (k = the page's 16 positions)
    const uint32_t pa[4] = {pack_bf16x2(pr[0][0], pr[0][1]), pack_bf16x2(pr[0][2], pr[0][3]),
                            pack_bf16x2(pr[1][0], pr[1][1]), pack_bf16x2(pr[1][2], pr[1][3])};

    // ---- zero V rows outside [lo, L) in this warp's two chunks ----
    if (pos0 < cur.lo || pos0 + kPage > cur.L) {
#pragma unroll 1
      for (int rr = 0; rr < kPage; ++rr) {
        const int pos = pos0 + rr;
        if ((pos < cur.lo || pos >= cur.L) && lane < 16) {
          const int ch = 2 * warp + (lane >> 3);
          st_shared_v4(vst + ch * kChunkBytes + rr * 128 + (lane & 7) * 16, make_uint4(0, 0, 0, 0));
        }
      }
      fence_proxy_async_smem();  // before TMA rewrites this stage
      __syncwarp();
    }

    // ---- O += P V over this warp's 128 dims ----
    {
      auto v_frag = [&](int np, uint32_t (&b)[4]) {
        const int ch = 2 * warp + (np >> 2);
        const int row = ((mi & 1) << 3) + lr;
        const int unit = 2 * (np & 3) + (mi >> 1);
        ldmatrix_x4_trans(vst + ch * kChunkBytes + swz(row, unit), b[0], b[1], b[2], b[3]);
      };
      uint32_t vb[kAhead + 1][4];
#pragma unroll
      for (int np = 0; np < kAhead; ++np) v_frag(np, vb[np]);
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        if (np + kAhead < 8) v_frag(np + kAhead, vb[(np + kAhead) % (kAhead + 1)]);
        const uint32_t (&b)[4] = vb[np % (kAhead + 1)];
        mma_bf16_16816(acc[2 * np], pa, b[0], b[1]);
        mma_bf16_16816(acc[2 * np + 1], pa, b[2], b[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.empty[stage]);

    if (f + 1 == cur.seg_end) {
      // ---------------- finish this sequence's segment ----------------
      float lt[2];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        lt[rr] = l[rr] + __shfl_xor_sync(0xffffffffu, l[rr], 1);
        lt[rr] += __shfl_xor_sync(0xffffffffu, lt[rr], 2);
      }
      if (cur.whole(t, sp)) {
        const size_t row0 = static_cast<size_t>(cur.b) * kHq + g;
        const float inv0 = lt[0] > 0.f ? 1.f / lt[0] : 0.f;
        const float inv1 = lt[1] > 0.f ? 1.f / lt[1] : 0.f;
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          const int d = dim0 + 8 * n + 2 * tq;
          store_out2(p, row0 * kD + d, acc[n][0] * inv0, acc[n][1] * inv0);
          store_out2(p, (row0 + 8) * kD + d, acc[n][2] * inv1, acc[n][3] * inv1);
        }
      } else if ((static_cast<int64_t>(gb) + cur.b + 1) * kHq > p.part_rows) {
        if (lane == 0) report(p.status, ATTN_DEV_INTERNAL);  // cannot happen: slot beyond the workspace
      } else {
        const size_t slot0 = (static_cast<size_t>(gb) + cur.b) * kHq + g;
        const size_t slot1 = slot0 + 8;
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          const int d = dim0 + 8 * n + 2 * tq;
          *reinterpret_cast<float2*>(p.part_o + slot0 * kD + d) = make_float2(acc[n][0], acc[n][1]);
          *reinterpret_cast<float2*>(p.part_o + slot1 * kD + d) = make_float2(acc[n][2], acc[n][3]);
        }
        if (warp == 0 && tq == 0) {
          p.part_ml[slot0] = make_float2(m[0], lt[0]);
          p.part_ml[slot1] = make_float2(m[1], lt[1]);
        }
      }
      reset();
    }
  }
}

}  // namespace global
}  // namespace pda
