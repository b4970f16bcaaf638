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
//   * warp 4 (producer) issues, per page, one 3-D TMA tensor copy for K and
//     one for V: the pool viewed as [8 chunks][num_pages*16 rows][64 dims],
//     a box of 8 x 16 x 64 (16 KB) that lands as eight [16 rows][64 dims]
//     tiles with the 128-byte swizzle, so that the ldmatrix reads below are
//     free of bank conflicts;
//   * warps 0..3 (consumers) each own 128 of the 512 dims: a warp computes
//     its partial S over its dims, the four partials are summed through
//     shared memory in a fixed order (so every warp holds the bitwise-same
//     S), each warp runs the same online softmax, and accumulates P*V for its
//     own 128 output dims; since all warps share (max, sum), each writes its
//     slice of o (or of the partial) with no further merge.
// Masking selects: logits of rows outside [lo, L) become -inf, and V rows
// outside [lo, L) of a partial page are overwritten with zeros in shared
// memory before the P*V product (0 * NaN would be NaN).
//
// Values-only cache (decode_kernel_shared).  On global layers keys and values
// come from one head x (Gemma-4-12B model page, "What to watch for": values =
// keys): V = rmsnormUnit(x) and K = rope(rmsnorm(x) * w_k) = rope(V * w_k),
// so the cache may hold V alone and the kernel rebuilds each key, rounded
// once to bf16, from the V page it already has in shared memory.  Only V is
// copied (half the bytes per page).  The rebuilt K never goes to memory: the
// S k-steps are dealt out so that each warp rebuilds exactly the B fragments
// it multiplies.  Warp w takes dims [16w, 16w + 16) of every 64-dim chunk:
// in the rotated chunk 0 and its partner chunk 4 (pairs (j, j + 256)) a lane
// holds both halves of each of its 8 pairs; in chunks 1-3 and 5-7 the key is
// the bf16 product V * w_k.
// The 8 angles per lane and page come from rope.cuh.  Two consecutive pages
// of a segment share one partial-S exchange and one softmax pass; the q
// fragments, w_k and the RoPE frequencies live in shared memory (each lane
// reads back only what it wrote) so that two pages fit in the registers.
#pragma once

#include <type_traits>

#include "common.cuh"
#include "rope.cuh"

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
constexpr int kSharedStages = 4;  // values-only pages are half the size
constexpr int kBlocksPerSm = 2;
constexpr int kRopePairs = ATTN_GLOBAL_ROPE_PAIRS;  // 64: dims [0, 64) turn with [256, 320)
constexpr int kMinPages = 4;
constexpr int kWarmPages = 2;  // pages per block pulled into L2 before the wait (32 KB each)
constexpr int kAhead = 2;  // ldmatrix fragments read ahead of their MMAs

static_assert(kHq == 16, "the m16n8k16 tiling uses the 16 query heads as the M dimension");
static_assert(kRopePairs == kChunk, "the rotated dims are exactly the first chunk and its partner chunk");

// Key rebuild of a values-only cache: w_k and the RoPE frequencies of the
// 64 active pairs, theta^(-2j/D) as float pairs.
struct KeyRebuild {
  const __nv_bfloat16* w_k;  // [512]
  TwoPi two_pi;
  FloatPair freq[kRopePairs];
};

struct KPages {
  alignas(1024) uint8_t k[kStages][kPageBytes];  // kChunks tiles of [16 rows][64 dims], swizzled
};
struct KeyWeights {
  alignas(16) uint4 qfrag[kConsumerWarps][8][32];  // q A fragments: per warp and S k-step, one word per lane
  uint32_t wk[kD / 2];                             // w_k as bf16x2 words
  FloatPair freq[kRopePairs];                      // RoPE frequencies of the active pairs
};

template <bool kShared>
struct Smem : std::conditional_t<kShared, KeyWeights, KPages> {
  static constexpr int kNumStages = kShared ? kSharedStages : kStages;
  alignas(1024) uint8_t v[kNumStages][kPageBytes];
  alignas(16) float4 xs[2][kConsumerWarps][kShared ? 4 : 2][32];  // partial-S exchange (n-tiles), double-buffered
  SeqTable table;
  alignas(8) uint64_t full[kNumStages];
  alignas(8) uint64_t empty[kNumStages];
};

constexpr size_t kSmemBytes = sizeof(Smem<false>) + 1024;  // + alignment slack
constexpr size_t kSharedSmemBytes = sizeof(Smem<true>) + 1024;
// kBlocksPerSm blocks, each with 1 KB reserved by the system, in 228 KB
static_assert(kBlocksPerSm * (kSmemBytes + 1024) <= 228 * 1024 &&
                  kBlocksPerSm * (kSharedSmemBytes + 1024) <= 228 * 1024,
              "shared memory of the resident blocks");

// byte offset of 16-byte unit `unit` of row `row` in a 128B-swizzled [16][64] tile
__device__ __forceinline__ uint32_t swz(int row, int unit) {
  return row * 128 + ((unit ^ (row & 7)) << 4);
}

// bf16x2 product rounded to nearest even (the exact product of two bf16 fits
// in fp32, so this is the product rounded once).
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// First of the 16 dims of S k-step ks of consumer warp w.  Values-only
// cache: dims [16w, 16w + 16) of every chunk, the rotated chunk 0 and its
// partner chunk 4 first.
template <bool kShared>
__device__ __forceinline__ int s_kstep_dim(int w, int ks) {
  if constexpr (kShared) {
    constexpr int kChunkOrder = 0x76532140;  // chunks 0, 4, 1, 2, 3, 5, 6, 7 as nibbles
    return ((kChunkOrder >> (4 * ks)) & 0xF) * kChunk + 16 * w;
  } else {
    return w * kDimsPerWarp + 16 * ks;
  }
}

template <bool kShared>
__device__ __forceinline__ void decode_body(const CUtensorMap* tm_k, const CUtensorMap* tm_v, const DecodeParams& p,
                                            const KeyRebuild* kr) {
  extern __shared__ uint8_t smem_raw[];
  using S = Smem<kShared>;
  constexpr int kNS = S::kNumStages;
  S& s = *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int gb = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int st = 0; st < kNS; ++st) {
      mbar_init(&s.full[st], 1);
      mbar_init(&s.empty[st], kConsumerWarps);
    }
    fence_mbar_init();
  }
  if (warp == kConsumerWarps && lane == 0) {
    if constexpr (!kShared) prefetch_tensor_map(tm_k);
    prefetch_tensor_map(tm_v);
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
      if constexpr (!kShared) bulk_prefetch_l2(p.k_pool + static_cast<size_t>(y) * kD, kPageBytes);
      bulk_prefetch_l2(p.v_pool + static_cast<size_t>(y) * kD, kPageBytes);
    });
  } else {
    warm_q(p, s.table, kHq * kD, 0, kHq * kD * 2, kConsumerWarps * 32);
  }
  wait_for_primary_grid();
  allow_dependent_launch();
  if constexpr (kShared) {
    if (warp < kConsumerWarps) {  // w_k to shared memory; published by confirm_seq_table's barrier
      const uint32_t* w32 = reinterpret_cast<const uint32_t*>(kr->w_k);
      for (int k = threadIdx.x; k < kD / 2; k += kConsumerWarps * 32) s.wk[k] = __ldg(w32 + k);
      if (threadIdx.x < kRopePairs) s.freq[threadIdx.x] = kr->freq[threadIdx.x];
    }
  }
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
    if constexpr (kShared) {
      produce_pages<kNS, kPageBytes>(p, t, sp, s.full, s.empty, first, [&](int stage, int32_t y) {
        tma_load_3d_hint(s.v[stage], tm_v, 0, y, 0, &s.full[stage], policy);
      });
    } else {
      produce_pages<kNS, 2 * kPageBytes>(p, t, sp, s.full, s.empty, first, [&](int stage, int32_t y) {
        // one copy per pool: the page's 16 rows as kChunks tiles of [16][64]
        tma_load_3d_hint(s.k[stage], tm_k, 0, y, 0, &s.full[stage], policy);
        tma_load_3d_hint(s.v[stage], tm_v, 0, y, 0, &s.full[stage], policy);
      });
    }
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

  // q as m16n8k16 A fragments over this warp's 128 S dims (8 k-steps of 16)
  // With a values-only cache each lane parks its fragments in shared memory
  // (it alone reads them back), which frees 32 registers for two-page groups.
  uint32_t qa_reg[kShared ? 1 : 8][4];
  uint32_t qfrag_addr = 0;
  if constexpr (kShared) qfrag_addr = smem_addr(&s.qfrag[warp][0][lane]);
  auto load_q = [&]() {
    const uint32_t* q_g = reinterpret_cast<const uint32_t*>(p.q + (static_cast<size_t>(cur.b) * kHq + g) * kD);
    const uint32_t* q_g8 = q_g + 8 * kD / 2;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int d = s_kstep_dim<kShared>(warp, ks) + 2 * tq;
      const uint4 v = make_uint4(__ldg(q_g + d / 2), __ldg(q_g8 + d / 2), __ldg(q_g + (d + 8) / 2),
                                 __ldg(q_g8 + (d + 8) / 2));
      if constexpr (kShared) {
        st_shared_v4(qfrag_addr + ks * 512, v);
      } else {
        qa_reg[ks][0] = v.x; qa_reg[ks][1] = v.y; qa_reg[ks][2] = v.z; qa_reg[ks][3] = v.w;
      }
    }
  };
  // the A fragment of S k-step ks
  auto qa = [&](int ks, uint32_t (&a)[4]) {
    if constexpr (kShared) {
      const uint4 v = ld_shared_v4(qfrag_addr + ks * 512);
      a[0] = v.x; a[1] = v.y; a[2] = v.z; a[3] = v.w;
    } else {
      a[0] = qa_reg[ks][0]; a[1] = qa_reg[ks][1]; a[2] = qa_reg[ks][2]; a[3] = qa_reg[ks][3];
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

  // Values-only cache: this lane's share of the key rebuild.  wk(ks, h): w_k
  // at dims (d + 2 tq, +1) for h = 0 and (d + 8 + 2 tq, +1) for h = 1, d the
  // k-step's first dim; freq(e): pair j = 16 w + 2 tq + (e & 1) + 8 (e >> 1).
  auto wk = [&](int ks, int h) -> uint32_t {
    if constexpr (kShared) return s.wk[(s_kstep_dim<kShared>(warp, ks) + 8 * h + 2 * tq) / 2];
    return 0u;
  };
  auto freq = [&](int e) -> FloatPair {
    if constexpr (kShared) return s.freq[16 * warp + 2 * tq + (e & 1) + 8 * (e >> 1)];
    return FloatPair{0.f, 0.f};
  };
  // byte offset of this lane's ldmatrix row in the tile of S k-step ks
  auto kstep_offset = [&](int ks) -> uint32_t {
    const int d = s_kstep_dim<kShared>(warp, ks);
    const int row = ((mi >> 1) << 3) + lr;
    return (d / kChunk) * kChunkBytes + swz(row, 2 * ((d % kChunk) / 16) + (mi & 1));
  };

  // the full-barrier wait of page i in stage st (a timeout is reported once and ends the waits)
  auto wait_page = [&](int i, int st) {
    if (ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(&s.full[st], (i / kNS) & 1));
      if (!ok && lane == 0) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
    }
  };

  // Values-only cache: NP (1 or 2) consecutive pages of one segment, with one
  // partial-S exchange and one softmax pass for all of them.  (The separate-
  // pool kernel runs its own one-page loop below.)
  auto page_group = [&](auto np_c, int i, int f, int it) {
    constexpr int NP = decltype(np_c)::value;
    constexpr int kEO = NP == 1 ? 2 : 1;  // accumulators per n-tile: even/odd k-steps, or one chain
    int pos0[NP], stage[NP];
    uint32_t vst[NP];
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      stage[j] = j == 0 ? i % kNS : (stage[0] + j == kNS ? 0 : stage[0] + j);
      pos0[j] = cur.pos0(t, f + j);
      vst[j] = smem_addr(s.v[stage[j]]);
    }

    // ---- partial S over this warp's dims, per page: two n-tiles of 8 positions ----
    //      The K fragments are read kAhead k-steps before their MMAs.
    float sa[NP][kEO][2][4];
#pragma unroll
    for (int j = 0; j < NP; ++j)
#pragma unroll
      for (int eo = 0; eo < kEO; ++eo)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sa[j][eo][nt][e] = 0.f;
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      wait_page(i + j, stage[j]);
      auto acc_of = [&](int ks, int nt) -> float (&)[4] { return sa[j][kEO == 2 ? (ks & 1) : 0][nt]; };
      if constexpr (kShared) {
        // K fragments rebuilt from the V page: k-steps 0 and 1 rotate together,
        // the rest are V * w_k.  Fragment register r holds position
        // pos0 + g + 8 (r >> 1) and dims (d + 8 (r & 1) + 2 tq, +1).
        uint32_t ka[4], kb[4];
        {
          uint32_t va[4], vb[4];
          ldmatrix_x4(vst[j] + kstep_offset(0), va[0], va[1], va[2], va[3]);
          ldmatrix_x4(vst[j] + kstep_offset(1), vb[0], vb[1], vb[2], vb[3]);
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const float2 a = bf16x2_to_float2(va[r]), b = bf16x2_to_float2(vb[r]);
            const float2 wa = bf16x2_to_float2(wk(0, r & 1)), wb = bf16x2_to_float2(wk(1, r & 1));
            const float a0 = a.x * wa.x, a1 = a.y * wa.y;  // exact
            const float b0 = b.x * wb.x, b1 = b.y * wb.y;
            const int pos = pos0[j] + g + 8 * (r >> 1), e = 2 * (r & 1);
            float c0, s0, c1, s1;
            rope_angle(kr->two_pi, freq(e), pos, c0, s0);
            rope_angle(kr->two_pi, freq(e + 1), pos, c1, s1);
            ka[r] = pack_bf16x2(fmaf(a0, c0, -b0 * s0), fmaf(a1, c1, -b1 * s1));
            kb[r] = pack_bf16x2(fmaf(b0, c0, a0 * s0), fmaf(b1, c1, a1 * s1));
          }
        }
        {
          uint32_t a[4];
          qa(0, a);
          mma_bf16_16816(acc_of(0, 0), a, ka[0], ka[1]);
          mma_bf16_16816(acc_of(0, 1), a, ka[2], ka[3]);
          qa(1, a);
          mma_bf16_16816(acc_of(1, 0), a, kb[0], kb[1]);
          mma_bf16_16816(acc_of(1, 1), a, kb[2], kb[3]);
        }
        auto k_frag = [&](int ks, uint32_t (&b)[4]) {
          ldmatrix_x4(vst[j] + kstep_offset(ks), b[0], b[1], b[2], b[3]);
#pragma unroll
          for (int r = 0; r < 4; ++r) b[r] = bf16x2_mul(b[r], wk(ks, r & 1));
        };
        constexpr int kAh = 1;  // one k-step ahead: 2.4 % faster than two on long contexts
        uint32_t kf[kAh + 1][4];
#pragma unroll
        for (int ks = 2; ks < 2 + kAh; ++ks) k_frag(ks, kf[ks % (kAh + 1)]);
#pragma unroll
        for (int ks = 2; ks < 8; ++ks) {
          if (ks + kAh < 8) k_frag(ks + kAh, kf[(ks + kAh) % (kAh + 1)]);
          const uint32_t (&b)[4] = kf[ks % (kAh + 1)];
          uint32_t a[4];
          qa(ks, a);
          mma_bf16_16816(acc_of(ks, 0), a, b[0], b[1]);
          mma_bf16_16816(acc_of(ks, 1), a, b[2], b[3]);
        }
      }
    }

    // ---- sum the four partials in a fixed order ----
    const int buf = it & 1;
#pragma unroll
    for (int j = 0; j < NP; ++j)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        float4 v = make_float4(sa[j][0][nt][0], sa[j][0][nt][1], sa[j][0][nt][2], sa[j][0][nt][3]);
        if constexpr (kEO == 2) {
          v.x += sa[j][1][nt][0]; v.y += sa[j][1][nt][1]; v.z += sa[j][1][nt][2]; v.w += sa[j][1][nt][3];
        }
        s.xs[buf][warp][2 * j + nt][lane] = v;
      }
    named_barrier_sync(1, kConsumerWarps * 32);
    float sc[NP][2][4];
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      float4 a0 = s.xs[buf][0][2 * j][lane], a1 = s.xs[buf][0][2 * j + 1][lane];
#pragma unroll
      for (int w = 1; w < kConsumerWarps; ++w) {
        const float4 c0 = s.xs[buf][w][2 * j][lane], c1 = s.xs[buf][w][2 * j + 1][lane];
        a0.x += c0.x; a0.y += c0.y; a0.z += c0.z; a0.w += c0.w;
        a1.x += c1.x; a1.y += c1.y; a1.z += c1.z; a1.w += c1.w;
      }
      sc[j][0][0] = a0.x; sc[j][0][1] = a0.y; sc[j][0][2] = a0.z; sc[j][0][3] = a0.w;
      sc[j][1][0] = a1.x; sc[j][1][1] = a1.y; sc[j][1][2] = a1.z; sc[j][1][3] = a1.w;
    }

    // ---- masked online softmax (log2 units) ----
    // sc[j][nt][e]: head g + 8*(e>>1), position pos0[j] + 8*nt + 2*tq + (e&1).
    // Positions outside [lo, L) get -inf (pages inside the range skip the
    // test); the factor log2(e) is applied inside the exponent.
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      if (pos0[j] < cur.lo || pos0[j] + kPage > cur.L) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int pos = pos0[j] + 8 * nt + 2 * tq + (e & 1);
            if (pos < cur.lo || pos >= cur.L) sc[j][nt][e] = -INFINITY;
          }
      }
    }
    float mx[2];
    mx[0] = fmaxf(fmaxf(sc[0][0][0], sc[0][0][1]), fmaxf(sc[0][1][0], sc[0][1][1]));
    mx[1] = fmaxf(fmaxf(sc[0][0][2], sc[0][0][3]), fmaxf(sc[0][1][2], sc[0][1][3]));
#pragma unroll
    for (int j = 1; j < NP; ++j) {
      mx[0] = fmaxf(mx[0], fmaxf(fmaxf(sc[j][0][0], sc[j][0][1]), fmaxf(sc[j][1][0], sc[j][1][1])));
      mx[1] = fmaxf(mx[1], fmaxf(fmaxf(sc[j][0][2], sc[j][0][3]), fmaxf(sc[j][1][2], sc[j][1][3])));
    }
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
    float pr[NP][2][4];
#pragma unroll
    for (int j = 0; j < NP; ++j)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) pr[j][nt][e] = ex2_approx(fmaf(sc[j][nt][e], kLog2e, -m_use[e >> 1]));
    float ls[2] = {(pr[0][0][0] + pr[0][0][1]) + (pr[0][1][0] + pr[0][1][1]),
                   (pr[0][0][2] + pr[0][0][3]) + (pr[0][1][2] + pr[0][1][3])};
#pragma unroll
    for (int j = 1; j < NP; ++j) {
      ls[0] += (pr[j][0][0] + pr[j][0][1]) + (pr[j][1][0] + pr[j][1][1]);
      ls[1] += (pr[j][0][2] + pr[j][0][3]) + (pr[j][1][2] + pr[j][1][3]);
    }
    l[0] = l[0] * scale[0] + ls[0];
    l[1] = l[1] * scale[1] + ls[1];
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

#pragma unroll
    for (int j = 0; j < NP; ++j) {
      // P of page j as the A fragment of one k16 step (k = its 16 positions)
      const uint32_t pa[4] = {pack_bf16x2(pr[j][0][0], pr[j][0][1]), pack_bf16x2(pr[j][0][2], pr[j][0][3]),
                              pack_bf16x2(pr[j][1][0], pr[j][1][1]), pack_bf16x2(pr[j][1][2], pr[j][1][3])};

      // ---- zero V rows outside [lo, L) in this warp's two chunks ----
      //      (after the exchange barrier: with a values-only cache every warp
      //      has read these chunks for its keys by then)
      if (pos0[j] < cur.lo || pos0[j] + kPage > cur.L) {
#pragma unroll 1
        for (int rr = 0; rr < kPage; ++rr) {
          const int pos = pos0[j] + rr;
          if ((pos < cur.lo || pos >= cur.L) && lane < 16) {
            const int ch = 2 * warp + (lane >> 3);
            st_shared_v4(vst[j] + ch * kChunkBytes + rr * 128 + (lane & 7) * 16, make_uint4(0, 0, 0, 0));
          }
        }
        fence_proxy_async_smem();  // before TMA rewrites this stage
        __syncwarp();
      }

      // ---- O += P V over this warp's 128 dims ----
      auto v_frag = [&](int np, uint32_t (&b)[4]) {
        const int ch = 2 * warp + (np >> 2);
        const int row = ((mi & 1) << 3) + lr;
        const int unit = 2 * (np & 3) + (mi >> 1);
        ldmatrix_x4_trans(vst[j] + ch * kChunkBytes + swz(row, unit), b[0], b[1], b[2], b[3]);
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
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.empty[stage[j]]);
    }

    if (f + NP == cur.seg_end) {
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
  };

  if constexpr (kShared) {
    int it = 0;  // page groups so far (parity of the exchange buffer)
    for (int i = 0; i < n_pages; ++it) {
      const int f = sp.begin + i;
      if (f >= t.prefix[cur.b + 1]) {
        cur.advance(p, t, sp, f);
        load_q();
        prefetch_next_q();
      }
      if (i + 1 < n_pages && f + 1 < cur.seg_end) {  // two pages of this segment
        page_group(std::integral_constant<int, 2>{}, i, f, it);
        i += 2;
      } else {
        page_group(std::integral_constant<int, 1>{}, i, f, it);
        i += 1;
      }
    }
  } else {
    for (int i = 0; i < n_pages; ++i) {
      const int f = sp.begin + i;
      if (f >= t.prefix[cur.b + 1]) {
        cur.advance(p, t, sp, f);
        load_q();
        prefetch_next_q();
      }
      const int stage = i % kNS;
      const int pos0 = cur.pos0(t, f);
      if (ok) {
        ok = __all_sync(0xffffffffu, mbar_wait(&s.full[stage], (i / kNS) & 1));
        if (!ok && lane == 0) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
      }
      const uint32_t vst = smem_addr(s.v[stage]);
      const uint32_t kst = smem_addr(s.k[stage]);

      // ---- partial S over this warp's dims: two n-tiles of 8 positions; even
      //      and odd k-steps accumulate separately (two chains of 4 MMAs) ----
      //      The K fragments are read kAhead k-steps before their MMAs.
      float se[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      float so[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
      auto k_frag = [&](int ks, uint32_t (&b)[4]) {
        ldmatrix_x4(kst + kstep_offset(ks), b[0], b[1], b[2], b[3]);
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
        mma_bf16_16816(s0, qa_reg[ks], b[0], b[1]);
        mma_bf16_16816(s1, qa_reg[ks], b[2], b[3]);
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
}

__global__ void __launch_bounds__(kThreads)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ DecodeParams p) {
  decode_body<false>(&tm_k, &tm_v, p, nullptr);
}

// Values-only cache: p.v_pool holds V; keys are rebuilt as rope(V * w_k).
__global__ void __launch_bounds__(kThreads, kBlocksPerSm)
    decode_kernel_shared(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ DecodeParams p,
                         const __grid_constant__ KeyRebuild kr) {
  decode_body<true>(nullptr, &tm_v, p, &kr);
}

}  // namespace global
}  // namespace pda
