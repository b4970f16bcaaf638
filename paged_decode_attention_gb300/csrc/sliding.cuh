// sliding.cuh -- decode kernel for the Gemma-4-12B sliding-window layers
// (slidingDecodeGQA: 16 query heads over 8 KV heads, D = 256, G = 2,
// scale 1), on CUDA cores.
//
// Grid (grid_x, 8): column c serves KV head c (query heads 2c, 2c+1); block
// g of a column streams its span of the flattened visible pages (see the
// balanced schedule in common.cuh):
//   * warp 4 (producer) reads block-table entries and issues one 2-D TMA
//     tensor copy per page for K and one for V: a 16-row x 256-column box
//     (8 KB) of the pool viewed as [num_pages*16 rows, 8*256], so the
//     KV-head slice of a page lands dense in shared memory;
//   * warps 0..3 (consumers) each own 4 of the 16 rows of every page and run
//     their own online softmax over them; lane j holds dims 8j..8j+7 of q,
//     of the K/V rows and of the output accumulator (packed fp32x2 FMAs);
//   * when a sequence's pages in the span end, the four warps' (max, sum,
//     accumulator) are merged through shared memory and written as o (the
//     span holds the whole sequence) or as a partial.  A partial is merged by
//     the combine kernel or, when the host plan bounds the blocks that share
//     a sequence (p.merge_in_grid), by the last of those blocks to finish:
//     each writes its partial, counts itself in with an atomic add, and the
//     one that completes the count reads the others' partials back and
//     writes o.  No block waits for another.
// Masking selects, never multiplies: rows outside [lo, L) get logit -inf
// and their V row is skipped, so NaN in unused slots cannot leak.
#pragma once

#include "common.cuh"

namespace pda {
namespace sliding {

constexpr int kHq = ATTN_SLIDING_HQ;    // 16
constexpr int kHkv = ATTN_SLIDING_HKV;  // 8
constexpr int kD = ATTN_SLIDING_D;      // 256
constexpr int kG = kHq / kHkv;          // 2
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kRowsPerWarp = kPage / kConsumerWarps;  // 4
constexpr int kRowBytes = kD * 2;                      // 512
constexpr int kTileBytes = kPage * kRowBytes;          // 8 KB per K (or V) page-head
constexpr int kStages = 4;
constexpr int kBlocksPerSm = 3;
constexpr int kMinPages = 4;
constexpr int kWarmPages = 4;  // pages per block pulled into L2 before the wait

static_assert(kG == 2, "the lane mapping below assumes two query heads per KV head");

struct Smem {
  alignas(128) uint8_t k[kStages][kTileBytes];
  alignas(128) uint8_t v[kStages][kTileBytes];
  alignas(16) float merge_o[kConsumerWarps][kG][kD];
  float merge_m[kConsumerWarps][kG];
  float merge_l[kConsumerWarps][kG];
  int32_t merge_last;  // this block completed the arrivals of the sequence it closes
  int32_t merge_cnt[kConsumerWarps];  // non-empty sequences before it, per consumer warp
  SeqTable table;
  alignas(8) uint64_t full[kStages];
  alignas(8) uint64_t empty[kStages];
};

constexpr size_t kSmemBytes = sizeof(Smem) + 128;  // + alignment slack
static_assert(kBlocksPerSm * (kSmemBytes + 1024) <= 228 * 1024, "shared memory of the resident blocks");

// The merge of a cut sequence by the last of its blocks, run by the 128
// consumer threads right after each has written its share (head h, dims
// d0..d0+3) of this block's partial (M, Lsum, O) to the workspace.
//
// Every contributor fences its partial, then one thread adds 1 to the
// sequence's counter; the contributor that raises it to the number of
// contributors (blocks g0..g1 of this column) holds the last partial.  It
// fences again, reads every partial of the sequence (its own from
// registers) in block order g0..g1, so the result does not depend on which
// block came last, merges them as the combine kernel would
//     o = sum_g 2^{m_g - M} O_g / sum_g 2^{m_g - M} l_g,
// writes o and puts the counter back to 0 for the next call (no other block
// of this call touches it again).  Partials read back bypass L1.
__device__ __forceinline__ void merge_partials(const DecodeParams& p, const SeqTable& t, Smem& s, int b, int g,
                                               int c, int h, int d0, float M, float Lsum, float4 O) {
  const int tt = threadIdx.x;
  int cnt = 0;  // non-empty sequences before b among b' = tt, tt + 128
  for (int j = tt; j < b; j += kConsumerWarps * 32) cnt += t.prefix[j + 1] > t.prefix[j];
  cnt = __reduce_add_sync(0xffffffffu, cnt);
  if ((tt & 31) == 0) s.merge_cnt[tt >> 5] = cnt;
  int32_t* counter = p.counters + b * kHkv + c;
  __threadfence();
  named_barrier_sync(1, kConsumerWarps * 32);
  int g0, g1;
  seq_blocks(t, b, s.merge_cnt[0] + s.merge_cnt[1] + s.merge_cnt[2] + s.merge_cnt[3], g0, g1);
  if (tt == 0) {
    const int before_me = atomicAdd(counter, 1);
    s.merge_last = before_me == g1 - g0;
    // more arrivals than contributors: the counter did not start at zero (a
    // workspace whose head was not zeroed before its first use)
    if (before_me > g1 - g0 || before_me < 0) report(p.status, ATTN_DEV_INTERNAL);
  }
  named_barrier_sync(1, kConsumerWarps * 32);
  if (!s.merge_last) return;
  if (tt == 0) *counter = 0;  // every contributor of this call has arrived
  __threadfence();
  if ((static_cast<int64_t>(g1) + b + 1) * kHq > p.part_rows || g < g0 || g > g1) {
    if (tt == 0) report(p.status, ATTN_DEV_INTERNAL);  // cannot happen: partials beyond the workspace
    return;
  }
  const int hq = c * kG + h;
  float rm = -INFINITY, rl = 0.f;
  float4 ro = make_float4(0.f, 0.f, 0.f, 0.f);
  constexpr int kBatch = 4;  // partials whose loads are in flight together
  for (int gb = g0; gb <= g1; gb += kBatch) {
    float2 e[kBatch];
    float4 a[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int gg = gb + j;
      if (gg > g1) {
        e[j] = make_float2(-INFINITY, 0.f);
        a[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      } else if (gg == g) {
        e[j] = make_float2(M, Lsum);
        a[j] = O;
      } else {
        const size_t sl = (static_cast<size_t>(gg) + b) * kHq + hq;
        e[j] = __ldcg(p.part_ml + sl);
        a[j] = __ldcg(reinterpret_cast<const float4*>(p.part_o + sl * kD + d0));
      }
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      if (e[j].y > 0.f) {  // a partial without a visible position adds nothing
        const float mn = fmaxf(rm, e[j].x);
        const float fr = rm == -INFINITY ? 0.f : exp2f(rm - mn);
        const float fe = exp2f(e[j].x - mn);
        rl = rl * fr + e[j].y * fe;
        ro.x = ro.x * fr + a[j].x * fe;
        ro.y = ro.y * fr + a[j].y * fe;
        ro.z = ro.z * fr + a[j].z * fe;
        ro.w = ro.w * fr + a[j].w * fe;
        rm = mn;
      }
    }
  }
  const float inv = rl > 0.f ? 1.f / rl : 0.f;
  const size_t row = static_cast<size_t>(b) * kHq + hq;
  store_out4(p, row * kD + d0, make_float4(ro.x * inv, ro.y * inv, ro.z * inv, ro.w * inv));
}

__global__ void __launch_bounds__(kThreads)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));

  const int g = blockIdx.x;
  const int c = blockIdx.y;
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
  build_seq_table_hint(p, s.table, g);  // ends with __syncthreads
  if (warp == kConsumerWarps) {
    warm_first_pages(p, s.table, kWarmPages, [&](int32_t y) {
      tma_prefetch_2d(&tm_k, c * kD, y);
      tma_prefetch_2d(&tm_v, c * kD, y);
    });
  } else {
    warm_q(p, s.table, kHq * kD, c * kG * kD, kG * kD * 2, kConsumerWarps * 32);
  }
  wait_for_primary_grid();
  // The dependent kernel is let launch only once this block's streaming is
  // done (below).  With no combine kernel after this one, the dependent is
  // the next call's kernel; a cache append launched at once would sit on
  // the SMs waiting for this grid (a step of appends and decodes measured
  // 12 % slower that way, back-to-back decodes 0.5 % faster).
  // The producer reads its first block-table entries while warp 0 confirms
  // the table; it reads them again if the table had to be rebuilt.
  int first = warp == kConsumerWarps ? page_entry(p, s.table, s.table.span, lane, false) : 0;
  confirm_seq_table(p, s.table, g);  // ends with __syncthreads
  const SeqTable& t = s.table;
  const Span sp = t.span;
  const int n_pages = sp.end - sp.begin;
  if (p.merge_in_grid && g == 0 && warp < kConsumerWarps) {
    // No combine kernel runs: block 0 of each column writes the empty sum of
    // the sequences with no visible position (L = 0).
    for (int b = 0; b < p.batch; ++b) {
      if (t.prefix[b + 1] != t.prefix[b]) continue;
      const size_t row = static_cast<size_t>(b) * kHq + c * kG + (threadIdx.x >> 6);
      store_out4(p, row * kD + (threadIdx.x & 63) * 4, make_float4(0.f, 0.f, 0.f, 0.f));
    }
  }
  if (n_pages <= 0) return;

  if (warp == kConsumerWarps) {
    // ---------------- producer ----------------
    const uint64_t policy = l2_policy_evict_first();
    const int x = c * kD;
    if (t.rebuilt) first = page_entry(p, t, sp, lane, true);
    produce_pages<kStages, 2 * kTileBytes>(p, t, sp, s.full, s.empty, first, [&](int stage, int32_t y) {
      tma_load_2d_hint(s.k[stage], &tm_k, x, y, &s.full[stage], policy);
      tma_load_2d_hint(s.v[stage], &tm_v, x, y, &s.full[stage], policy);
    });
    allow_dependent_launch();
    return;
  }

  // ---------------- consumers ----------------
  const int hq0 = c * kG;
  // after the reduce-scatter, lane holds the logit of (row r_mine, head h_mine)
  const int j_mine = (lane >> 2) & 7;
  const int r_mine = j_mine >> 1;
  const int h_mine = j_mine & 1;

  PageCursor cur;
  cur.start(p, t, sp);
  // q of the current sequence as fp32 pairs; qn holds the raw bf16 words of
  // the next sequence of the span, loaded one segment ahead
  float2 qf[kG][4];
  uint4 qn[kG];
  auto load_q_raw = [&](int b) {
#pragma unroll
    for (int h = 0; h < kG; ++h)
      qn[h] = ld_global_nc_v4(p.q + (static_cast<size_t>(b) * kHq + hq0 + h) * kD + 8 * lane);
  };
  auto take_q = [&]() {
#pragma unroll
    for (int h = 0; h < kG; ++h) {
      qf[h][0] = bf16x2_to_float2(qn[h].x);
      qf[h][1] = bf16x2_to_float2(qn[h].y);
      qf[h][2] = bf16x2_to_float2(qn[h].z);
      qf[h][3] = bf16x2_to_float2(qn[h].w);
    }
  };
  load_q_raw(cur.b);
  take_q();
  int nb = next_seq_in_span(p, t, sp, cur.b);
  if (nb >= 0) load_q_raw(nb);

  float m[kG], l[kG];  // running max (log2 units) and sum, identical in every lane
  float2 acc[kG][4];
  auto reset = [&]() {
#pragma unroll
    for (int h = 0; h < kG; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[h][k] = make_float2(0.f, 0.f);
    }
  };
  reset();
  bool ok = true;

  for (int i = 0; i < n_pages; ++i) {
    const int f = sp.begin + i;
    if (f >= t.prefix[cur.b + 1]) {
      cur.advance(p, t, sp, f);  // lands on nb, whose q is already in qn
      take_q();
      nb = next_seq_in_span(p, t, sp, cur.b);
      if (nb >= 0) load_q_raw(nb);
    }
    const int stage = i % kStages;
    if (ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(&s.full[stage], (i / kStages) & 1));
      if (!ok && lane == 0) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
    }
    const int pos0 = cur.pos0(t, f) + warp * kRowsPerWarp;
    const uint32_t kbase = smem_addr(s.k[stage]) + warp * kRowsPerWarp * kRowBytes + lane * 16;
    const uint32_t vbase = smem_addr(s.v[stage]) + warp * kRowsPerWarp * kRowBytes + lane * 16;

    // partial logits over this lane's 8 dims: part[row*2 + head]
    float part[8];
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
      const uint4 kw = ld_shared_v4(kbase + rr * kRowBytes);
      const float2 k0 = bf16x2_to_float2(kw.x), k1 = bf16x2_to_float2(kw.y);
      const float2 k2 = bf16x2_to_float2(kw.z), k3 = bf16x2_to_float2(kw.w);
#pragma unroll
      for (int h = 0; h < kG; ++h) {
        float2 u = __fmul2_rn(qf[h][0], k0);
        u = __ffma2_rn(qf[h][1], k1, u);
        u = __ffma2_rn(qf[h][2], k2, u);
        u = __ffma2_rn(qf[h][3], k3, u);
        part[rr * 2 + h] = u.x + u.y;
      }
    }
    // reduce-scatter over 32 lanes: 4 + 2 + 1 exchanges, then an all-reduce
    // over the remaining 4-lane group
    {
      const bool up = lane & 16;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float send = up ? part[k] : part[k + 4];
        const float keep = up ? part[k + 4] : part[k];
        part[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
      }
    }
    {
      const bool up = lane & 8;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float send = up ? part[k] : part[k + 2];
        const float keep = up ? part[k + 2] : part[k];
        part[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
      }
    }
    {
      const bool up = lane & 4;
      const float send = up ? part[0] : part[1];
      const float keep = up ? part[1] : part[0];
      part[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    part[0] += __shfl_xor_sync(0xffffffffu, part[0], 2);
    part[0] += __shfl_xor_sync(0xffffffffu, part[0], 1);

    // masked online softmax, in log2 units (exp(x) = exp2(x * log2 e))
    const int pos_mine = pos0 + r_mine;
    const bool vis_mine = pos_mine >= cur.lo && pos_mine < cur.L;
    const float s2 = vis_mine ? part[0] * kLog2e : -INFINITY;
    float pm = fmaxf(s2, __shfl_xor_sync(0xffffffffu, s2, 8));
    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));  // max over the 4 rows of head h_mine
    const float pm_other = __shfl_xor_sync(0xffffffffu, pm, 4);
    const float page_max[kG] = {h_mine ? pm_other : pm, h_mine ? pm : pm_other};
    float m_use[kG], scale[kG];
#pragma unroll
    for (int h = 0; h < kG; ++h) {
      const float m_new = fmaxf(m[h], page_max[h]);
      m_use[h] = m_new == -INFINITY ? 0.f : m_new;
      scale[h] = exp2f(m[h] - m_use[h]);
      m[h] = m_new;
    }
    const float pv = exp2f(s2 - (h_mine ? m_use[1] : m_use[0]));
    float ps = pv + __shfl_xor_sync(0xffffffffu, pv, 8);
    ps += __shfl_xor_sync(0xffffffffu, ps, 16);
    const float ps_other = __shfl_xor_sync(0xffffffffu, ps, 4);
    l[0] = l[0] * scale[0] + (h_mine ? ps_other : ps);
    l[1] = l[1] * scale[1] + (h_mine ? ps : ps_other);

    float pj[8];  // probability of (row, head) j = row*2 + head; lanes 4j..4j+3 hold it
#pragma unroll
    for (int j = 0; j < 8; ++j) pj[j] = __shfl_sync(0xffffffffu, pv, 4 * j);

    if (scale[0] != 1.f || scale[1] != 1.f) {  // same in every lane; multiplying by 1 is exact
#pragma unroll
      for (int h = 0; h < kG; ++h) {
        const float2 sc = make_float2(scale[h], scale[h]);
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[h][k] = __fmul2_rn(acc[h][k], sc);
      }
    }
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
      const int pos = pos0 + rr;
      if (pos >= cur.lo && pos < cur.L) {  // warp-uniform
        const uint4 vw = ld_shared_v4(vbase + rr * kRowBytes);
        const float2 v0 = bf16x2_to_float2(vw.x), v1 = bf16x2_to_float2(vw.y);
        const float2 v2 = bf16x2_to_float2(vw.z), v3 = bf16x2_to_float2(vw.w);
#pragma unroll
        for (int h = 0; h < kG; ++h) {
          const float2 pp = make_float2(pj[rr * 2 + h], pj[rr * 2 + h]);
          acc[h][0] = __ffma2_rn(pp, v0, acc[h][0]);
          acc[h][1] = __ffma2_rn(pp, v1, acc[h][1]);
          acc[h][2] = __ffma2_rn(pp, v2, acc[h][2]);
          acc[h][3] = __ffma2_rn(pp, v3, acc[h][3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.empty[stage]);

    if (f + 1 == cur.seg_end) {
      // ---------------- finish this sequence's segment ----------------
#pragma unroll
      for (int h = 0; h < kG; ++h) {
        float4* dst = reinterpret_cast<float4*>(&s.merge_o[warp][h][8 * lane]);
        dst[0] = make_float4(acc[h][0].x, acc[h][0].y, acc[h][1].x, acc[h][1].y);
        dst[1] = make_float4(acc[h][2].x, acc[h][2].y, acc[h][3].x, acc[h][3].y);
      }
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < kG; ++h) {
          s.merge_m[warp][h] = m[h];
          s.merge_l[warp][h] = l[h];
        }
      }
      named_barrier_sync(1, kConsumerWarps * 32);
      const int tt = threadIdx.x;  // 0..127: 2 heads x 64 groups of 4 dims
      const int h = tt >> 6;
      const int d0 = (tt & 63) * 4;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, s.merge_m[w][h]);
      float Lsum = 0.f;
      float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float fw = exp2f(s.merge_m[w][h] - M);
          Lsum += fw * s.merge_l[w][h];
          const float4 a = *reinterpret_cast<const float4*>(&s.merge_o[w][h][d0]);
          O.x += fw * a.x;
          O.y += fw * a.y;
          O.z += fw * a.z;
          O.w += fw * a.w;
        }
      }
      if (cur.whole(t, sp)) {
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
        const size_t row = static_cast<size_t>(cur.b) * kHq + hq0 + h;
        store_out4(p, row * kD + d0, make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv));
      } else if ((static_cast<int64_t>(g) + cur.b + 1) * kHq > p.part_rows) {
        if (tt == 0) report(p.status, ATTN_DEV_INTERNAL);  // cannot happen: slot beyond the workspace
      } else {
        const size_t slot = (static_cast<size_t>(g) + cur.b) * kHq + hq0 + h;
        *reinterpret_cast<float4*>(p.part_o + slot * kD + d0) = O;
        if (d0 == 0) p.part_ml[slot] = make_float2(M, Lsum);
        if (p.merge_in_grid) merge_partials(p, t, s, cur.b, g, c, h, d0, M, Lsum, O);
      }
      named_barrier_sync(1, kConsumerWarps * 32);  // merge buffers free again
      reset();
    }
  }
  allow_dependent_launch();
}

}  // namespace sliding
}  // namespace pda
