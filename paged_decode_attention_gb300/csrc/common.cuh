// common.cuh -- launch parameters, the balanced page schedule and the TMA
// page producer shared by the decode kernels.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "attn_decode.h"
#include "ptx.cuh"

namespace pda {

constexpr int kPage = ATTN_PAGE_SIZE;  // token rows per cache page
constexpr int kMaxBatch = ATTN_MAX_BATCH;
constexpr int kMaxSplits = 1024;       // blocks per KV head the host plan may launch
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeParams {
  const __nv_bfloat16* q;      // [batch, Hq, D]
  const __nv_bfloat16* k_pool; // [num_pages, 16, Hkv, D] (read through the tensor maps; raw for L2 prefetches)
  const __nv_bfloat16* v_pool;
  const int32_t* block_table;  // [batch, max_blocks]
  const int32_t* seq_lens;     // [batch]
  void* o;                     // [batch, Hq, D], bf16 or fp32
  float* part_o;               // [grid_x + batch, Hq, D]: partial outputs, slot = block + sequence
  float2* part_ml;             // [grid_x + batch, Hq]: (running max in log2 units, sum)
  int32_t* status;             // optional ATTN_DEV_* word
  int64_t num_pages;
  int32_t batch;
  int32_t max_blocks;
  int32_t window;              // > 0 sliding rule, <= 0 none
  int32_t grid_x;              // blocks sharing the pages of one KV head
  int32_t min_pages;           // smallest span a block is given
  int32_t out_f32;
  int64_t part_rows;           // rows [Hq-row granularity] the workspace holds: (grid_x + batch) * Hq
  int32_t* counters;           // [batch][Hkv] arrivals per cut sequence (zero between calls)
  int32_t merge_in_grid;       // cut sequences are merged by their last block (no combine kernel)
};

// ---------------------------------------------------------------------------
// Balanced schedule.
//
// Sequence b's visible positions are [lo_b, L_b) with the query at
// p = L_b - 1 (Attention.lean decodeGQA) and, for a window w, lo_b =
// max(0, L_b - w) (Attention.lean slidingGQA: p - w < l <= p).  They occupy
// logical pages lo_b/16 .. (L_b-1)/16.  Concatenating every sequence's
// visible pages gives N pages.  Each sequence a block starts also costs it a
// fixed amount of work (loading its q, closing its segment), so spans are cut
// on a weighted list in which every non-empty sequence is preceded by
// kSeqWeight virtual pages.  With W weighted pages in all, block g of grid_x
// takes the weighted range [g*per, min((g+1)*per, W)), per = max(min_pages,
// ceil(W / grid_x)), mapped back to a contiguous range of real pages (a
// virtual page maps to the first page of its sequence), so every block gets
// the same amount of work whatever the mix of lengths.  A sequence that lies
// inside one span is finished by that block; one that straddles spans leaves
// a partial result in slot (block + b), an injective numbering because spans
// and sequences are both in order; the combine kernel, or the last of the
// sequence's blocks (sliding kernel, merge in the grid), merges them.
// ---------------------------------------------------------------------------
constexpr int kSeqWeight = 1;  // virtual pages charged per sequence start

struct Span {
  int begin, end;  // flattened real pages of this block
};

struct SeqTable {
  int32_t prefix[kMaxBatch + 1];  // prefix[b] = visible pages of sequences < b
  int32_t len[kMaxBatch];         // L_b, clamped (clamp_len)
  int32_t per;                    // weighted pages per block
  Span span;                      // this block's pages
  int32_t rebuilt;                // confirm_seq_table found seq_lens changed since the hint pass
};

__device__ __forceinline__ int first_visible(int L, int window) {
  return (window > 0 && L > window) ? L - window : 0;
}

__device__ __forceinline__ int visible_pages(int L, int window) {
  return L > 0 ? (L - 1) / kPage - first_visible(L, window) / kPage + 1 : 0;
}

// L_b clamped to [0, min(max_blocks*16, ATTN_MAX_SEQ_LEN)]: the block table
// holds no more positions, and the bound keeps every page count and prefix
// sum well inside int32.  A length outside is reported once per block.
__device__ __forceinline__ int clamp_len(const DecodeParams& p, int L, bool report_it) {
  const int cap = p.max_blocks < ATTN_MAX_SEQ_LEN / kPage ? p.max_blocks * kPage : ATTN_MAX_SEQ_LEN;
  if (L < 0 || L > cap) {
    if (report_it) report(p.status, ATTN_DEV_BAD_SEQ_LEN);
    return L < 0 ? 0 : cap;
  }
  return L;
}

__device__ __forceinline__ int span_pages(int total, int grid_x, int min_pages) {
  const int per = (total + grid_x - 1) / grid_x;
  return per > min_pages ? per : min_pages;
}

// Fills the table and block g's span; run by warp 0 alone.  kHint: the pass
// that runs before griddepcontrol.wait, whose results only aim prefetches.
// Its seq_lens reads go through ld.global.cg, so no line that might still
// change is kept in L1, and it reports nothing.
template <bool kHint>
__device__ __forceinline__ void scan_seq_lens(const DecodeParams& p, SeqTable& t, int g) {
  const int lane = threadIdx.x;
  {
    // pass 1: lengths, prefix sums of visible pages, non-empty sequences
    int carry = 0, nonempty = 0;
    if (lane == 0) t.prefix[0] = 0;
    for (int b0 = 0; b0 < p.batch; b0 += 32) {
      const int b = b0 + lane;
      const int L = b < p.batch ? clamp_len(p, kHint ? __ldcg(p.seq_lens + b) : p.seq_lens[b], !kHint) : 0;
      int v = visible_pages(L, p.window);
      nonempty += __popc(__ballot_sync(0xffffffffu, v > 0));
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      if (b < p.batch) {
        t.len[b] = L;
        t.prefix[b + 1] = carry + v;
      }
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    __syncwarp();
    // block g's weighted range [w0, w1) and the real pages it maps to
    const int total = carry + kSeqWeight * nonempty;
    const int per = span_pages(total, p.grid_x, p.min_pages);
    const long long u0 = static_cast<long long>(g) * per;
    const int w0 = u0 < total ? static_cast<int>(u0) : total;
    const int w1 = w0 + per < total ? w0 + per : total;
    // pass 2: weighted prefix wprefix[b] = prefix[b] + kSeqWeight * (non-empty
    // sequences before b); for u < total the owner of weighted position u is
    // the largest b with wprefix[b] <= u (on a run of equal values, the
    // non-empty sequence that ends it).
    int own0 = 0, wp0 = 0, own1 = 0, wp1 = 0, before = 0;
    const unsigned lt = (1u << lane) - 1u;
    for (int b0 = 0; b0 < p.batch; b0 += 32) {
      const int b = b0 + lane;
      const bool in = b < p.batch;
      const unsigned ne = __ballot_sync(0xffffffffu, in && t.len[b] > 0);
      const int wp = in ? t.prefix[b] + kSeqWeight * (before + __popc(ne & lt)) : 0;
      const unsigned c0 = __ballot_sync(0xffffffffu, in && wp <= w0);
      const unsigned c1 = __ballot_sync(0xffffffffu, in && wp <= w1);
      if (c0) {
        const int l = 31 - __clz(c0);
        own0 = b0 + l;
        wp0 = __shfl_sync(0xffffffffu, wp, l);
      }
      if (c1) {
        const int l = 31 - __clz(c1);
        own1 = b0 + l;
        wp1 = __shfl_sync(0xffffffffu, wp, l);
      }
      before += __popc(ne);
    }
    if (lane == 0) {
      t.per = per;
      const int o0 = w0 - wp0 - kSeqWeight, o1 = w1 - wp1 - kSeqWeight;
      t.span.begin = w0 >= total ? carry : t.prefix[own0] + (o0 > 0 ? o0 : 0);
      t.span.end = w1 >= total ? carry : t.prefix[own1] + (o1 > 0 ? o1 : 0);
    }
  }
  __syncwarp();
}

// Before griddepcontrol.wait: the table from hint reads.  Called by every
// thread of the block; ends with __syncthreads.
__device__ __forceinline__ void build_seq_table_hint(const DecodeParams& p, SeqTable& t, int g) {
  if (threadIdx.x < 32) scan_seq_lens<true>(p, t, g);
  __syncthreads();
}

// After griddepcontrol.wait: re-reads seq_lens and rebuilds the table only if
// a length differs from the hint pass (t.rebuilt tells the producer), so in
// the usual case the schedule costs one read here.  Called by every thread of
// the block; ends with a __syncthreads that also publishes anything written
// before it.  From here on the table is exact.
__device__ __forceinline__ void confirm_seq_table(const DecodeParams& p, SeqTable& t, int g) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    bool differ = false;
    for (int b0 = 0; b0 < p.batch; b0 += 32) {
      const int b = b0 + lane;
      const int L = b < p.batch ? clamp_len(p, p.seq_lens[b], true) : 0;
      differ |= __any_sync(0xffffffffu, b < p.batch && L != t.len[b]);
    }
    __syncwarp();
    if (differ) scan_seq_lens<false>(p, t, g);
    if (lane == 0) t.rebuilt = differ;
  }
  __syncthreads();
}

// The sequence holding flattened page f: the largest b < batch with
// prefix[b] <= f (on a run of equal values, the non-empty sequence that ends it).
__device__ __forceinline__ int seq_of(const SeqTable& t, int batch, int f) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (t.prefix[mid] <= f) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Run by one warp before griddepcontrol.wait, on a table built with kHint:
// lane i looks up page i of the span (i < n) and calls warm(y) with its row
// coordinate in the pools, to pull it into L2 while the previous kernel in
// the stream finishes.  Anything read here may be stale, which costs at most
// a useless prefetch: every index is range-checked, the block-table read
// bypasses L1, and nothing is written.
template <typename Warm>
__device__ __forceinline__ void warm_first_pages(const DecodeParams& p, const SeqTable& t, int n, Warm warm) {
  const int lane = threadIdx.x & 31;
  const int f = t.span.begin + lane;
  if (lane >= n || f >= t.span.end) return;
  const int b = seq_of(t, p.batch, f);
  const int lp = first_visible(t.len[b], p.window) / kPage + (f - t.prefix[b]);
  if (lp < 0 || lp >= p.max_blocks) return;
  const int phys = __ldcg(p.block_table + static_cast<int64_t>(b) * p.max_blocks + lp);
  if (phys >= 0 && static_cast<int64_t>(phys) < p.num_pages) warm(phys * kPage);
}

// Before griddepcontrol.wait, by threads [0, n): pull into L2 the `bytes` of q
// (from element `offset` of its sequence's [Hq, D] block) that the
// consumers load first: the span's first sequence, as the hint table has it.
__device__ __forceinline__ void warm_q(const DecodeParams& p, const SeqTable& t, int hq_d, int offset, int bytes,
                                       int n) {
  if (t.span.end <= t.span.begin) return;
  const int b = seq_of(t, p.batch, t.span.begin);
  const uint8_t* base = reinterpret_cast<const uint8_t*>(p.q + static_cast<size_t>(b) * hq_d + offset);
  const int i = threadIdx.x;  // one 128-byte line each
  if (i < n && i * 128 < bytes) prefetch_l2(base + i * 128);
}

// ---------------------------------------------------------------------------
// Output stores
// ---------------------------------------------------------------------------
__device__ __forceinline__ void store_out4(const DecodeParams& p, size_t idx, float4 v) {
  if (p.out_f32) {
    *reinterpret_cast<float4*>(static_cast<float*>(p.o) + idx) = v;
  } else {
    uint2 w;
    w.x = pack_bf16x2(v.x, v.y);
    w.y = pack_bf16x2(v.z, v.w);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.o) + idx) = w;
  }
}

__device__ __forceinline__ void store_out2(const DecodeParams& p, size_t idx, float a, float b) {
  if (p.out_f32) {
    *reinterpret_cast<float2*>(static_cast<float*>(p.o) + idx) = make_float2(a, b);
  } else {
    *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(p.o) + idx) = pack_bf16x2(a, b);
  }
}

// ---------------------------------------------------------------------------
// Producer side of the page pipeline, run by one whole warp.  Walks the
// block's span of flattened pages, reads their block-table entries 32 at a
// time (one entry per lane, fetched a batch ahead), and has lane 0 issue the
// TMA copies `issue(stage, y)` for page row coordinate y.  A page id outside
// [0, num_pages) is replaced by a fully out-of-range coordinate, which the
// copy engine fills with zeros, and ATTN_DEV_BAD_PAGE is raised.  Before it
// returns, the warp waits (bounded) until every copy it issued has landed,
// so no copy is in flight when the block retires.
// ---------------------------------------------------------------------------
// Block-table entry of page i of span sp (0 past its end).  A logical page
// outside the table cannot come from a consistent schedule: it gives -1 and,
// with report_it, ATTN_DEV_INTERNAL.  The producer also calls it while the
// table may still be rebuilt (report_it false, result discarded then), so
// every index is range-checked whatever the table holds.
__device__ __forceinline__ int page_entry(const DecodeParams& p, const SeqTable& t, const Span& sp, int i,
                                          bool report_it) {
  if (i < 0 || i >= sp.end - sp.begin) return 0;
  const int f = sp.begin + i;
  const int b = seq_of(t, p.batch, f);
  const int lp = first_visible(t.len[b], p.window) / kPage + (f - t.prefix[b]);
  if (lp < 0 || lp >= p.max_blocks) {
    if (report_it) report(p.status, ATTN_DEV_INTERNAL);
    return -1;
  }
  return p.block_table[static_cast<int64_t>(b) * p.max_blocks + lp];
}

// first: this lane's page_entry(sp, lane), read ahead by the caller.
template <int kStages, int kTxBytes, typename Issue>
__device__ __forceinline__ void produce_pages(const DecodeParams& p, const SeqTable& t, const Span& sp,
                                              uint64_t* full, uint64_t* empty, int first, Issue issue) {
  const int lane = threadIdx.x & 31;
  const int n_pages = sp.end - sp.begin;
  auto entry = [&](int i) -> int { return page_entry(p, t, sp, i, true); };
  int nxt = first;
  int cur = 0;
  int issued = 0;
  bool ok = true;
  for (int i = 0; i < n_pages; ++i) {
    if ((i & 31) == 0) {
      cur = nxt;
      nxt = entry(i + 32 + lane);
    }
    const int phys = __shfl_sync(0xffffffffu, cur, i & 31);
    const int stage = i % kStages;
    if (i >= kStages) {
      const int w = lane == 0 ? static_cast<int>(mbar_wait(&empty[stage], ((i / kStages) - 1) & 1)) : 0;
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
        y = -kPage;
      } else {
        y = phys * kPage;
      }
      mbar_arrive_expect_tx(&full[stage], kTxBytes);
      issue(stage, y);
    }
    ++issued;
    __syncwarp();
  }
  if (lane == 0) {
    // the last phase issued on each stage must have completed
    for (int st = 0; st < kStages && st < issued; ++st) {
      const int uses = (issued - 1 - st) / kStages + 1;
      if (!mbar_wait(&full[st], (uses - 1) & 1)) report(p.status, ATTN_DEV_WAIT_TIMEOUT);
    }
  }
}

// Consumer-side walk over the span: which sequence the current page belongs
// to, its first position, and whether it closes a segment (the last page of
// its sequence inside this span).
struct PageCursor {
  int b;        // current sequence
  int L, lo;    // its visible positions [lo, L)
  int seg_end;  // flattened index one past its last page in this span

  __device__ __forceinline__ void start(const DecodeParams& p, const SeqTable& t, const Span& sp) {
    b = seq_of(t, p.batch, sp.begin);
    load(p, t, sp);
  }
  __device__ __forceinline__ void load(const DecodeParams& p, const SeqTable& t, const Span& sp) {
    L = t.len[b];
    lo = first_visible(L, p.window);
    seg_end = t.prefix[b + 1] < sp.end ? t.prefix[b + 1] : sp.end;
  }
  // position of row 0 of flattened page f (f within sequence b)
  __device__ __forceinline__ int pos0(const SeqTable& t, int f) const {
    return (lo / kPage + (f - t.prefix[b])) * kPage;
  }
  // move to the sequence of flattened page f (skipping empty sequences)
  __device__ __forceinline__ void advance(const DecodeParams& p, const SeqTable& t, const Span& sp, int f) {
    if (f >= t.prefix[b + 1]) {
      do { ++b; } while (f >= t.prefix[b + 1]);
      load(p, t, sp);
    }
  }
  // true when this block holds every visible page of sequence b
  __device__ __forceinline__ bool whole(const SeqTable& t, const Span& sp) const {
    return t.prefix[b] >= sp.begin && t.prefix[b + 1] <= sp.end;
  }
};

// The first sequence after b with a visible page inside the span, or -1.
// It is the sequence PageCursor::advance moves to when b's pages end.
__device__ __forceinline__ int next_seq_in_span(const DecodeParams& p, const SeqTable& t, const Span& sp, int b) {
  int nb = b + 1;
  while (nb < p.batch && t.prefix[nb + 1] == t.prefix[nb]) ++nb;  // skip empty sequences
  return (nb < p.batch && t.prefix[nb] < sp.end) ? nb : -1;
}

// The blocks g0..g1 whose spans hold pages of sequence b (b non-empty), given
// the number of non-empty sequences before it: its real pages sit at weighted
// positions prefix[b] + kSeqWeight * (nonempty_before + 1) onwards.  The
// combine kernel derives the same range from seq_lens.
__device__ __forceinline__ void seq_blocks(const SeqTable& t, int b, int nonempty_before, int& g0, int& g1) {
  const int w = t.prefix[b] + kSeqWeight * (nonempty_before + 1);
  const int n = t.prefix[b + 1] - t.prefix[b];
  g0 = w / t.per;
  g1 = (w + n - 1) / t.per;
}

// Lets the dependent (combine) grid launch while this grid runs.
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Waits until the grid this one depends on has completed and its writes are visible.
__device__ __forceinline__ void wait_for_primary_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace pda
