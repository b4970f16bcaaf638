// common.cuh -- launch parameters and the per-(sequence, split) visible range
// shared by the decode kernels.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "attn_decode.h"
#include "ptx.cuh"

namespace pda {

constexpr int kPage = ATTN_PAGE_SIZE;       // token rows per cache page
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeParams {
  const __nv_bfloat16* q;      // [batch, Hq, D]
  const int32_t* block_table;  // [batch, max_blocks]
  const int32_t* seq_lens;     // [batch]
  void* o;                     // [batch, Hq, D], bf16 or fp32
  float* part_o;               // [batch, Hq, num_splits, D]  (num_splits > 1)
  float2* part_ml;             // [batch, Hq, num_splits]: (running max in log2 units, sum)
  int32_t* status;             // optional ATTN_DEV_* word
  int64_t num_pages;
  int32_t batch;
  int32_t max_blocks;
  int32_t window;              // > 0 sliding rule, <= 0 none
  int32_t num_splits;
  int32_t pages_per_split;
  int32_t out_f32;
};

// Visible positions [lo, L) of sequence b and the page range [page_begin,
// page_end) of one split.  Decode query at p = L-1 (Attention.lean
// decodeGQA); with a window w the visible keys are p-w < l <= p
// (Attention.lean slidingGQA).  Splits cut the visible pages into runs of
// pages_per_split, counted from the first visible page; the last split takes
// whatever remains, so an understated max_seq_len costs speed, not results.
struct SplitRange {
  int L;
  int lo;
  int page_begin;
  int page_end;
};

__device__ __forceinline__ SplitRange split_range(const DecodeParams& p, int b, int split) {
  SplitRange r;
  int L = p.seq_lens[b];
  const int L_cap = p.max_blocks * kPage;
  if (L < 0 || L > L_cap) {
    if (threadIdx.x == 0) report(p.status, ATTN_DEV_BAD_SEQ_LEN);
    L = L < 0 ? 0 : L_cap;
  }
  r.L = L;
  r.lo = (p.window > 0 && L > p.window) ? L - p.window : 0;
  r.page_begin = r.page_end = 0;
  if (L > 0) {
    const int first = r.lo / kPage;
    const int last = (L - 1) / kPage;  // inclusive
    const int begin = first + split * p.pages_per_split;
    int end = (split == p.num_splits - 1) ? last + 1 : begin + p.pages_per_split;
    if (end > last + 1) end = last + 1;
    if (begin <= last) {
      r.page_begin = begin;
      r.page_end = end;
    }
  }
  return r;
}

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

// Producer side of the page pipeline, run by one whole warp: walks the pages
// of a split, reads their block-table entries 32 at a time (one coalesced
// load per 32 pages, fetched a batch ahead), and has lane 0 issue the TMA
// copies `issue(stage, y)` for page row coordinate y.  A page id outside
// [0, num_pages) is replaced by a fully out-of-range coordinate, which the
// copy engine fills with zeros, and ATTN_DEV_BAD_PAGE is raised.  Before it
// returns, the warp waits (bounded) until every copy it issued has landed,
// so no copy is in flight when the block retires.
template <int kStages, int kTxBytes, typename Issue>
__device__ __forceinline__ void produce_pages(const DecodeParams& p, int b, const SplitRange& r,
                                              uint64_t* full, uint64_t* empty, Issue issue) {
  const int lane = threadIdx.x & 31;
  const int n_pages = r.page_end - r.page_begin;
  const int32_t* bt = p.block_table + static_cast<int64_t>(b) * p.max_blocks + r.page_begin;
  int nxt = lane < n_pages ? bt[lane] : 0;
  int cur = 0;
  int issued = 0;
  bool ok = true;
  for (int i = 0; i < n_pages; ++i) {
    if ((i & 31) == 0) {
      cur = nxt;
      const int j = i + 32 + lane;
      nxt = j < n_pages ? bt[j] : 0;
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

}  // namespace pda
