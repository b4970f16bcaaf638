// combine.cuh -- merges the partial results of sequences whose pages were
// split across blocks by the balanced schedule (common.cuh).
//
// A block g that held only part of sequence b left, in slot g + b, an
// unnormalised output O_g = sum_l e^{s_l - m_g} v_l, its running max m_g
// (log2 units) and sum l_g = sum_l e^{s_l - m_g}.  With M = max_g m_g the
// softmax over the union of the spans is
//     o = sum_g 2^{m_g - M} O_g / sum_g 2^{m_g - M} l_g,
// an exact regrouping of the one softmax over all visible positions
// (Attention.lean `softmax`).  Partials with l_g = 0 get weight 0 and are
// never read.  Rows of sequences with no visible position are written as 0
// (the empty sum); rows finished whole by one block are left untouched.
//
// One single-warp block per (row b*Hq + h, slice of 128 dims): each lane owns
// 4 dims and keeps 16 partial rows in flight, so a row with tens of
// partials costs a couple of L2 round trips.  The schedule arithmetic runs
// before griddepcontrol.wait, overlapping the decode kernel (the combine is
// launched as its programmatic dependent).
#pragma once

#include "common.cuh"

namespace pda {

constexpr int kCombineCols = 128;  // dims per combine block
constexpr int kCombineInFlight = 16;

template <int kD>
__global__ void __launch_bounds__(32) combine_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int kSlices = kD / kCombineCols;
  __shared__ float w_s[kMaxSplits];

  const int h = blockIdx.x / kSlices;
  const int slice = blockIdx.x % kSlices;
  const int b = blockIdx.y;
  const int Hq = gridDim.x / kSlices;
  const int lane = threadIdx.x;
  const size_t row = static_cast<size_t>(b) * Hq + h;
  const int d0 = slice * kCombineCols + lane * 4;

  // the schedule: pages before sequence b, its own pages, and the total
  int before = 0, mine = 0, total = 0;
  for (int j = lane; j < p.batch; j += 32) {
    const int n = visible_pages(clamp_len(p, p.seq_lens[j], false), p.window);
    total += n;
    before += j < b ? n : 0;
    mine += j == b ? n : 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    mine += __shfl_xor_sync(0xffffffffu, mine, o);
    total += __shfl_xor_sync(0xffffffffu, total, o);
  }
  if (mine == 0) {
    store_out4(p, row * kD + d0, make_float4(0.f, 0.f, 0.f, 0.f));
    return;
  }
  const int per = span_pages(total, p.grid_x, p.min_pages);
  const int g0 = before / per;
  const int g1 = (before + mine - 1) / per;
  if (g0 == g1) return;  // one block held the whole sequence and wrote o
  const int ns = g1 - g0 + 1;
  if (ns > kMaxSplits || (static_cast<int64_t>(g1) + b + 1) * Hq > p.part_rows) {
    if (lane == 0) report(p.status, ATTN_DEV_INTERNAL);  // cannot happen: partials beyond the workspace
    return;
  }

  wait_for_primary_grid();

  // weights 2^{m_g - M} over the partials that saw a visible position
  const float2* ml = p.part_ml + (static_cast<size_t>(g0) + b) * Hq + h;
  float mx = -INFINITY;
  for (int i = lane; i < ns; i += 32) {
    const float2 e = ml[static_cast<size_t>(i) * Hq];
    w_s[i] = e.y > 0.f ? e.x : -INFINITY;
    mx = fmaxf(mx, w_s[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float ls = 0.f;
  for (int i = lane; i < ns; i += 32) {
    const float wi = (mx == -INFINITY || w_s[i] == -INFINITY) ? 0.f : exp2f(w_s[i] - mx);
    ls += wi * ml[static_cast<size_t>(i) * Hq].y;
    w_s[i] = wi;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
  __syncwarp();

  // o = sum_g w_g O_g / sum_g w_g l_g
  const size_t stride = static_cast<size_t>(Hq) * kD;
  const float* base = p.part_o + ((static_cast<size_t>(g0) + b) * Hq + h) * kD + d0;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i0 = 0; i0 < ns; i0 += kCombineInFlight) {
    float4 a[kCombineInFlight];
#pragma unroll
    for (int j = 0; j < kCombineInFlight; ++j) {
      const int i = i0 + j;
      a[j] = (i < ns && w_s[i] != 0.f) ? *reinterpret_cast<const float4*>(base + i * stride)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < kCombineInFlight; ++j) {
      const int i = i0 + j;
      const float wi = i < ns ? w_s[i] : 0.f;
      O.x += wi * a[j].x;
      O.y += wi * a[j].y;
      O.z += wi * a[j].z;
      O.w += wi * a[j].w;
    }
  }
  const float inv = ls > 0.f ? 1.f / ls : 0.f;
  store_out4(p, row * kD + d0, make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv));
}

}  // namespace pda
