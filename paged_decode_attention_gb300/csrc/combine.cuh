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
// One 4-warp block per (row b*Hq + h, slice of 128 dims).  Warp w takes the
// partials i = w, w+4, ...; each lane owns 4 dims and issues the (m, l) pair
// and the 16-byte slice of up to kPerWarp partials in one go, so a row costs
// one memory round trip (more only beyond 4*kPerWarp partials).  The maxima
// and the weighted sums are then merged across the warps in shared memory.
// The schedule arithmetic runs before griddepcontrol.wait, overlapping the
// decode kernel (the combine is launched as its programmatic dependent).
#pragma once

#include "common.cuh"

namespace pda {

constexpr int kCombineCols = 128;  // dims per combine block
constexpr int kCombineWarps = 4;
constexpr int kPerWarp = 8;        // partials a warp keeps in flight per round (74 registers: one
                                   // block fits beside the decode blocks of an SM)

template <int kD>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int kSlices = kD / kCombineCols;
  __shared__ float s_max[kCombineWarps];
  __shared__ float s_l[kCombineWarps];
  __shared__ float4 s_o[kCombineWarps][32];

  const int h = blockIdx.x / kSlices;
  const int slice = blockIdx.x % kSlices;
  const int b = blockIdx.y;
  const int Hq = gridDim.x / kSlices;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const size_t row = static_cast<size_t>(b) * Hq + h;
  const int d0 = slice * kCombineCols + lane * 4;

  // The schedule, on the decode kernels' weighted page list (kSeqWeight
  // virtual pages before every non-empty sequence): weighted pages before
  // sequence b, its own real pages, and the weighted total.  Warp 0 reads
  // seq_lens four at a time and shares the three sums.
  __shared__ int s_sched[3];
  if (warp == 0) {
    int before = 0, mine = 0, total = 0;
    const int nvec = p.batch >> 2;  // seq_lens is 16-byte aligned
    for (int v = lane; v <= nvec; v += 32) {
      int L[4];
      if (v < nvec) {
        const int4 w = reinterpret_cast<const int4*>(p.seq_lens)[v];
        L[0] = w.x; L[1] = w.y; L[2] = w.z; L[3] = w.w;
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) L[k] = 4 * v + k < p.batch ? p.seq_lens[4 * v + k] : 0;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int j = 4 * v + k;
        const int n = j < p.batch ? visible_pages(clamp_len(p, L[k], false), p.window) : 0;
        const int wn = n > 0 ? n + kSeqWeight : 0;
        total += wn;
        before += j < b ? wn : 0;
        mine += j == b ? n : 0;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      before += __shfl_xor_sync(0xffffffffu, before, o);
      mine += __shfl_xor_sync(0xffffffffu, mine, o);
      total += __shfl_xor_sync(0xffffffffu, total, o);
    }
    if (lane == 0) {
      s_sched[0] = before;
      s_sched[1] = mine;
      s_sched[2] = total;
    }
  }
  __syncthreads();
  // A block with nothing to merge returns at once, except block (0, 0),
  // which first waits for the decode grid: the combine grid then cannot
  // complete before the decode grid, so the next kernel in the stream, which
  // waits for the combine grid, also finds the decode grid's work done.
  const auto done = [&]() {
    if (blockIdx.x == 0 && blockIdx.y == 0) wait_for_primary_grid();
  };
  const int before = s_sched[0], mine = s_sched[1], total = s_sched[2];
  if (mine == 0) {
    if (warp == 0) store_out4(p, row * kD + d0, make_float4(0.f, 0.f, 0.f, 0.f));
    done();
    return;
  }
  const int per = span_pages(total, p.grid_x, p.min_pages);
  const int g0 = (before + kSeqWeight) / per;
  const int g1 = (before + kSeqWeight + mine - 1) / per;
  if (g0 == g1) {  // one block held the whole sequence and wrote o
    done();
    return;
  }
  const int ns = g1 - g0 + 1;
  if (ns > kMaxSplits || (static_cast<int64_t>(g1) + b + 1) * Hq > p.part_rows) {
    if (threadIdx.x == 0) report(p.status, ATTN_DEV_INTERNAL);  // cannot happen: partials beyond the workspace
    done();
    return;
  }

  wait_for_primary_grid();
  allow_dependent_launch();  // the next kernel may start its prologue

  const size_t stride = static_cast<size_t>(Hq) * kD;
  const float2* ml = p.part_ml + (static_cast<size_t>(g0) + b) * Hq + h;
  const float* base = p.part_o + ((static_cast<size_t>(g0) + b) * Hq + h) * kD + d0;

  // This warp's partials, kPerWarp per round: running (max, sum, output) of
  // the rounds so far, in the same log2 units as the decode kernels.
  float wm = -INFINITY, wl = 0.f;
  float4 wo = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int r0 = warp; r0 < ns; r0 += kCombineWarps * kPerWarp) {
    float2 e[kPerWarp];
    float4 a[kPerWarp];
#pragma unroll
    for (int j = 0; j < kPerWarp; ++j) {
      const int i = r0 + j * kCombineWarps;
      e[j] = i < ns ? ml[static_cast<size_t>(i) * Hq] : make_float2(-INFINITY, 0.f);
      a[j] = i < ns ? *reinterpret_cast<const float4*>(base + i * stride) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float rm = wm;
#pragma unroll
    for (int j = 0; j < kPerWarp; ++j)
      if (e[j].y > 0.f) rm = fmaxf(rm, e[j].x);
    if (rm == -INFINITY) continue;
    const float cw = wm == -INFINITY ? 0.f : exp2f(wm - rm);
    wl *= cw;
    wo.x *= cw; wo.y *= cw; wo.z *= cw; wo.w *= cw;
#pragma unroll
    for (int j = 0; j < kPerWarp; ++j) {
      if (e[j].y > 0.f) {  // partials without a visible position are skipped, whatever they hold
        const float w = exp2f(e[j].x - rm);
        wl += w * e[j].y;
        wo.x += w * a[j].x; wo.y += w * a[j].y; wo.z += w * a[j].z; wo.w += w * a[j].w;
      }
    }
    wm = rm;
  }

  // merge the warps
  if (lane == 0) s_max[warp] = wm;
  __syncthreads();
  float M = s_max[0];
#pragma unroll
  for (int w = 1; w < kCombineWarps; ++w) M = fmaxf(M, s_max[w]);
  const float f = (M == -INFINITY || wm == -INFINITY) ? 0.f : exp2f(wm - M);
  if (lane == 0) s_l[warp] = f * wl;
  s_o[warp][lane] = make_float4(f * wo.x, f * wo.y, f * wo.z, f * wo.w);
  __syncthreads();
  if (warp == 0) {
    float L = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) {
      L += s_l[w];
      const float4 v = s_o[w][lane];
      O.x += v.x; O.y += v.y; O.z += v.z; O.w += v.w;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    store_out4(p, row * kD + d0, make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv));
  }
}

}  // namespace pda
