// combine.cuh -- merges the per-split partial results of the decode kernels.
//
// Split i of row (b, h) left an unnormalised output O_i = sum_l e^{s_l - m_i} v_l,
// its running max m_i (log2 units) and sum l_i = sum_l e^{s_l - m_i}.  With
// M = max_i m_i the softmax over the union of the splits is
//     o = sum_i 2^{m_i - M} O_i / sum_i 2^{m_i - M} l_i,
// an exact regrouping of the one softmax over all visible positions
// (Attention.lean `softmax`).  Splits without a visible position (l_i = 0)
// are skipped outright, so uninitialised workspace never enters the sum.
#pragma once

#include "common.cuh"

namespace pda {

template <int kD>
__global__ void __launch_bounds__(kD / 4) combine_kernel(const __grid_constant__ DecodeParams p) {
  const int h = blockIdx.x;
  const int b = blockIdx.y;
  const int Hq = gridDim.x;
  const int d0 = threadIdx.x * 4;
  const size_t row = static_cast<size_t>(b) * Hq + h;
  const float2* ml = p.part_ml + row * p.num_splits;
  float M = -INFINITY;
  for (int i = 0; i < p.num_splits; ++i) {
    const float2 e = ml[i];
    if (e.y > 0.f) M = fmaxf(M, e.x);
  }
  float Lsum = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int i = 0; i < p.num_splits; ++i) {
      const float2 e = ml[i];
      if (e.y > 0.f) {
        const float w = exp2f(e.x - M);
        Lsum += w * e.y;
        const float4 a = *reinterpret_cast<const float4*>(p.part_o + (row * p.num_splits + i) * kD + d0);
        O.x += w * a.x;
        O.y += w * a.y;
        O.z += w * a.z;
        O.w += w * a.w;
      }
    }
  }
  const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
  store_out4(p, row * kD + d0, make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv));
}

}  // namespace pda
