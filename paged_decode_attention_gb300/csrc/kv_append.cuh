// kv_append.cuh -- the steps that feed the decode for one new token per
// sequence: per-head norms, RoPE, and the append of the token's key and value
// to the paged cache (Gemma-4-12B model page, "Compute-graph nodes"):
//
//   attn.qk_norm  y[i] = x[i] / sqrt(sum_j x[j]^2 / D + eps) * w[i]   (q and k heads)
//   attn.v_norm   y[i] = x[i] / sqrt(sum_j x[j]^2 / D + eps)           (v heads)
//   attn.rope     rotate pairs (i, i + D/2) by pos * theta^(-2i/D), i < active
//
// Sliding layers: theta 10,000, all 128 pairs of D = 256 active, q 16 heads,
// k and v 8 heads each.  Global layers: theta 1,000,000, the first 64 of the
// 256 pairs of D = 512 active, q 16 heads and one head x whose qk_norm and
// RoPE give the key and whose v_norm gives the value ("values = keys").
//
// One warp per head row of one token.  Lane l holds dims [V l, V l + V) and
// their rotation partners [D/2 + V l, D/2 + V l + V), V = D / 64, so a pair
// never leaves its lane.  Sums of squares are reduced with shuffles in fp32.
// The rotation angle pos * f_i is formed without the rounding of pos * f_i
// in fp32 (which reaches 0.016 rad at pos = 262143): f_i is split on the
// host into f_hi + f_lo, the product pos * f_hi is carried as a float plus
// its exact fma remainder, and the turns are removed with a three-part
// 2*pi (Cody and Waite's additive range reduction) before __sincosf of an
// argument in [-pi, pi].  Outputs are rounded once to bf16 (nearest even).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "common.cuh"

namespace pda {
namespace append {

constexpr int kMaxPairs = 128;

struct AppendParams {
  const __nv_bfloat16* qkv;    // [B, row_len]
  const __nv_bfloat16* w_q;    // [D]
  const __nv_bfloat16* w_k;    // [D]
  const int32_t* block_table;  // [B, max_blocks]
  const int32_t* positions;    // [B]
  __nv_bfloat16* q_out;        // [B, Hq, D]
  __nv_bfloat16* k_pool;       // [num_pages, 16, Hkv, D]
  __nv_bfloat16* v_pool;
  int32_t* status;             // optional ATTN_DEV_* word
  int64_t num_pages;
  int32_t batch;
  int32_t max_blocks;
  float eps;
  float two_pi[3];             // 2*pi = two_pi[0] + two_pi[1] + two_pi[2]; [0], [1] with 8 significant bits
  float inv_two_pi;
  float freq_hi[kMaxPairs];    // theta^(-2i/D) = freq_hi[i] + freq_lo[i]
  float freq_lo[kMaxPairs];
};

// cos and sin of pos * (freq_hi + freq_lo) for an integer 0 <= pos < 2^24.
__device__ __forceinline__ void rope_angle(const AppendParams& p, int i, int pos, float& c, float& s) {
  const float fp = static_cast<float>(pos);  // exact
  const float hi = fp * p.freq_hi[i];
  const float err = fmaf(fp, p.freq_hi[i], -hi);  // pos * freq_hi - hi, exactly
  const float small = fmaf(fp, p.freq_lo[i], err);
  const float n = rintf(hi * p.inv_two_pi);
  float r = fmaf(-n, p.two_pi[0], hi);  // n * two_pi[0] and n * two_pi[1] are exact for n < 2^16
  r = fmaf(-n, p.two_pi[1], r);
  r = fmaf(-n, p.two_pi[2], r);
  r += small;
  __sincosf(r, &s, &c);
}

template <int kD>
struct Row {
  static constexpr int kV = kD / 64;  // dims per lane in each half
  float lo[kV], hi[kV];               // dims [kV*lane, +kV) and [D/2 + kV*lane, +kV)
};

template <int kD>
__device__ __forceinline__ void load_row(const __nv_bfloat16* src, Row<kD>& r) {
  const int lane = threadIdx.x & 31;
  constexpr int kV = Row<kD>::kV;
#pragma unroll
  for (int j = 0; j < kV; j += 2) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + kV * lane + j));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + kD / 2 + kV * lane + j));
    r.lo[j] = a.x; r.lo[j + 1] = a.y;
    r.hi[j] = b.x; r.hi[j + 1] = b.y;
  }
}

// x / sqrt(mean(x^2) + eps), times w when given.
template <int kD>
__device__ __forceinline__ void normalise(Row<kD>& r, const __nv_bfloat16* w, float eps) {
  const int lane = threadIdx.x & 31;
  constexpr int kV = Row<kD>::kV;
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kV; ++j) ss = fmaf(r.lo[j], r.lo[j], fmaf(r.hi[j], r.hi[j], ss));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float inv = rsqrtf(ss / static_cast<float>(kD) + eps);
#pragma unroll
  for (int j = 0; j < kV; ++j) {
    r.lo[j] *= inv;
    r.hi[j] *= inv;
  }
  if (w) {
#pragma unroll
    for (int j = 0; j < kV; ++j) {
      r.lo[j] *= __bfloat162float(w[kV * lane + j]);
      r.hi[j] *= __bfloat162float(w[kD / 2 + kV * lane + j]);
    }
  }
}

template <int kD, int kPairs>
__device__ __forceinline__ void rotate(const AppendParams& p, Row<kD>& r, int pos) {
  const int lane = threadIdx.x & 31;
  constexpr int kV = Row<kD>::kV;
#pragma unroll
  for (int j = 0; j < kV; ++j) {
    const int i = kV * lane + j;
    if (i < kPairs) {
      float c, s;
      rope_angle(p, i, pos, c, s);
      const float a = r.lo[j], b = r.hi[j];
      r.lo[j] = a * c - b * s;
      r.hi[j] = b * c + a * s;
    }
  }
}

template <int kD>
__device__ __forceinline__ void store_row(__nv_bfloat16* dst, const Row<kD>& r) {
  const int lane = threadIdx.x & 31;
  constexpr int kV = Row<kD>::kV;
#pragma unroll
  for (int j = 0; j < kV; j += 2) {
    *reinterpret_cast<uint32_t*>(dst + kV * lane + j) = pack_bf16x2(r.lo[j], r.lo[j + 1]);
    *reinterpret_cast<uint32_t*>(dst + kD / 2 + kV * lane + j) = pack_bf16x2(r.hi[j], r.hi[j + 1]);
  }
}

// Warps of a token: q heads 0..kHq-1, then one warp per KV head (key, and
// value when shared), then, unless shared, one warp per value head.
template <int kD, int kHq, int kHkv, int kPairs, bool kShared>
__global__ void __launch_bounds__(128) append_kernel(const __grid_constant__ AppendParams p) {
  constexpr int kRowsPerToken = kHq + (kShared ? 1 : 2 * kHkv);
  constexpr int kRowLen = kHq * kD + (kShared ? kD : 2 * kHkv * kD);
  static_assert(!kShared || kHkv == 1, "a shared key/value source is one head");
  // The previous kernel in the stream may still be writing qkv or the tables.
  wait_for_primary_grid();
  allow_dependent_launch();
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (gw >= p.batch * kRowsPerToken) return;
  const int b = gw / kRowsPerToken;
  const int r = gw % kRowsPerToken;
  const int pos = p.positions[b];
  const __nv_bfloat16* row = p.qkv + static_cast<size_t>(b) * kRowLen;
  Row<kD> x;

  if (r < kHq) {  // query head r
    load_row<kD>(row + r * kD, x);
    normalise<kD>(x, p.w_q, p.eps);
    rotate<kD, kPairs>(p, x, pos < 0 ? 0 : pos);
    store_row<kD>(p.q_out + (static_cast<size_t>(b) * kHq + r) * kD, x);
    return;
  }

  // the token's cache slot
  const int page = pos >= 0 ? pos / ATTN_PAGE_SIZE : -1;
  if (pos < 0 || pos >= ATTN_MAX_SEQ_LEN || page >= p.max_blocks) {
    if ((threadIdx.x & 31) == 0) report(p.status, ATTN_DEV_BAD_SEQ_LEN);
    return;
  }
  const int32_t phys = p.block_table[static_cast<int64_t>(b) * p.max_blocks + page];
  if (phys < 0 || static_cast<int64_t>(phys) >= p.num_pages) {
    if ((threadIdx.x & 31) == 0) report(p.status, ATTN_DEV_BAD_PAGE);
    return;
  }
  const size_t slot = static_cast<size_t>(phys) * ATTN_PAGE_SIZE + pos % ATTN_PAGE_SIZE;

  const int c = kShared ? 0 : (r - kHq) % kHkv;
  const bool is_value = !kShared && r >= kHq + kHkv;
  load_row<kD>(row + kHq * kD + (is_value ? (kHkv + c) * kD : c * kD), x);
  if (is_value) {
    normalise<kD>(x, nullptr, p.eps);
    store_row<kD>(p.v_pool + (slot * kHkv + c) * kD, x);
    return;
  }
  if (kShared) {  // the value is the same head, normalised without weights
    Row<kD> v = x;
    normalise<kD>(v, nullptr, p.eps);
    store_row<kD>(p.v_pool + (slot * kHkv + c) * kD, v);
  }
  normalise<kD>(x, p.w_k, p.eps);
  rotate<kD, kPairs>(p, x, pos);
  store_row<kD>(p.k_pool + (slot * kHkv + c) * kD, x);
}

}  // namespace append
}  // namespace pda
