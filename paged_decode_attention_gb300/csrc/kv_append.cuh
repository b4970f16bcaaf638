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
// never leaves its lane; each half is one 8- or 16-byte access.  Sums of
// squares are reduced with shuffles in fp32.
//
// RoPE angles as in rope.cuh.  f_i is not looked up per lane (a kernel-
// parameter table read at 32 different offsets is served one offset at a
// time): lane l forms it as
//   theta^(-2 V l / D) * theta^(-2 j / D),  j = i - V l,
// the first factor the product of theta^(-2 V 2^k / D) over the set bits k
// of l, every factor a host-computed float pair read at the same offset by
// all lanes, and every product a double-float product (Dekker's, with the
// fma giving the exact error of the leading product).
//
// Outputs are rounded once to bf16 (nearest even).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "common.cuh"
#include "rope.cuh"

namespace pda {
namespace append {

constexpr int kLaneBits = 5;  // lanes 0..31
constexpr int kMaxV = 8;      // D / 64 for D = 512

struct AppendParams {
  const __nv_bfloat16* qkv;    // [B, row_len]
  const __nv_bfloat16* w_q;    // [D]
  const __nv_bfloat16* w_k;    // [D]
  const int32_t* block_table;  // [B, max_blocks]
  const int32_t* positions;    // [B]
  __nv_bfloat16* q_out;        // [B, Hq, D]
  __nv_bfloat16* k_pool;       // [num_pages, 16, Hkv, D]; null: values-only global cache
  __nv_bfloat16* v_pool;
  int32_t* status;             // optional ATTN_DEV_* word
  int64_t num_pages;
  int32_t batch;
  int32_t max_blocks;
  float eps;
  TwoPi two_pi;
  FloatPair lane_factor[kLaneBits];  // theta^(-2 V 2^k / D)
  FloatPair dim_factor[kMaxV];       // theta^(-2 j / D), j < V
};

// theta^(-2 V lane / D): the lane's share of its frequencies.
__device__ __forceinline__ FloatPair lane_frequency(const AppendParams& p, int lane) {
  FloatPair f{1.f, 0.f};
#pragma unroll
  for (int k = 0; k < kLaneBits; ++k) {
    const FloatPair m = (lane >> k) & 1 ? p.lane_factor[k] : FloatPair{1.f, 0.f};
    f = df_mul(f, m);
  }
  return f;
}

template <int kD>
struct Row {
  static constexpr int kV = kD / 64;  // dims per lane in each half
  float lo[kV], hi[kV];               // dims [kV*lane, +kV) and [D/2 + kV*lane, +kV)
};

// kV consecutive bf16 (8 or 16 bytes) <-> fp32
template <int kV>
__device__ __forceinline__ void load_bf16(const __nv_bfloat16* src, float* out) {
  static_assert(kV == 4 || kV == 8, "one 8- or 16-byte access");
  uint32_t w[kV / 2];
  if constexpr (kV == 8) {
    const uint4 u = *reinterpret_cast<const uint4*>(src);
    w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
  } else {
    const uint2 u = *reinterpret_cast<const uint2*>(src);
    w[0] = u.x; w[1] = u.y;
  }
#pragma unroll
  for (int j = 0; j < kV / 2; ++j) {
    const float2 f = bf16x2_to_float2(w[j]);
    out[2 * j] = f.x;
    out[2 * j + 1] = f.y;
  }
}

template <int kV>
__device__ __forceinline__ void store_bf16(__nv_bfloat16* dst, const float* in) {
  uint32_t w[kV / 2];
#pragma unroll
  for (int j = 0; j < kV / 2; ++j) w[j] = pack_bf16x2(in[2 * j], in[2 * j + 1]);
  if constexpr (kV == 8) {
    *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
  }
}

template <int kD>
__device__ __forceinline__ void load_row(const __nv_bfloat16* src, Row<kD>& r) {
  constexpr int kV = Row<kD>::kV;
  const int lane = threadIdx.x & 31;
  load_bf16<kV>(src + kV * lane, r.lo);
  load_bf16<kV>(src + kD / 2 + kV * lane, r.hi);
}

template <int kD>
__device__ __forceinline__ void store_row(__nv_bfloat16* dst, const Row<kD>& r) {
  constexpr int kV = Row<kD>::kV;
  const int lane = threadIdx.x & 31;
  store_bf16<kV>(dst + kV * lane, r.lo);
  store_bf16<kV>(dst + kD / 2 + kV * lane, r.hi);
}

// x / sqrt(mean(x^2) + eps)
template <int kD>
__device__ __forceinline__ void normalise(Row<kD>& r, float eps) {
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
}

template <int kD>
__device__ __forceinline__ void scale(Row<kD>& r, const Row<kD>& w) {
#pragma unroll
  for (int j = 0; j < Row<kD>::kV; ++j) {
    r.lo[j] *= w.lo[j];
    r.hi[j] *= w.hi[j];
  }
}

template <int kD, int kPairs>
__device__ __forceinline__ void rotate(const AppendParams& p, Row<kD>& r, int pos) {
  constexpr int kV = Row<kD>::kV;
  const int lane = threadIdx.x & 31;
  if (kV * lane >= kPairs) return;  // kPairs is a multiple of kV
  const FloatPair fl = lane_frequency(p, lane);
#pragma unroll
  for (int j = 0; j < kV; ++j) {
    float c, s;
    rope_angle(p.two_pi, df_mul(fl, p.dim_factor[j]), pos, c, s);
    const float a = r.lo[j], b = r.hi[j];
    r.lo[j] = a * c - b * s;
    r.hi[j] = b * c + a * s;
  }
}

// Warps of a token: q heads 0..kHq-1, then one warp per KV head (key, and
// value when shared), then, unless shared, one warp per value head.
template <int kD, int kHq, int kHkv, int kPairs, bool kShared>
__global__ void __launch_bounds__(128) append_kernel(const __grid_constant__ AppendParams p) {
  constexpr int kRowsPerToken = kHq + (kShared ? 1 : 2 * kHkv);
  constexpr int kRowLen = kHq * kD + (kShared ? kD : 2 * kHkv * kD);
  static_assert(!kShared || kHkv == 1, "a shared key/value source is one head");
  static_assert(kPairs % Row<kD>::kV == 0 && kPairs <= kD / 2, "whole lanes of active pairs");
  // The previous kernel in the stream may still be writing qkv or the tables.
  wait_for_primary_grid();
  allow_dependent_launch();
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (gw >= p.batch * kRowsPerToken) return;
  const int b = gw / kRowsPerToken;
  const int r = gw % kRowsPerToken;
  const int is_q = r < kHq;
  const int c = kShared ? 0 : (r - kHq) % kHkv;
  const bool is_value = !kShared && r >= kHq + kHkv;
  const __nv_bfloat16* row = p.qkv + static_cast<size_t>(b) * kRowLen;
  const __nv_bfloat16* src = is_q ? row + r * kD : row + kHq * kD + (is_value ? (kHkv + c) * kD : c * kD);

  // independent loads first: position, the row, its norm weights
  const int pos = p.positions[b];
  Row<kD> x, w;
  load_row<kD>(src, x);
  if (!is_value) load_row<kD>(is_q ? p.w_q : p.w_k, w);

  if (is_q) {
    normalise<kD>(x, p.eps);
    scale<kD>(x, w);
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

  normalise<kD>(x, p.eps);
  if (is_value || kShared) store_row<kD>(p.v_pool + (slot * kHkv + c) * kD, x);  // v_norm: no weights
  if (is_value || (kShared && p.k_pool == nullptr)) return;  // a values-only cache rebuilds keys when read
  scale<kD>(x, w);
  rotate<kD, kPairs>(p, x, pos);
  store_row<kD>(p.k_pool + (slot * kHkv + c) * kD, x);
}

}  // namespace append
}  // namespace pda
