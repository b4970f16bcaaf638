// rope.cuh -- accurate RoPE angles in fp32 (attn.rope, Gemma-4-12B model
// page, "Compute-graph nodes"; the per-layer constants under "What to watch
// for"): pair i of a head turns by pos * theta^(-2i/D).
//
// pos * f_i rounded to fp32 is off by up to 0.016 rad at pos = 262143, so f_i
// is carried as a pair of floats hi + lo (about 46 significant bits),
// pos * f_i as a float plus its exact fma remainder, and the turns are removed
// with a three-part 2*pi (Cody and Waite's additive range reduction) before
// __sincosf of an argument in [-pi, pi].
#pragma once

#include <cstdint>

namespace pda {

struct FloatPair {  // hi + lo, |lo| <= ulp(hi) / 2
  float hi, lo;
};

// 2*pi as three floats, [0] and [1] with 8 significant bits each (so n * part
// is exact for n < 2^16 turns), [2] the float nearest to the rest; and 1/(2 pi).
struct TwoPi {
  float part[3];
  float inv;
};

// a * b in double-float arithmetic: relative error about 2^-46.
__device__ __forceinline__ FloatPair df_mul(FloatPair a, FloatPair b) {
  const float p = a.hi * b.hi;
  float e = fmaf(a.hi, b.hi, -p);  // exact error of p
  e = fmaf(a.hi, b.lo, fmaf(a.lo, b.hi, e));
  const float hi = p + e;
  return {hi, e - (hi - p)};
}

// cos and sin of pos * (f.hi + f.lo) for an integer 0 <= pos < 2^24 and an
// angle below 2^16 turns.
__device__ __forceinline__ void rope_angle(const TwoPi& tp, FloatPair f, int pos, float& c, float& s) {
  const float fp = static_cast<float>(pos);  // exact
  const float hi = fp * f.hi;
  const float err = fmaf(fp, f.hi, -hi);  // pos * f.hi - hi, exactly
  const float small = fmaf(fp, f.lo, err);
  const float n = rintf(hi * tp.inv);
  float r = fmaf(-n, tp.part[0], hi);  // n * part[0] and n * part[1] are exact
  r = fmaf(-n, tp.part[1], r);
  r = fmaf(-n, tp.part[2], r);
  r += small;
  __sincosf(r, &s, &c);
}

}  // namespace pda
