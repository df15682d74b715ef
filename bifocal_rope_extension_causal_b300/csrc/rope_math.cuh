// Rotary-embedding angles, accurate at long positions.
//
// RoPE (RoFormer) turns coordinate pair i by the angle n * omega_i with
// omega_i = theta^(-2i/d).  At n ~ 1.3e5 the angle is ~1.3e5 rad, and the
// float product n * omega_i is already off by ~1e-2 rad there, so the angle
// is formed and reduced modulo 2*pi in double precision (n is exact, the
// product is correctly rounded to ~1.5e-11 rad, the reduction uses 2*pi split
// into two doubles), and only the reduced angle in [-pi, pi] goes to the
// float sincosf.  The result is within ~3e-7 rad of the exact angle.
#pragma once
#include <stdint.h>

namespace jl {

// 2*pi as the nearest double plus the rounding remainder.
constexpr double kTwoPiHi = 6.283185307179586;
constexpr double kTwoPiLo = 2.4492935982947064e-16;
constexpr double kInvTwoPi = 0.15915494309189535;

__device__ __forceinline__ float2 rope_cos_sin(long long n, double omega) {
  const double a = static_cast<double>(n) * omega;
  const double m = rint(a * kInvTwoPi);
  double r = fma(-m, kTwoPiHi, a);
  r = fma(-m, kTwoPiLo, r);
  float s, c;
  sincosf(static_cast<float>(r), &s, &c);
  return make_float2(c, s);
}

// Rotate pair (x, y) = (x_i, x_{i+d/2}) by the angle with cosine/sine cs.
__device__ __forceinline__ float2 rotate_pair(float x, float y, float2 cs) {
  return make_float2(x * cs.x - y * cs.y, y * cs.x + x * cs.y);
}

// Product of two rotations: angle(a) + angle(b).
__device__ __forceinline__ float2 compose(float2 a, float2 b) {
  return make_float2(a.x * b.x - a.y * b.y, a.y * b.x + a.x * b.y);
}

}  // namespace jl
