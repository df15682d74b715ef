// Correctly rounded RoPE operands: bf16(R_n x) for the exact rotation.
//
// The tensor cores take the rotated Q and K in bf16, so every rotated
// element is rounded once.  That rounding is a discrete decision; an fp32
// rotation with fp32 cos/sin (error ~1e-7 relative) lands on the other side
// of a bf16 rounding midpoint for ~1e-4 of the elements, and on a peaked
// softmax one such flip in the dominant key moves the row's log-sum-exp by
// ~3e-3.  Here the rounding is that of the exact value:
//
//   * cos/sin of n * omega_i come as double-float pairs (hi + lo, ~48 bits)
//     from the product of three table rotations R_{a 2^20} R_{b 2^10} R_c
//     (n = a 2^20 + b 2^10 + c < 2^30), built per call in fp64 with the
//     angle reduced in double-double (build_rope_tables in rope_prepass.cu);
//   * each element first takes the plain fp32 value v = x c - y s; only
//     when v lies within its error bound of a bf16 rounding midpoint (about
//     5e-4 of the elements) is it recomputed in double-float arithmetic and
//     rounded by the sign of the remainder.
//
// Double-float arithmetic: Dekker/Knuth error-free transformations
// (two_prod by FMA, two_sum) on fp32 pairs.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

namespace jl {

struct DF {
  float hi, lo;
};

__device__ __forceinline__ DF two_prod(float a, float b) {
  const float p = a * b;
  return {p, fmaf(a, b, -p)};
}
__device__ __forceinline__ DF two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  return {s, (a - (s - bb)) + (b - bb)};
}
__device__ __forceinline__ DF df_norm(float hi, float lo) {
  const float s = hi + lo;
  return {s, lo - (s - hi)};
}
__device__ __forceinline__ DF df_mul(DF a, DF b) {
  DF p = two_prod(a.hi, b.hi);
  p.lo = fmaf(a.hi, b.lo, fmaf(a.lo, b.hi, p.lo));
  return df_norm(p.hi, p.lo);
}
__device__ __forceinline__ DF df_add(DF a, DF b) {
  DF s = two_sum(a.hi, b.hi);
  s.lo += a.lo + b.lo;
  return two_sum(s.hi, s.lo);  // s.hi may have cancelled below s.lo
}
__device__ __forceinline__ DF df_neg(DF a) { return {-a.hi, -a.lo}; }

// A rotation as double-float (cos, sin).
struct DFRot {
  DF c, s;
};
__device__ __forceinline__ DFRot df_compose(DFRot a, DFRot b) {
  return {df_add(df_mul(a.c, b.c), df_neg(df_mul(a.s, b.s))), df_add(df_mul(a.s, b.c), df_mul(a.c, b.s))};
}

// x c - y s for bf16-exact x, y and double-float c, s, as a double-float.
__device__ __forceinline__ DF df_rot(float x, float y, DF c, DF s) {
  const DF p1 = two_prod(x, c.hi), p2 = two_prod(y, s.hi);
  DF d = two_sum(p1.hi, -p2.hi);
  d.lo += (p1.lo - p2.lo) + fmaf(x, c.lo, -y * s.lo);
  return two_sum(d.hi, d.lo);  // d.hi may have cancelled below d.lo
}

// bf16 bits of the exact value represented by the double-float v (|v.lo|
// below half an fp32 ulp of v.hi): round v.hi to nearest even unless v.hi
// is exactly a bf16 midpoint, where the remainder decides.
__device__ __forceinline__ uint16_t round_df_bf16(DF v) {
  const uint32_t b = __float_as_uint(v.hi);
  if ((b & 0xffffu) == 0x8000u && v.lo != 0.f) {
    const uint32_t trunc = b >> 16;  // magnitude rounded down
    const bool up = (v.lo > 0.f) == (v.hi > 0.f);  // remainder moves the magnitude up
    return static_cast<uint16_t>(up ? trunc + 1 : trunc);
  }
  return __bfloat16_as_ushort(__float2bfloat16_rn(v.hi));
}

// bf16 bits of x c - y s (the exact rotation, correctly rounded).
__device__ __forceinline__ uint16_t rot_bf16(float x, float y, DF c, DF s) {
  const float v = fmaf(x, c.hi, -(y * s.hi));
  // |v - exact| <= 2^-24 (|y s| + |v| + |x c.lo| + |y s.lo|) <= 3 * 2^-24 (|x| + |y|)
  // with |c|, |s| <= 1 and |v| <= |x| + |y|; the test uses 2^-21 (|x| + |y|).
  // Only the midpoint of v's own bf16 interval can lie that close while
  // that interval is wider than 2^-12 (|x| + |y|), i.e. |v| >= 2^-9 (|x| + |y|);
  // smaller |v| (a cancelling rotation) always takes the exact path.
  const float xy = fabsf(x) + fabsf(y);
  const float bound = 4.76837158203125e-7f * xy;
  const uint32_t b = __float_as_uint(v);
  const float mid = __uint_as_float((b & 0xffff0000u) | 0x8000u);
  if (fabsf(v - mid) > bound && fabsf(v) >= 1.953125e-3f * xy)
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  return round_df_bf16(df_rot(x, y, c, s));
}

}  // namespace jl
