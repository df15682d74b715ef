// RoPE pre-pass: rotate raw Q or K once, at absolute and at aliased positions,
// and the correction pass that turns cached absolute-position keys into
// aliased-position keys.
//
// The bifocal score (paper digest page, "Method", Eq. 1) needs every query
// and key rotated twice: R_p x at the absolute position p for local pairs and
// R_f(p) x at the aliased position f(p) = floor(p / G) for remote pairs.  The
// rotations depend only on the row, so they are done once here (O(L * H * d)
// work) instead of once per score tile, into head-major [B, H, L, d] layouts
// in which one attention tile is one contiguous block.  For keys that are
// already in a KV cache (rotated at their absolute position k), the aliased
// rotation is reached by the correction R_{f(k) - k} ("KV cache invariant",
// R_a R_b = R_{a+b}) without touching the cache.
//
// Every output element is the exact rotation rounded to bf16 (exact_rope.cuh):
// cos/sin come from three per-call tables of double-float rotations,
// R_n = R_{a 2^20} R_{b 2^10} R_c, built by rope_table_kernel in fp64.
//
// Thread layout: a thread owns frequency pair i0 = 2 * threadIdx.x (and
// i0 + 1) of one position and loops over the heads, so the rotation of a
// (position, frequency) is composed once and reused by every head.  Loads
// and stores are 4-byte bf16x2, contiguous across the threads of a row.
#include <cuda_bf16.h>

#include "exact_rope.cuh"
#include "internal.h"
#include "positions.cuh"
#include "rope_math.cuh"

namespace jl {
namespace {

struct View {
  __nv_bfloat16* base;
  long long sb, sh, sr;
};
View as_view(const TensorView& t) {
  return {static_cast<__nv_bfloat16*>(const_cast<void*>(t.base)), t.sb, t.sh, t.sr};
}

__device__ __forceinline__ void store_bits(const View& v, int b, int h, int p, int i0, int half, uint32_t xs,
                                           uint32_t ys) {
  __nv_bfloat16* row = v.base + b * v.sb + h * v.sh + static_cast<long long>(p) * v.sr;
  *reinterpret_cast<uint32_t*>(row + i0) = xs;
  *reinterpret_cast<uint32_t*>(row + half + i0) = ys;
}

// Table entry of level l (0, 1, 2), index j < 1024, frequency i:
// R_{j 2^(10 l)} as float4 {cos hi, cos lo, sin hi, sin lo}.
__global__ void __launch_bounds__(256)
rope_table_kernel(float4* __restrict__ tab, int half, RopeFreqs freqs) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= kRopeTableRows * half) return;
  const int i = idx % half, row = idx / half;
  const int level = row / 1024, j = row % 1024;
  const double n = ldexp(static_cast<double>(j), 10 * level);  // exact
  const double w = freqs.w[i];
  // n * w = p + e exactly, reduced modulo 2 pi (split in two doubles).
  const double p = n * w;
  const double e = fma(n, w, -p);
  const double k = rint(p * kInvTwoPi);
  double r = fma(-k, kTwoPiHi, p);
  r = fma(-k, kTwoPiLo, r) + e;
  double sn, cs;
  sincos(r, &sn, &cs);
  const float ch = static_cast<float>(cs), sh = static_cast<float>(sn);
  tab[idx] = make_float4(ch, static_cast<float>(cs - ch), sh, static_cast<float>(sn - sh));
}

__device__ __forceinline__ DFRot table_rot(const float4* tab, int half, int row, int i) {
  const float4 t = tab[row * half + i];
  return {{t.x, t.y}, {t.z, t.w}};
}

// R_n for 0 <= n < 2^30 as a double-float rotation.
__device__ __forceinline__ DFRot rope_rot(const float4* tab, int half, int n, int i) {
  DFRot r = table_rot(tab, half, n & 1023, i);
  if (n >= 1024) r = df_compose(r, table_rot(tab, half, 1024 + ((n >> 10) & 1023), i));
  if (n >= (1 << 20)) r = df_compose(r, table_rot(tab, half, 2048 + (n >> 20), i));
  return r;
}

// bf16x2 words of (x0, x1) and (y0, y1) rotated by r0, r1 (pair i0, i0 + 1).
__device__ __forceinline__ void rotate_words(float2 xs, float2 ys, const DFRot& r0, const DFRot& r1, uint32_t& wx,
                                             uint32_t& wy) {
  const uint32_t a0 = rot_bf16(xs.x, ys.x, r0.c, r0.s), a1 = rot_bf16(xs.y, ys.y, r1.c, r1.s);
  const uint32_t b0 = rot_bf16(ys.x, -xs.x, r0.c, r0.s), b1 = rot_bf16(ys.y, -xs.y, r1.c, r1.s);
  wx = a0 | (a1 << 16);
  wy = b0 | (b1 << 16);
}

template <int D>
__global__ void __launch_bounds__(256)
rope_prepass_kernel(const __nv_bfloat16* __restrict__ x, int B, int C, int H, int G, int pos0,
                    const float4* __restrict__ tab, View out_abs, View out_rem, View out_cache) {
  constexpr int kHalf = D / 2;
  const int i0 = 2 * threadIdx.x;  // frequency pair (i0, i0 + 1)
  const long long row = static_cast<long long>(blockIdx.x) * blockDim.y + threadIdx.y;  // b*C + p
  if (row >= static_cast<long long>(B) * C) return;
  const int b = static_cast<int>(row / C);
  const int p = static_cast<int>(row - static_cast<long long>(b) * C);
  const int pos = pos0 + p;

  const DFRot ra0 = rope_rot(tab, kHalf, pos, i0), ra1 = rope_rot(tab, kHalf, pos, i0 + 1);
  DFRot rr0 = ra0, rr1 = ra1;
  const bool rem = out_rem.base != nullptr;
  if (rem) {
    const int fp = alias(pos, G);
    rr0 = rope_rot(tab, kHalf, fp, i0);
    rr1 = rope_rot(tab, kHalf, fp, i0 + 1);
  }
  for (int h = 0; h < H; ++h) {
    const __nv_bfloat16* src = x + (row * H + h) * D;
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + i0));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + kHalf + i0));
    uint32_t wx, wy;
    rotate_words(lo, hi, ra0, ra1, wx, wy);
    if (out_abs.base != nullptr) store_bits(out_abs, b, h, p, i0, kHalf, wx, wy);
    if (out_cache.base != nullptr) store_bits(out_cache, b, h, p, i0, kHalf, wx, wy);
    if (rem) {
      rotate_words(lo, hi, rr0, rr1, wx, wy);
      store_bits(out_rem, b, h, p, i0, kHalf, wx, wy);
    }
  }
}

// rem[b, h, k] = R_{f(k) - k} cache[b, k, h] for k < P0.
template <int D>
__global__ void __launch_bounds__(256)
rope_correct_kernel(const __nv_bfloat16* __restrict__ cache, int B, int P0, int Lcap, int H, int G,
                    const float4* __restrict__ tab, View out_rem) {
  constexpr int kHalf = D / 2;
  const int i0 = 2 * threadIdx.x;
  const long long row = static_cast<long long>(blockIdx.x) * blockDim.y + threadIdx.y;  // b*P0 + k
  if (row >= static_cast<long long>(B) * P0) return;
  const int b = static_cast<int>(row / P0);
  const int k = static_cast<int>(row - static_cast<long long>(b) * P0);
  const int m = -alias_offset(k, G);  // R_{f(k) - k} = R_{-m}: cos as R_m, sin negated
  DFRot r0 = rope_rot(tab, kHalf, m, i0), r1 = rope_rot(tab, kHalf, m, i0 + 1);
  r0.s = df_neg(r0.s);
  r1.s = df_neg(r1.s);
  for (int h = 0; h < H; ++h) {
    const __nv_bfloat16* src = cache + ((static_cast<long long>(b) * Lcap + k) * H + h) * D;
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + i0));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + kHalf + i0));
    uint32_t wx, wy;
    rotate_words(lo, hi, r0, r1, wx, wy);
    store_bits(out_rem, b, h, k, i0, kHalf, wx, wy);
  }
}

}  // namespace

cudaError_t launch_rope_tables(void* tables, int d, const RopeFreqs& freqs, cudaStream_t stream) {
  if (d != 64 && d != 128) return cudaErrorInvalidValue;
  const int n = kRopeTableRows * (d / 2);
  rope_table_kernel<<<(n + 255) / 256, 256, 0, stream>>>(static_cast<float4*>(tables), d / 2, freqs);
  return cudaGetLastError();
}

cudaError_t launch_rope_prepass(const void* x, int B, int C, int H, int d, int G, int pos0,
                                const void* tables, TensorView abs, TensorView rem,
                                TensorView cache, cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * C;
  if (rows == 0) return cudaSuccess;
  const auto* xin = static_cast<const __nv_bfloat16*>(x);
  const auto* tab = static_cast<const float4*>(tables);
  if (d == 128) {
    const dim3 block(32, 8), grid(static_cast<unsigned>((rows + 7) / 8));
    rope_prepass_kernel<128><<<grid, block, 0, stream>>>(xin, B, C, H, G, pos0, tab, as_view(abs),
                                                          as_view(rem), as_view(cache));
  } else if (d == 64) {
    const dim3 block(16, 16), grid(static_cast<unsigned>((rows + 15) / 16));
    rope_prepass_kernel<64><<<grid, block, 0, stream>>>(xin, B, C, H, G, pos0, tab, as_view(abs),
                                                         as_view(rem), as_view(cache));
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_rope_correct(const void* k_cache, int B, int P0, int Lcap, int H, int d, int G,
                                const void* tables, TensorView rem, cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * P0;
  if (rows == 0) return cudaSuccess;
  const auto* kc = static_cast<const __nv_bfloat16*>(k_cache);
  const auto* tab = static_cast<const float4*>(tables);
  if (d == 128) {
    const dim3 block(32, 8), grid(static_cast<unsigned>((rows + 7) / 8));
    rope_correct_kernel<128><<<grid, block, 0, stream>>>(kc, B, P0, Lcap, H, G, tab, as_view(rem));
  } else if (d == 64) {
    const dim3 block(16, 16), grid(static_cast<unsigned>((rows + 15) / 16));
    rope_correct_kernel<64><<<grid, block, 0, stream>>>(kc, B, P0, Lcap, H, G, tab, as_view(rem));
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace jl
