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
// Thread layout: a thread owns frequency pair i0 = 2 * threadIdx.x (and
// i0 + 1) of one position and loops over the heads, so the accurate angle
// (double-precision reduction, see rope_math.cuh) is computed once per
// (position, frequency) and reused by every head.  Loads and stores are
// 4-byte bf16x2, contiguous across the threads of a row.
#include <cuda_bf16.h>

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

__device__ __forceinline__ void store_pair(const View& v, int b, int h, int p, int i0, int half, float2 r0,
                                           float2 r1) {
  __nv_bfloat16* row = v.base + b * v.sb + h * v.sh + static_cast<long long>(p) * v.sr;
  *reinterpret_cast<__nv_bfloat162*>(row + i0) = __floats2bfloat162_rn(r0.x, r1.x);
  *reinterpret_cast<__nv_bfloat162*>(row + half + i0) = __floats2bfloat162_rn(r0.y, r1.y);
}

template <int D>
__global__ void __launch_bounds__(256)
rope_prepass_kernel(const __nv_bfloat16* __restrict__ x, int B, int C, int H, int G, int pos0,
                    RopeFreqs freqs, View out_abs, View out_rem, View out_cache) {
  constexpr int kHalf = D / 2;
  const int i0 = 2 * threadIdx.x;  // frequency pair (i0, i0 + 1)
  const long long row = static_cast<long long>(blockIdx.x) * blockDim.y + threadIdx.y;  // b*C + p
  if (row >= static_cast<long long>(B) * C) return;
  const int b = static_cast<int>(row / C);
  const int p = static_cast<int>(row - static_cast<long long>(b) * C);
  const int pos = pos0 + p;

  const float2 ca0 = rope_cos_sin(pos, freqs.w[i0]);
  const float2 ca1 = rope_cos_sin(pos, freqs.w[i0 + 1]);
  float2 cr0 = ca0, cr1 = ca1;
  const bool rem = out_rem.base != nullptr;
  if (rem) {
    const int fp = alias(pos, G);
    cr0 = rope_cos_sin(fp, freqs.w[i0]);
    cr1 = rope_cos_sin(fp, freqs.w[i0 + 1]);
  }
  for (int h = 0; h < H; ++h) {
    const __nv_bfloat16* src = x + (row * H + h) * D;
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + i0));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + kHalf + i0));
    const float2 a0 = rotate_pair(lo.x, hi.x, ca0), a1 = rotate_pair(lo.y, hi.y, ca1);
    if (out_abs.base != nullptr) store_pair(out_abs, b, h, p, i0, kHalf, a0, a1);
    if (out_cache.base != nullptr) store_pair(out_cache, b, h, p, i0, kHalf, a0, a1);
    if (rem) store_pair(out_rem, b, h, p, i0, kHalf, rotate_pair(lo.x, hi.x, cr0), rotate_pair(lo.y, hi.y, cr1));
  }
}

// rem[b, h, k] = R_{f(k) - k} cache[b, k, h] for k < P0.
template <int D>
__global__ void __launch_bounds__(256)
rope_correct_kernel(const __nv_bfloat16* __restrict__ cache, int B, int P0, int Lcap, int H, int G,
                    RopeFreqs freqs, View out_rem) {
  constexpr int kHalf = D / 2;
  const int i0 = 2 * threadIdx.x;
  const long long row = static_cast<long long>(blockIdx.x) * blockDim.y + threadIdx.y;  // b*P0 + k
  if (row >= static_cast<long long>(B) * P0) return;
  const int b = static_cast<int>(row / P0);
  const int k = static_cast<int>(row - static_cast<long long>(b) * P0);
  const int delta = alias_offset(k, G);
  const float2 c0 = rope_cos_sin(delta, freqs.w[i0]);
  const float2 c1 = rope_cos_sin(delta, freqs.w[i0 + 1]);
  for (int h = 0; h < H; ++h) {
    const __nv_bfloat16* src = cache + ((static_cast<long long>(b) * Lcap + k) * H + h) * D;
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + i0));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + kHalf + i0));
    store_pair(out_rem, b, h, k, i0, kHalf, rotate_pair(lo.x, hi.x, c0), rotate_pair(lo.y, hi.y, c1));
  }
}

}  // namespace

cudaError_t launch_rope_prepass(const void* x, int B, int C, int H, int d, int G, int pos0,
                                const RopeFreqs& freqs, TensorView abs, TensorView rem,
                                TensorView cache, cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * C;
  if (rows == 0) return cudaSuccess;
  const auto* xin = static_cast<const __nv_bfloat16*>(x);
  if (d == 128) {
    const dim3 block(32, 8), grid(static_cast<unsigned>((rows + 7) / 8));
    rope_prepass_kernel<128><<<grid, block, 0, stream>>>(xin, B, C, H, G, pos0, freqs, as_view(abs),
                                                          as_view(rem), as_view(cache));
  } else if (d == 64) {
    const dim3 block(16, 16), grid(static_cast<unsigned>((rows + 15) / 16));
    rope_prepass_kernel<64><<<grid, block, 0, stream>>>(xin, B, C, H, G, pos0, freqs, as_view(abs),
                                                         as_view(rem), as_view(cache));
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_rope_correct(const void* k_cache, int B, int P0, int Lcap, int H, int d, int G,
                                const RopeFreqs& freqs, TensorView rem, cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * P0;
  if (rows == 0) return cudaSuccess;
  const auto* kc = static_cast<const __nv_bfloat16*>(k_cache);
  if (d == 128) {
    const dim3 block(32, 8), grid(static_cast<unsigned>((rows + 7) / 8));
    rope_correct_kernel<128><<<grid, block, 0, stream>>>(kc, B, P0, Lcap, H, G, freqs, as_view(rem));
  } else if (d == 64) {
    const dim3 block(16, 16), grid(static_cast<unsigned>((rows + 15) / 16));
    rope_correct_kernel<64><<<grid, block, 0, stream>>>(kc, B, P0, Lcap, H, G, freqs, as_view(rem));
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace jl
