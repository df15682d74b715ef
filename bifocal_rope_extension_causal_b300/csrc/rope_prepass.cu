// RoPE pre-pass: rotate raw Q or K once, at absolute and at aliased positions.
//
// The bifocal score (paper digest page, "Method", Eq. 1) needs every query
// and key rotated twice: R_p x at the absolute position p for local pairs and
// R_f(p) x at the aliased position f(p) = floor(p / G) for remote pairs.  The
// rotations depend only on the row, so they are done once here (O(L * H * d)
// work) instead of once per score tile, and written in a head-major layout
// [B, H, L, d] in which one attention tile is one contiguous block.
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

template <int D>
__global__ void __launch_bounds__(256)
rope_prepass_kernel(const __nv_bfloat16* __restrict__ x, int B, int L, int H, int G,
                    RopeFreqs freqs, __nv_bfloat16* __restrict__ out_abs,
                    __nv_bfloat16* __restrict__ out_rem, __nv_bfloat16* __restrict__ out_cache) {
  constexpr int kHalf = D / 2;
  const int i0 = 2 * threadIdx.x;  // frequency pair (i0, i0 + 1)
  const long long row = static_cast<long long>(blockIdx.x) * blockDim.y + threadIdx.y;  // b*L + p
  if (row >= static_cast<long long>(B) * L) return;
  const int b = static_cast<int>(row / L);
  const int p = static_cast<int>(row - static_cast<long long>(b) * L);

  const float2 ca0 = rope_cos_sin(p, freqs.w[i0]);
  const float2 ca1 = rope_cos_sin(p, freqs.w[i0 + 1]);
  float2 cr0 = ca0, cr1 = ca1;
  const bool rem = out_rem != nullptr;
  if (rem) {
    const int fp = alias(p, G);
    cr0 = rope_cos_sin(fp, freqs.w[i0]);
    cr1 = rope_cos_sin(fp, freqs.w[i0 + 1]);
  }

  for (int h = 0; h < H; ++h) {
    const __nv_bfloat16* src = x + (row * H + h) * D;
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + i0));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + kHalf + i0));
    const long long dst = ((static_cast<long long>(b) * H + h) * L + p) * D;

    float2 r0 = rotate_pair(lo.x, hi.x, ca0);
    float2 r1 = rotate_pair(lo.y, hi.y, ca1);
    const __nv_bfloat162 a_lo = __floats2bfloat162_rn(r0.x, r1.x);
    const __nv_bfloat162 a_hi = __floats2bfloat162_rn(r0.y, r1.y);
    *reinterpret_cast<__nv_bfloat162*>(out_abs + dst + i0) = a_lo;
    *reinterpret_cast<__nv_bfloat162*>(out_abs + dst + kHalf + i0) = a_hi;
    if (out_cache != nullptr) {
      __nv_bfloat16* c = out_cache + (row * H + h) * D;
      *reinterpret_cast<__nv_bfloat162*>(c + i0) = a_lo;
      *reinterpret_cast<__nv_bfloat162*>(c + kHalf + i0) = a_hi;
    }
    if (rem) {
      r0 = rotate_pair(lo.x, hi.x, cr0);
      r1 = rotate_pair(lo.y, hi.y, cr1);
      *reinterpret_cast<__nv_bfloat162*>(out_rem + dst + i0) = __floats2bfloat162_rn(r0.x, r1.x);
      *reinterpret_cast<__nv_bfloat162*>(out_rem + dst + kHalf + i0) =
          __floats2bfloat162_rn(r0.y, r1.y);
    }
  }
}

}  // namespace

cudaError_t launch_rope_prepass(const void* x, int B, int L, int H, int d, int G,
                                const RopeFreqs& freqs, void* out_abs, void* out_rem,
                                void* out_cache, cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * L;
  const auto* xin = static_cast<const __nv_bfloat16*>(x);
  auto* oa = static_cast<__nv_bfloat16*>(out_abs);
  auto* orr = static_cast<__nv_bfloat16*>(out_rem);
  auto* oc = static_cast<__nv_bfloat16*>(out_cache);
  if (d == 128) {
    const dim3 block(32, 8);
    const dim3 grid(static_cast<unsigned>((rows + 7) / 8));
    rope_prepass_kernel<128><<<grid, block, 0, stream>>>(xin, B, L, H, G, freqs, oa, orr, oc);
  } else if (d == 64) {
    const dim3 block(16, 16);
    const dim3 grid(static_cast<unsigned>((rows + 15) / 16));
    rope_prepass_kernel<64><<<grid, block, 0, stream>>>(xin, B, L, H, G, freqs, oa, orr, oc);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace jl
