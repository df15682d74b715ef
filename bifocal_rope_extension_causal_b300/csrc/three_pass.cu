// Inclusion-exclusion merge of the three-pass form of bifocal attention.
//
// Paper digest page, "Method", Eq. 7: the bifocal attention of a query row is
// assembled from three ordinary causal attention passes over the same keys,
//   A  local window (0 <= q - k <= w0) at absolute rotations,
//   B  every causal key at aliased rotations,
//   C  local window at aliased rotations,
// whose unnormalised sums combine as A + B - C: B - C is the remote part at
// aliased rotations and A replaces the local part.  With each pass reduced to
// its normalised output o_X and log-sum-exp l_X,
//   o = (e^{l_A} o_A + e^{l_B} o_B - e^{l_C} o_C) / (e^{l_A} + e^{l_B} - e^{l_C}),
//   l = log(e^{l_A} + e^{l_B} - e^{l_C}),
// evaluated with the exponents shifted by M = max(l_A, l_B) (l_C <= l_B, since
// C scores a subset of B's pairs with the same values).
//
// The kernel is one streaming pass over the three outputs (HBM-bound): 16
// threads per (b, q, h) row of d = 128 (8 for d = 64), 16 bytes per thread per
// tensor, in place on o (which holds o_B on entry).
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"

namespace jl {
namespace {

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&x)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__global__ void __launch_bounds__(256)
three_pass_merge_kernel(const __nv_bfloat16* __restrict__ o_a, const float* __restrict__ lse_a,
                        __nv_bfloat16* o, const float* __restrict__ lse_b,
                        const __nv_bfloat16* __restrict__ o_c, const float* __restrict__ lse_c,
                        float* __restrict__ lse_out, long long rows, int L, int Hq, int d) {
  const int per_row = d / 8;  // threads per row
  const long long gt = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long row = gt / per_row;  // (b * L + q) * Hq + h
  const int part = static_cast<int>(gt - row * per_row);
  if (row >= rows) return;
  const int h = static_cast<int>(row % Hq);
  const long long bq = row / Hq;
  const int q = static_cast<int>(bq % L);
  const long long b = bq / L;
  const long long li = (b * Hq + h) * L + q;
  const float la = lse_a[li], lb = lse_b[li], lc = lse_c[li];
  const float M = fmaxf(la, lb);
  const float wa = expf(la - M), wb = expf(lb - M), wc = expf(lc - M);
  const float den = wa + wb - wc;
  const float inv = 1.f / den;
  const long long off = row * d + part * 8;
  float xa[8], xb[8], xc[8];
  load8(o_a + off, xa);
  load8(o + off, xb);
  load8(o_c + off, xc);
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float y0 = (wa * xa[2 * i] + wb * xb[2 * i] - wc * xc[2 * i]) * inv;
    const float y1 = (wa * xa[2 * i + 1] + wb * xb[2 * i + 1] - wc * xc[2 * i + 1]) * inv;
    const __nv_bfloat162 p2 = __floats2bfloat162_rn(y0, y1);
    w[i] = *reinterpret_cast<const uint32_t*>(&p2);
  }
  *reinterpret_cast<uint4*>(o + off) = make_uint4(w[0], w[1], w[2], w[3]);
  if (lse_out != nullptr && part == 0) lse_out[li] = M + logf(den);
}

}  // namespace

cudaError_t launch_three_pass_merge(const void* o_a, const float* lse_a, void* o, const float* lse_b,
                                    const void* o_c, const float* lse_c, float* lse_out, int B, int L,
                                    int Hq, int d, cudaStream_t stream) {
  if (d != 64 && d != 128) return cudaErrorInvalidValue;
  const long long rows = static_cast<long long>(B) * L * Hq;
  const long long threads = rows * (d / 8);
  if (threads == 0) return cudaSuccess;
  const long long blocks = (threads + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  three_pass_merge_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(o_a), lse_a, static_cast<__nv_bfloat16*>(o), lse_b,
      static_cast<const __nv_bfloat16*>(o_c), lse_c, lse_out, rows, L, Hq, d);
  return cudaGetLastError();
}

}  // namespace jl
