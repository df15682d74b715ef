// Decode: one new query token against an absolute-position KV cache.
//
// Paper digest page, "Method", "KV cache invariant": the cache keeps keys
// rotated at their absolute position j and is never rewritten when G grows;
// a remote key is corrected on the fly by the rotation R_{Delta_k},
// Delta_k = f(j) - j, because R_a R_b = R_{a+b} turns R_j x_j into
// R_{f(j)} x_j, while the query is rotated at f(q) (Delta_q = f(q) - q).
//
// Work split.  The key range [0, L) is cut into `nsplit` contiguous slices
// (whole 64-key blocks), one CTA each; a CTA covers all KV heads of its slice
// (warp w <-> KV head w), so per-key rotation tables are built once and
// shared by all heads.  Each CTA writes an unnormalised partial (running max
// m, sum l, sum p v) per query head; a second kernel merges the slices with
// log-sum-exp weights.
//
// Memory path.  Each warp streams its head's K and V rows (256 B each per
// key) through its own 3-stage shared-memory ring with 16-byte cp.async
// copies (16 lanes per row: fully coalesced), so the bytes in flight do not
// depend on registers; keys past the slice end are zero-filled.
//
// Rotation accuracy.  Delta(j) reaches ~1e5, so its angle is reduced in
// double precision once per CTA (first block); later blocks step the base
// by R_{-n} with 0 <= n <= 64 from a per-CTA table, and within a block
// key j0 + t uses base(j0) * R_{-n(t)}.  The R_{-n} table is built from
// accurately reduced powers of two, R_{-2^b}, with the frequency split in
// two floats so that 2^b * omega_hi is exact.
//
// Lane layout.  A warp takes 8 keys per step: half-warp `half` (lane >> 4)
// holds keys of parity `half`, lane m = lane & 15 holds head-dim elements
// 4m..4m+3 and 64+4m..64+4m+3 (the rotate-half partners); the 16-lane
// partial dot products are summed with a transpose-reduction.
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>

#include "internal.h"
#include "positions.cuh"
#include "rope_math.cuh"

namespace jl {
namespace {

constexpr int kD = 128;
constexpr int kBlockKeys = 64;  // keys per rotation-table block
constexpr int kStep = 8;        // keys per warp step
constexpr int kSlots = kStep / 2;
constexpr int kStages = 3;      // per-warp ring depth
constexpr int kMaxSplits = 512;
constexpr int kStageBytes = kStep * 2 * kD * 2;  // K and V rows of one step

struct DecodeKParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kc;
  const __nv_bfloat16* vc;
  float* part_o;   // [nsplit, B, Hq, 128]
  float* part_ml;  // [nsplit, B, Hq, 2]
  int B, L, Lcap, Hq, Hkv, w0, G, keys_per_split;
  float scale_log2;
  RopeFreqs freqs;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void unpack4(uint2 u, float (&f)[4]) {
  f[0] = __uint_as_float(u.x << 16);
  f[1] = __uint_as_float(u.x & 0xffff0000u);
  f[2] = __uint_as_float(u.y << 16);
  f[3] = __uint_as_float(u.y & 0xffff0000u);
}

// Sum v[0..3] over the 16 lanes of a half-warp; on return lane m holds the
// full sum of slot (m >> 2).
__device__ __forceinline__ float transpose_reduce4(const float (&v)[4], int m) {
  const bool u3 = m & 8, u2 = m & 4;
  float a[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = u3 ? v[i] : v[i + 2];
    const float keep = u3 ? v[i + 2] : v[i];
    a[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  const float send = u2 ? a[0] : a[1];
  const float keep = u2 ? a[1] : a[0];
  float c = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  c += __shfl_xor_sync(0xffffffffu, c, 2);
  c += __shfl_xor_sync(0xffffffffu, c, 1);
  return c;
}

template <int GQ>
__global__ void __launch_bounds__(256, 1)
decode_partial_kernel(DecodeKParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* s_qa = reinterpret_cast<float*>(smem_raw);              // [Hq][128], pre-scaled
  float* s_qr = s_qa + p.Hq * kD;                                // [Hq][128]
  float2* s_offs = reinterpret_cast<float2*>(s_qr + p.Hq * kD);  // [65][64]: R_{-n}
  float2* s_cs = s_offs + (kBlockKeys + 1) * 64;                 // [64][64]: this block
  float2* s_base = s_cs + kBlockKeys * 64;                       // [64]
  float2* s_pow = s_base + 64;                                   // [7][64]: R_{-2^b}
  unsigned char* s_ring = reinterpret_cast<unsigned char*>(s_pow + 7 * 64);  // [warps][stages]
  __shared__ float2 s_qcs[2][64];

  const int tid = threadIdx.x, nthr = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int half = lane >> 4, m = lane & 15;
  const int b = blockIdx.y, split = blockIdx.x;
  const int js = split * p.keys_per_split;
  const int je = min(p.L, js + p.keys_per_split);
  const int qpos = p.L - 1;
  const bool bifocal = p.G > 1;
  const int first_local = qpos - p.w0;  // keys j >= first_local are local

  const int hk = warp;
  const bool active = hk < p.Hkv;
  const long long row_stride = static_cast<long long>(p.Hkv) * kD;
  const __nv_bfloat16* kbase = p.kc + (static_cast<long long>(b) * p.Lcap * p.Hkv + hk) * kD;
  const __nv_bfloat16* vbase = p.vc + (static_cast<long long>(b) * p.Lcap * p.Hkv + hk) * kD;
  const uint32_t ring = static_cast<uint32_t>(__cvta_generic_to_shared(s_ring)) +
                        static_cast<uint32_t>(warp * kStages * kStageBytes);
  const int nsteps = (je - js + kStep - 1) / kStep;

  // Stage layout: K rows of the step's 8 keys (256 B each), then V rows.
  auto issue_step = [&](int it) {
    if (active && it < nsteps) {
      const int jstep = js + it * kStep;
      const uint32_t st = ring + static_cast<uint32_t>((it % kStages) * kStageBytes);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int idx = i * 32 + lane;  // 256 chunks of 16 B
        const int tensor = idx >> 7, key = (idx >> 4) & 7, c = idx & 15;
        const int j = jstep + key;
        const bool ok = j < je;
        const __nv_bfloat16* src =
            (tensor ? vbase : kbase) + (ok ? static_cast<long long>(j) * row_stride : 0) + c * 8;
        cp_async16(st + static_cast<uint32_t>(idx * 16), src, ok ? 16 : 0);
      }
    }
    cp_async_commit();
  };
  // Start the stream before the set-up work below.
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) issue_step(s);

  // Query rotations: R_{L-1} x_q and R_{f(L-1)} x_q, times scale * log2(e).
  for (int i = tid; i < 64; i += nthr) {
    s_qcs[0][i] = rope_cos_sin(qpos, p.freqs.w[i]);
    s_qcs[1][i] = rope_cos_sin(alias(qpos, p.G), p.freqs.w[i]);
  }
  const bool any_remote = bifocal && js < first_local;
  if (any_remote) {
    // R_{-2^b}, b = 0..6, from the frequency split omega = hi + lo with hi
    // holding 17 significant bits (so 2^b * hi is exact in float).
    for (int idx = tid; idx < 7 * 64; idx += nthr) {
      const int bb = idx / 64, i = idx % 64;
      const double w = p.freqs.w[i];
      const float whi = __uint_as_float(__float_as_uint(static_cast<float>(w)) & 0xffffff80u);
      const float wlo = static_cast<float>(w - static_cast<double>(whi));
      const float n = static_cast<float>(1 << bb);
      float sn, cn;
      sincosf(n * whi, &sn, &cn);
      const float e = n * wlo;  // |e| < 1e-3: second-order small-angle rotation
      const float2 r = compose(make_float2(cn, sn), make_float2(1.f - 0.5f * e * e, e));
      s_pow[idx] = make_float2(r.x, -r.y);  // R_{-2^b}
    }
    for (int i = tid; i < 64; i += nthr) s_offs[i] = make_float2(1.f, 0.f);
    __syncthreads();
    // R_{-n} = R_{-(n - 2^b)} R_{-2^b}, b = top bit of n, built layer by layer.
    for (int bb = 0; bb < 7; ++bb) {
      const int lo = 1 << bb, cnt = min(lo, kBlockKeys + 1 - lo);
      for (int idx = tid; idx < cnt * 64; idx += nthr) {
        const int n = lo + idx / 64, i = idx % 64;
        s_offs[n * 64 + i] = compose(s_offs[(n - lo) * 64 + i], s_pow[bb * 64 + i]);
      }
      __syncthreads();
    }
    for (int i = tid; i < 64; i += nthr) s_base[i] = rope_cos_sin(alias_offset(js, p.G), p.freqs.w[i]);
  }
  __syncthreads();
  const __nv_bfloat16* qin = p.q + static_cast<long long>(b) * p.Hq * kD;
  for (int idx = tid; idx < p.Hq * 64; idx += nthr) {
    const int h = idx / 64, i = idx % 64;
    const float x = __bfloat162float(qin[h * kD + i]);
    const float y = __bfloat162float(qin[h * kD + 64 + i]);
    const float2 ra = rotate_pair(x, y, s_qcs[0][i]);
    const float2 rr = rotate_pair(x, y, s_qcs[1][i]);
    s_qa[h * kD + i] = ra.x * p.scale_log2;
    s_qa[h * kD + 64 + i] = ra.y * p.scale_log2;
    s_qr[h * kD + i] = rr.x * p.scale_log2;
    s_qr[h * kD + 64 + i] = rr.y * p.scale_log2;
  }
  __syncthreads();

  float o[GQ][8];
  float m_run[GQ], l_part[GQ];
#pragma unroll
  for (int h = 0; h < GQ; ++h) {
    m_run[h] = -INFINITY;
    l_part[h] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[h][e] = 0.f;
  }

  for (int it = 0; it < nsteps; ++it) {
    const int jstep = js + it * kStep;
    const int j0 = js + (it / (kBlockKeys / kStep)) * kBlockKeys;  // block base
    if ((it % (kBlockKeys / kStep)) == 0 && bifocal && j0 < first_local) {
      // Rotation table of this 64-key block: cs[t] = base(j0) R_{-n(t)}.
      __syncthreads();
      if (j0 != js) {
        const int jp = j0 - kBlockKeys;  // advance the base from the previous block
        const int n = alias_offset(jp, p.G) - alias_offset(j0, p.G);
        for (int i = tid; i < 64; i += nthr) s_base[i] = compose(s_base[i], s_offs[n * 64 + i]);
      }
      __syncthreads();
      const int fj0 = alias(j0, p.G);
      for (int idx = tid; idx < kBlockKeys * 64; idx += nthr) {
        const int t = idx / 64, i = idx % 64;
        const int n = t - (alias(j0 + t, p.G) - fj0);
        s_cs[idx] = compose(s_base[i], s_offs[n * 64 + i]);
      }
      __syncthreads();
    }
    issue_step(it + kStages - 1);
    cp_async_wait<kStages - 1>();
    __syncwarp();
    if (!active) continue;

    const unsigned char* st = s_ring + (warp * kStages + it % kStages) * kStageBytes;
    const bool all_local = !bifocal || jstep >= first_local;
    const bool all_remote = bifocal && jstep + kStep - 1 < first_local;
    float z[GQ];
    auto scores = [&](const float* qs, bool rot, float (&out)[GQ]) {
      float sc[GQ][kSlots];
      float qlo[GQ][4], qhi[GQ][4];
#pragma unroll
      for (int h = 0; h < GQ; ++h) {
        const float4 a = *reinterpret_cast<const float4*>(qs + (hk * GQ + h) * kD + 4 * m);
        const float4 c = *reinterpret_cast<const float4*>(qs + (hk * GQ + h) * kD + 64 + 4 * m);
        qlo[h][0] = a.x; qlo[h][1] = a.y; qlo[h][2] = a.z; qlo[h][3] = a.w;
        qhi[h][0] = c.x; qhi[h][1] = c.y; qhi[h][2] = c.z; qhi[h][3] = c.w;
      }
#pragma unroll
      for (int s = 0; s < kSlots; ++s) {
        const int key = 2 * s + half;
        const uint2 klo = *reinterpret_cast<const uint2*>(st + key * 256 + 8 * m);
        const uint2 khi = *reinterpret_cast<const uint2*>(st + key * 256 + 128 + 8 * m);
        float x[4], y[4];
        unpack4(klo, x);
        unpack4(khi, y);
        if (rot) {
          const int t = (jstep - j0) + key;
          const float4 c01 = *reinterpret_cast<const float4*>(s_cs + t * 64 + 4 * m);
          const float4 c23 = *reinterpret_cast<const float4*>(s_cs + t * 64 + 4 * m + 2);
          const float2 cs[4] = {make_float2(c01.x, c01.y), make_float2(c01.z, c01.w),
                                make_float2(c23.x, c23.y), make_float2(c23.z, c23.w)};
#pragma unroll
          for (int f = 0; f < 4; ++f) {
            const float2 r = rotate_pair(x[f], y[f], cs[f]);
            x[f] = r.x;
            y[f] = r.y;
          }
        }
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
          float acc = 0.f;
#pragma unroll
          for (int f = 0; f < 4; ++f) acc = fmaf(qlo[h][f], x[f], fmaf(qhi[h][f], y[f], acc));
          sc[h][s] = acc;
        }
      }
#pragma unroll
      for (int h = 0; h < GQ; ++h) out[h] = transpose_reduce4(sc[h], m);
    };
    if (all_local) {
      scores(s_qa, false, z);
    } else if (all_remote) {
      scores(s_qr, true, z);
    } else {
      float zr[GQ];
      scores(s_qa, false, z);
      scores(s_qr, true, zr);
      const int j = jstep + 2 * (m >> 2) + half;
#pragma unroll
      for (int h = 0; h < GQ; ++h)
        if (j < first_local) z[h] = zr[h];
    }
    const int jmine = jstep + 2 * (m >> 2) + half;
    const bool valid = jmine < je;
    float pr[GQ];
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
      const float zz = valid ? z[h] : -INFINITY;
      float bm = zz;
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
      const float m_new = fmaxf(m_run[h], bm);
      const float alpha = exp2f(m_run[h] - m_new);
      m_run[h] = m_new;
      pr[h] = exp2f(zz - m_new);
      l_part[h] = l_part[h] * alpha + ((m & 3) ? 0.f : pr[h]);
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int e = 0; e < 8; ++e) o[h][e] *= alpha;
      }
    }
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
      const int key = 2 * s + half;
      const uint2 vlo = *reinterpret_cast<const uint2*>(st + (kStep + key) * 256 + 8 * m);
      const uint2 vhi = *reinterpret_cast<const uint2*>(st + (kStep + key) * 256 + 128 + 8 * m);
      float x[4], y[4];
      unpack4(vlo, x);
      unpack4(vhi, y);
#pragma unroll
      for (int h = 0; h < GQ; ++h) {
        const float ps = __shfl_sync(0xffffffffu, pr[h], half * 16 + 4 * s);
#pragma unroll
        for (int f = 0; f < 4; ++f) {
          o[h][f] = fmaf(ps, x[f], o[h][f]);
          o[h][4 + f] = fmaf(ps, y[f], o[h][4 + f]);
        }
      }
    }
    __syncwarp();  // the stage is refilled by the next issue_step
  }
  cp_async_wait<0>();

  if (!active) return;
  // Combine the two key parities and the 16-lane partial sums.
#pragma unroll
  for (int h = 0; h < GQ; ++h) {
#pragma unroll
    for (int e = 0; e < 8; ++e) o[h][e] += __shfl_xor_sync(0xffffffffu, o[h][e], 16);
    float l = l_part[h];
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    const int hq = hk * GQ + h;
    const long long slot = (static_cast<long long>(split) * p.B + b) * p.Hq + hq;
    if (half == 0) {
      float* dst = p.part_o + slot * kD;
      *reinterpret_cast<float4*>(dst + 4 * m) = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
      *reinterpret_cast<float4*>(dst + 64 + 4 * m) = make_float4(o[h][4], o[h][5], o[h][6], o[h][7]);
    }
    if (lane == 0) {
      p.part_ml[slot * 2] = m_run[h];
      p.part_ml[slot * 2 + 1] = l;
    }
  }
}

// Merge the per-slice partials of one (batch, query head): log-sum-exp
// weights exp2(m_s - M), output sum_s w_s o_s / sum_s w_s l_s.
__global__ void __launch_bounds__(128)
decode_merge_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                    int nsplit, int BH, __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  const int bh = blockIdx.x, e = threadIdx.x;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, part_ml[(static_cast<long long>(s) * BH + bh) * 2]);
  float num = 0.f, den = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const long long slot = static_cast<long long>(s) * BH + bh;
    const float w = exp2f(part_ml[slot * 2] - M);
    den = fmaf(w, part_ml[slot * 2 + 1], den);
    num = fmaf(w, part_o[slot * kD + e], num);
  }
  out[static_cast<long long>(bh) * kD + e] = __float2bfloat16_rn(num / den);
  if (lse != nullptr && e == 0) lse[bh] = (M + log2f(den)) * 0.69314718055994531f;
}

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  }
  return n;
}

}  // namespace

int decode_max_splits() { return kMaxSplits; }

size_t decode_workspace_bytes(int B, int Hq, int d, int Lcap) {
  (void)Lcap;
  return static_cast<size_t>(kMaxSplits) * B * Hq * (d + 2) * sizeof(float);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.d != kD) return cudaErrorInvalidValue;
  const int GQ = a.Hq / a.Hkv;
  const int nblocks = (a.L + kBlockKeys - 1) / kBlockKeys;
  const int target = std::min(num_sms(), kMaxSplits);
  const int bps = (nblocks + target - 1) / target;
  const int nsplit = (nblocks + bps - 1) / bps;

  DecodeKParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.kc = static_cast<const __nv_bfloat16*>(a.k_cache);
  p.vc = static_cast<const __nv_bfloat16*>(a.v_cache);
  p.part_o = a.part;
  p.part_ml = a.part + static_cast<size_t>(kMaxSplits) * a.B * a.Hq * kD;
  p.B = a.B; p.L = a.L; p.Lcap = a.Lcap; p.Hq = a.Hq; p.Hkv = a.Hkv;
  p.w0 = a.w0; p.G = a.G; p.keys_per_split = bps * kBlockKeys;
  p.scale_log2 = a.scale_log2;
  p.freqs = a.freqs;

  const int warps = std::max(a.Hkv, 1);
  const size_t smem = static_cast<size_t>(2) * a.Hq * kD * sizeof(float) +
                      static_cast<size_t>((kBlockKeys + 1) * 64 + kBlockKeys * 64 + 64 + 7 * 64) *
                          sizeof(float2) +
                      static_cast<size_t>(warps) * kStages * kStageBytes;
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  const dim3 grid(nsplit, a.B);
  cudaError_t err = cudaSuccess;
#define JL_DECODE_CASE(GQV)                                                                      \
  case GQV:                                                                                      \
    err = cudaFuncSetAttribute(decode_partial_kernel<GQV>,                                       \
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);          \
    if (err != cudaSuccess) return err;                                                          \
    decode_partial_kernel<GQV><<<grid, 32 * warps, smem, stream>>>(p);                           \
    break;
  switch (GQ) {
    JL_DECODE_CASE(1)
    JL_DECODE_CASE(2)
    JL_DECODE_CASE(4)
    JL_DECODE_CASE(8)
    default:
      return cudaErrorInvalidValue;
  }
#undef JL_DECODE_CASE
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  decode_merge_kernel<<<a.B * a.Hq, kD, 0, stream>>>(p.part_o, p.part_ml, nsplit, a.B * a.Hq,
                                                     static_cast<__nv_bfloat16*>(a.o), a.lse);
  return cudaGetLastError();
}

}  // namespace jl
