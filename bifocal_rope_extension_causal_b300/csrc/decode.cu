// Decode: one new query token against an absolute-position KV cache.
//
// Paper digest page, "Method", "KV cache invariant": the cache keeps keys
// rotated at their absolute position j and is never rewritten when G grows;
// a remote key is corrected on the fly by the rotation R_{Delta_k},
// Delta_k = f(j) - j, because R_a R_b = R_{a+b} turns R_j x_j into
// R_{f(j)} x_j, while the query is rotated at f(q) (Delta_q = f(q) - q).
//
// Work split.  The key range [0, L) is cut into `nsplit` contiguous slices
// (whole 64-key blocks), one CTA each, about one per SM; a CTA covers all KV
// heads of its slice (warp w <-> KV head w), so the per-key rotation tables
// are built once and shared by all heads.  Each CTA writes an unnormalised
// partial (running max m, sum l, sum p v) per query head; a second kernel,
// launched as a programmatic dependent of the first, merges the slices with
// log-sum-exp weights.
//
// Memory path.  kWarpsPerHead warps per KV head take alternate 8-key steps;
// each streams its head's K and V rows (256 B each per key) through its own
// kStages-deep shared-memory ring with 16-byte cp.async copies (16 lanes per
// row: fully coalesced; keys past the slice end are zero-filled).
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
// 4m..4m+3 and 64+4m..64+4m+3 (the rotate-half partners).  Rotation, dot
// products and the P V update use packed two-wide fp32 FMAs.  The 16-lane
// partial dot products of the step's GQ x 4 (head, key) scores are summed
// with one transpose-reduction that leaves each sum in one lane, and the
// softmax runs once per (head, key) through a small per-warp exchange
// buffer in shared memory.
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
constexpr int kStages = 2;      // per-warp ring depth
constexpr int kWarpsPerHead = 2;  // warps sharing a KV head (alternate steps)
constexpr int kMaxSplits = 512;
constexpr int kStageBytes = kStep * 2 * kD * 2;  // K and V rows of one step
constexpr float kRescaleThreshold = 8.0f;        // log2 units

// Per-warp exchange buffer (z[GQ][8], p[8][GQ], alpha[GQ]) in floats, padded
// to 16 bytes so that the cp.async ring after it stays 16-byte aligned.
__host__ __device__ constexpr int exchange_floats(int gq) { return (17 * gq + 3) / 4 * 4; }

struct DecodeKParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kc;
  const __nv_bfloat16* vc;
  float* part_o;   // [nsplit, B, Hq, 128]
  float* part_ml;  // [nsplit, B, Hq, 2]
  int* status;     // device status word
  const int* seqlens;  // per-sequence lengths [B] (device) or nullptr: every sequence has length L
  int B, L, Lcap, Hq, Hkv, w0, G, wp, keys_per_split;
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

// Four bf16 (two 32-bit words) to two float pairs.
__device__ __forceinline__ void unpack4(uint2 u, float2& a, float2& b) {
  a = make_float2(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u));
  b = make_float2(__uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

__device__ __forceinline__ float2 neg2(float2 a) { return make_float2(-a.x, -a.y); }

// Sum the V values of every lane over the 16 lanes of a half-warp.  On
// return lane m holds kOut = max(1, V / 16) full sums v[0..kOut), which are
// the original indices (m / kDup) * kOut + k, kDup = max(1, 16 / V).
template <int V>
__device__ __forceinline__ void transpose_reduce(float (&v)[V], int m) {
  int n = V;
#pragma unroll
  for (int b = 3; b >= 0; --b) {
    const int sh = 1 << b;
    if (n > 1) {
      const bool up = (m >> b) & 1;
      const int hf = n / 2;
#pragma unroll
      for (int k = 0; k < V / 2; ++k) {
        if (k < hf) {
          const float send = up ? v[k] : v[k + hf];
          const float keep = up ? v[k + hf] : v[k];
          v[k] = keep + __shfl_xor_sync(0xffffffffu, send, sh);
        }
      }
      n = hf;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], sh);
    }
  }
}

template <int GQ>
__global__ void __launch_bounds__(512, 1)
decode_partial_kernel(DecodeKParams p) {
  constexpr int kV = GQ * kSlots;                 // scores per half-warp per step
  constexpr int kOut = kV >= 16 ? kV / 16 : 1;    // sums held per lane after the reduction
  constexpr int kDup = kV >= 16 ? 1 : 16 / kV;    // lanes holding the same sum
  constexpr int kOwn = (GQ * 8 + 31) / 32;        // (head, key) pairs per lane in the softmax
  constexpr int kBlockSteps = kBlockKeys / kStep;  // global steps per table block (8)
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int nwarps = blockDim.x >> 5;
  float* s_qa = reinterpret_cast<float*>(smem_raw);                 // [Hq][128], pre-scaled
  float* s_qr = s_qa + p.Hq * kD;                                   // [Hq][128]
  float* s_c = s_qr + p.Hq * kD;                                    // [64 keys][64] cos
  float* s_s = s_c + kBlockKeys * 64;                               // [64 keys][64] sin
  float2* s_lo = reinterpret_cast<float2*>(s_s + kBlockKeys * 64);  // [8][64]: R_{-b}
  float2* s_hi = s_lo + 8 * 64;                                     // [9][64]: R_{-8a}
  float2* s_base = s_hi + 9 * 64;                                   // [64]
  float* s_x = reinterpret_cast<float*>(s_base + 64);               // per-warp exchange buffers
  unsigned char* s_ring = reinterpret_cast<unsigned char*>(s_x + nwarps * exchange_floats(GQ));
  __shared__ float2 s_qcs[2][64];

  // Let the merge kernel (a programmatic dependent) launch early; it waits
  // for this grid's completion before reading the partials.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

  const int tid = threadIdx.x, nthr = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int half = lane >> 4, m = lane & 15;
  const int b = blockIdx.y, split = blockIdx.x;
  // This sequence's length (the new token is at position L - 1) and group
  // size; per-sequence lengths outside [1, Lcap] are clamped and flagged.
  int L = p.L, G = p.G;
  if (p.seqlens != nullptr) {
    L = p.seqlens[b];
    if (L < 1 || L > p.Lcap) {
      if (threadIdx.x == 0 && split == 0) atomicCAS(p.status, 0, 30);
      L = min(max(L, 1), p.Lcap);
    }
    G = static_cast<int>(group_size(L, p.wp));
  }
  const int js = split * p.keys_per_split;
  const int je = max(js, min(L, js + p.keys_per_split));  // empty slice past the sequence end
  const int qpos = L - 1;
  const bool bifocal = G > 1;
  const int first_local = qpos - p.w0;  // keys j >= first_local are local

  // kWarpsPerHead warps per KV head: warp `par` of a head takes the global
  // steps it = kWarpsPerHead * u + par.
  const int hk = warp % p.Hkv, par = warp / p.Hkv;
  const long long row_stride = static_cast<long long>(p.Hkv) * kD;
  const __nv_bfloat16* kbase = p.kc + (static_cast<long long>(b) * p.Lcap * p.Hkv + hk) * kD;
  const __nv_bfloat16* vbase = p.vc + (static_cast<long long>(b) * p.Lcap * p.Hkv + hk) * kD;
  unsigned char* my_ring = s_ring + warp * kStages * kStageBytes;
  const uint32_t ring = static_cast<uint32_t>(__cvta_generic_to_shared(my_ring));
  float* xz = s_x + warp * exchange_floats(GQ);  // z[GQ][8]
  float* xp = xz + 8 * GQ;                       // p[8][GQ]
  float* xa = xp + 8 * GQ;                       // alpha[GQ]
  const int nsteps = (je - js + kStep - 1) / kStep;
  const int nlocal = (nsteps + kWarpsPerHead - 1) / kWarpsPerHead;  // local steps (warp 0 of a head)

  // Stage layout: K rows of the step's 8 keys (256 B each), then V rows.
  auto issue_step = [&](int u) {
    const int it = kWarpsPerHead * u + par;
    if (it < nsteps) {
      const int jstep = js + it * kStep;
      const uint32_t st = ring + static_cast<uint32_t>((u % kStages) * kStageBytes);
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
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) issue_step(s);

  // Query rotations R_{L-1} and R_{f(L-1)}, and the small rotation tables.
  for (int i = tid; i < 64; i += nthr) {
    s_qcs[0][i] = rope_cos_sin(qpos, p.freqs.w[i]);
    s_qcs[1][i] = rope_cos_sin(alias(qpos, G), p.freqs.w[i]);
  }
  const bool any_remote = bifocal && js < first_local;
  if (any_remote) {
    // R_{-b} (b < 8) and R_{-8a} (a <= 8) with omega = hi + lo, hi holding
    // 17 significant bits so that n * hi is exact in float for n <= 64.
    for (int idx = tid; idx < 17 * 64; idx += nthr) {
      const int r = idx / 64, i = idx % 64;
      const int n = r < 8 ? r : 8 * (r - 8);
      const double w = p.freqs.w[i];
      const float whi = __uint_as_float(__float_as_uint(static_cast<float>(w)) & 0xffffff80u);
      const float wlo = static_cast<float>(w - static_cast<double>(whi));
      float sn, cn;
      sincosf(static_cast<float>(n) * whi, &sn, &cn);
      const float e = static_cast<float>(n) * wlo;  // |e| < 1e-3
      const float2 rr = compose(make_float2(cn, sn), make_float2(1.f - 0.5f * e * e, e));
      (r < 8 ? s_lo : s_hi)[(r < 8 ? r : r - 8) * 64 + i] = make_float2(rr.x, -rr.y);  // R_{-n}
    }
    for (int i = tid; i < 64; i += nthr) s_base[i] = rope_cos_sin(alias_offset(js, G), p.freqs.w[i]);
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
  // (The first table build below starts with a barrier.)

  float2 o[GQ][4];
#pragma unroll
  for (int h = 0; h < GQ; ++h)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[h][e] = make_float2(0.f, 0.f);
  float m_run[kOwn], l_run[kOwn];
#pragma unroll
  for (int k = 0; k < kOwn; ++k) {
    m_run[k] = -INFINITY;
    l_run[k] = 0.f;
  }

  constexpr int kBlockLocal = kBlockSteps / kWarpsPerHead;  // local steps per table block
  for (int u = 0; u < nlocal; ++u) {
    const int it = kWarpsPerHead * u + par;
    const int blk = u / kBlockLocal;
    const int j0 = js + blk * kBlockKeys;  // table block base
    if ((u % kBlockLocal) == 0) {
      __syncthreads();  // previous table no longer read; q (first pass) written
      if (bifocal && j0 < first_local) {
        if (blk > 0) {
          const int n = alias_offset(j0 - kBlockKeys, G) - alias_offset(j0, G);  // 0..64
          for (int i = tid; i < 64; i += nthr)
            s_base[i] = compose(compose(s_base[i], s_hi[(n >> 3) * 64 + i]), s_lo[(n & 7) * 64 + i]);
          __syncthreads();
        }
        const int fj0 = alias(j0, G);
        for (int idx = tid; idx < kBlockKeys * 64; idx += nthr) {
          const int t = idx / 64, i = idx % 64;
          const int n = t - (alias(j0 + t, G) - fj0);  // 0..63
          const float2 cs = compose(compose(s_base[i], s_hi[(n >> 3) * 64 + i]), s_lo[(n & 7) * 64 + i]);
          s_c[idx] = cs.x;
          s_s[idx] = cs.y;
        }
      }
      __syncthreads();
    }
    issue_step(u + kStages - 1);
    cp_async_wait<kStages - 1>();
    __syncwarp();
    if (it >= nsteps) continue;

    const int jstep = js + it * kStep;
    const unsigned char* st = my_ring + (u % kStages) * kStageBytes;
    const bool all_local = !bifocal || jstep >= first_local;
    const bool all_remote = bifocal && jstep + kStep - 1 < first_local;

    // Full scores of this step's keys; lane m ends with sums (m/kDup)*kOut+k
    // of the index h * 4 + s (key 2s + half).
    auto scores = [&](const float* qs, bool rot, float (&zout)[kOut]) {
      float sc[kV];
#pragma unroll
      for (int s = 0; s < kSlots; ++s) {
        const int key = 2 * s + half;
        float2 x01, x23, y01, y23;
        unpack4(*reinterpret_cast<const uint2*>(st + key * 256 + 8 * m), x01, x23);
        unpack4(*reinterpret_cast<const uint2*>(st + key * 256 + 128 + 8 * m), y01, y23);
        if (rot) {
          const int t = (jstep - j0) + key;
          const float4 c = *reinterpret_cast<const float4*>(s_c + t * 64 + 4 * m);
          const float4 sn = *reinterpret_cast<const float4*>(s_s + t * 64 + 4 * m);
          const float2 c01 = make_float2(c.x, c.y), c23 = make_float2(c.z, c.w);
          const float2 s01 = make_float2(sn.x, sn.y), s23 = make_float2(sn.z, sn.w);
          // (x, y) -> (x c - y s, y c + x s)
          const float2 nx01 = __ffma2_rn(y01, neg2(s01), __fmul2_rn(x01, c01));
          const float2 nx23 = __ffma2_rn(y23, neg2(s23), __fmul2_rn(x23, c23));
          y01 = __ffma2_rn(x01, s01, __fmul2_rn(y01, c01));
          y23 = __ffma2_rn(x23, s23, __fmul2_rn(y23, c23));
          x01 = nx01;
          x23 = nx23;
        }
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
          const float* qh = qs + (hk * GQ + h) * kD;
          const float4 a = *reinterpret_cast<const float4*>(qh + 4 * m);
          const float4 c = *reinterpret_cast<const float4*>(qh + 64 + 4 * m);
          float2 acc = __fmul2_rn(make_float2(a.x, a.y), x01);
          acc = __ffma2_rn(make_float2(a.z, a.w), x23, acc);
          acc = __ffma2_rn(make_float2(c.x, c.y), y01, acc);
          acc = __ffma2_rn(make_float2(c.z, c.w), y23, acc);
          sc[h * kSlots + s] = acc.x + acc.y;
        }
      }
      transpose_reduce<kV>(sc, m);
#pragma unroll
      for (int k = 0; k < kOut; ++k) zout[k] = sc[k];
    };

    float z[kOut];
    if (all_local) {
      scores(s_qa, false, z);
    } else if (all_remote) {
      scores(s_qr, true, z);
    } else {
      float zr[kOut];
      scores(s_qa, false, z);
      scores(s_qr, true, zr);
#pragma unroll
      for (int k = 0; k < kOut; ++k) {
        const int i = (m / kDup) * kOut + k;  // = h * 4 + s
        if (jstep + 2 * (i % kSlots) + half < first_local) z[k] = zr[k];
      }
    }
    // Publish the step's scores: xz[h][key].
#pragma unroll
    for (int k = 0; k < kOut; ++k) {
      const int i = (m / kDup) * kOut + k;
      xz[(i / kSlots) * 8 + 2 * (i % kSlots) + half] = z[k];
    }
    __syncwarp();
    // Online softmax, one lane per (head, key); a head's 8 keys are 8
    // consecutive lanes.  The max used for the exponentials is raised only
    // when it grows by more than kRescaleThreshold.
    bool any_rescale = false;
#pragma unroll
    for (int k = 0; k < kOwn; ++k) {
      const int idx = k * 32 + lane;
      const bool own = idx < GQ * 8;
      const int h = idx >> 3, key = idx & 7;
      const bool valid = own && (jstep + key < je);
      const float zz = valid ? xz[idx] : -INFINITY;
      float bm = zz;
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
      float alpha = 1.f;
      if (bm > m_run[k] + kRescaleThreshold) {
        alpha = exp2f(m_run[k] - bm);
        m_run[k] = bm;
      }
      const float mexp = m_run[k] == -INFINITY ? 0.f : m_run[k];
      const float pr = exp2f(zz - mexp);
      l_run[k] = l_run[k] * alpha + pr;
      if (own) {
        xp[key * GQ + h] = pr;
        if (key == 0) xa[h] = alpha;
      }
      any_rescale |= alpha != 1.f;
    }
    any_rescale = __any_sync(0xffffffffu, any_rescale);
    __syncwarp();
    if (any_rescale) {
#pragma unroll
      for (int h = 0; h < GQ; ++h) {
        const float a = xa[h];
        const float2 a2 = make_float2(a, a);
#pragma unroll
        for (int e = 0; e < 4; ++e) o[h][e] = __fmul2_rn(o[h][e], a2);
      }
    }
    // O += P V (keys past the slice end have p = 0 and zero-filled rows).
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
      const int key = 2 * s + half;
      float2 v01, v23, w01, w23;
      unpack4(*reinterpret_cast<const uint2*>(st + (kStep + key) * 256 + 8 * m), v01, v23);
      unpack4(*reinterpret_cast<const uint2*>(st + (kStep + key) * 256 + 128 + 8 * m), w01, w23);
      float pk[GQ];
      if constexpr (GQ % 4 == 0) {
#pragma unroll
        for (int h = 0; h < GQ; h += 4) {
          const float4 q4 = *reinterpret_cast<const float4*>(xp + key * GQ + h);
          pk[h] = q4.x;
          pk[h + 1] = q4.y;
          pk[h + 2] = q4.z;
          pk[h + 3] = q4.w;
        }
      } else {
#pragma unroll
        for (int h = 0; h < GQ; ++h) pk[h] = xp[key * GQ + h];
      }
#pragma unroll
      for (int h = 0; h < GQ; ++h) {
        const float2 p2 = make_float2(pk[h], pk[h]);
        o[h][0] = __ffma2_rn(p2, v01, o[h][0]);
        o[h][1] = __ffma2_rn(p2, v23, o[h][1]);
        o[h][2] = __ffma2_rn(p2, w01, o[h][2]);
        o[h][3] = __ffma2_rn(p2, w23, o[h][3]);
      }
    }
    __syncwarp();  // the stage and the exchange buffer are rewritten next step
  }
  cp_async_wait<0>();

  // Per-head statistics of this warp: m (shared by the head's 8 lanes) and
  // l summed over them; combine the two key parities of o within the warp.
  float mh[kOwn], lh[kOwn];
#pragma unroll
  for (int k = 0; k < kOwn; ++k) {
    float l = l_run[k];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    mh[k] = m_run[k];
    lh[k] = l;
  }
#pragma unroll
  for (int h = 0; h < GQ; ++h)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      o[h][e].x += __shfl_xor_sync(0xffffffffu, o[h][e].x, 16);
      o[h][e].y += __shfl_xor_sync(0xffffffffu, o[h][e].y, 16);
    }
  // With two warps per head, the second hands its state to the first
  // through its (now idle) ring: o [GQ][128] then (m, l) [GQ][2].
  float* hand = reinterpret_cast<float*>(my_ring);
  if constexpr (kWarpsPerHead == 2) __syncthreads();
  if (kWarpsPerHead == 2 && par == 1) {
    if (half == 0) {
#pragma unroll
      for (int h = 0; h < GQ; ++h) {
        *reinterpret_cast<float4*>(hand + h * kD + 4 * m) = make_float4(o[h][0].x, o[h][0].y, o[h][1].x, o[h][1].y);
        *reinterpret_cast<float4*>(hand + h * kD + 64 + 4 * m) =
            make_float4(o[h][2].x, o[h][2].y, o[h][3].x, o[h][3].y);
      }
    }
#pragma unroll
    for (int k = 0; k < kOwn; ++k) {
      const int idx = k * 32 + lane;
      if (idx < GQ * 8 && (idx & 7) == 0) {
        hand[GQ * kD + 2 * (idx >> 3)] = mh[k];
        hand[GQ * kD + 2 * (idx >> 3) + 1] = lh[k];
      }
    }
  }
  if constexpr (kWarpsPerHead == 2) __syncthreads();
  if (par != 0) return;
  const float* other = reinterpret_cast<const float*>(s_ring + (warp + p.Hkv) * kStages * kStageBytes);
  const bool paired = kWarpsPerHead == 2;
  // Merge state of head h: M = max(m0, m1), scales 2^(m0-M), 2^(m1-M).
#pragma unroll
  for (int h = 0; h < GQ; ++h) {
    const float m1 = paired ? other[GQ * kD + 2 * h] : -INFINITY;
    const float l1 = paired ? other[GQ * kD + 2 * h + 1] : 0.f;
    // This warp's m and l of head h live in lanes 8h..8h+7 of iteration h / 4.
    float m0 = 0.f, l0 = 0.f;
#pragma unroll
    for (int k = 0; k < kOwn; ++k) {
      const float mk = __shfl_sync(0xffffffffu, mh[k], (h * 8) & 31);
      const float lk = __shfl_sync(0xffffffffu, lh[k], (h * 8) & 31);
      if (k == (h * 8) / 32) {
        m0 = mk;
        l0 = lk;
      }
    }
    const float M = fmaxf(m0, m1);
    const float a0 = M == -INFINITY ? 0.f : exp2f(m0 - M);
    const float a1 = M == -INFINITY ? 0.f : exp2f(m1 - M);
    const int hq = hk * GQ + h;
    const long long slot = (static_cast<long long>(split) * p.B + b) * p.Hq + hq;
    if (half == 0) {
      const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 b0 = paired ? *reinterpret_cast<const float4*>(other + h * kD + 4 * m) : zero4;
      const float4 b1 = paired ? *reinterpret_cast<const float4*>(other + h * kD + 64 + 4 * m) : zero4;
      float* dst = p.part_o + slot * kD;
      *reinterpret_cast<float4*>(dst + 4 * m) =
          make_float4(a0 * o[h][0].x + a1 * b0.x, a0 * o[h][0].y + a1 * b0.y, a0 * o[h][1].x + a1 * b0.z,
                      a0 * o[h][1].y + a1 * b0.w);
      *reinterpret_cast<float4*>(dst + 64 + 4 * m) =
          make_float4(a0 * o[h][2].x + a1 * b1.x, a0 * o[h][2].y + a1 * b1.y, a0 * o[h][3].x + a1 * b1.z,
                      a0 * o[h][3].y + a1 * b1.w);
    }
    if (lane == 0) {
      p.part_ml[slot * 2] = M;
      p.part_ml[slot * 2 + 1] = a0 * l0 + a1 * l1;
    }
  }
}

// Merge the per-slice partials of one (batch, query head) with log-sum-exp
// weights: out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s, M = max m_s.
// One pass: each warp folds its slices (loaded four at a time, independent
// loads) into a running (max, sum, vector); the eight warps combine in
// shared memory.  A lane owns four output elements.
__global__ void __launch_bounds__(256)
decode_merge_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                    int nsplit, int BH, __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  __shared__ float s_m[8], s_l[8];
  __shared__ float4 s_acc[8][32];
  // The partials are written by the preceding grid.
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  const int bh = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float M = -INFINITY, Lsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = warp; s0 < nsplit; s0 += 32) {
    float ms[4], ls[4];
    float4 os[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int s = s0 + 8 * k;
      if (s < nsplit) {
        const long long slot = static_cast<long long>(s) * BH + bh;
        ms[k] = part_ml[slot * 2];
        ls[k] = part_ml[slot * 2 + 1];
        os[k] = *reinterpret_cast<const float4*>(part_o + slot * kD + 4 * lane);
      } else {
        ms[k] = -INFINITY;
        ls[k] = 0.f;
        os[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float Mn = fmaxf(M, ms[k]);
      if (Mn == -INFINITY) continue;
      const float a = exp2f(M - Mn), w = exp2f(ms[k] - Mn);
      Lsum = Lsum * a + ls[k] * w;
      acc.x = acc.x * a + os[k].x * w;
      acc.y = acc.y * a + os[k].y * w;
      acc.z = acc.z * a + os[k].z * w;
      acc.w = acc.w * a + os[k].w * w;
      M = Mn;
    }
  }
  s_acc[warp][lane] = acc;
  if (lane == 0) {
    s_m[warp] = M;
    s_l[warp] = Lsum;
  }
  __syncthreads();
  if (warp == 0) {
    float Mt = s_m[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) Mt = fmaxf(Mt, s_m[w]);
    float D = 0.f;
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const float a = s_m[w] == -INFINITY ? 0.f : exp2f(s_m[w] - Mt);
      D += a * s_l[w];
      const float4 v = s_acc[w][lane];
      t.x += a * v.x;
      t.y += a * v.y;
      t.z += a * v.z;
      t.w += a * v.w;
    }
    const float inv = 1.f / D;
    __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(out + static_cast<long long>(bh) * kD + 4 * lane);
    dst[0] = __floats2bfloat162_rn(t.x * inv, t.y * inv);
    dst[1] = __floats2bfloat162_rn(t.z * inv, t.w * inv);
    if (lse != nullptr && lane == 0) lse[bh] = (Mt + log2f(D)) * 0.69314718055994531f;
  }
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
  p.w0 = a.w0; p.G = a.G; p.wp = a.wp; p.keys_per_split = bps * kBlockKeys;
  p.seqlens = a.seqlens;
  p.status = device_status_ptr();
  if (p.status == nullptr) return cudaErrorInvalidSymbol;
  p.scale_log2 = a.scale_log2;
  p.freqs = a.freqs;

  const int warps = kWarpsPerHead * a.Hkv;
  const size_t smem = static_cast<size_t>(2) * a.Hq * kD * sizeof(float) +           // q
                      static_cast<size_t>(2) * kBlockKeys * 64 * sizeof(float) +     // cos, sin
                      static_cast<size_t>(8 + 9 + 1) * 64 * sizeof(float2) +         // R_-b, R_-8a, base
                      static_cast<size_t>(warps) * exchange_floats(GQ) * sizeof(float) +
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

  // The merge waits on the partial kernel through griddepcontrol.wait, so it
  // may be launched before that kernel finishes.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B * a.Hq);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_merge_kernel, static_cast<const float*>(p.part_o),
                            static_cast<const float*>(p.part_ml), nsplit, a.B * a.Hq,
                            static_cast<__nv_bfloat16*>(a.o), a.lse);
}

}  // namespace jl
