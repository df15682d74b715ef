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
// heads of its slice (two warps per KV head), so the per-key rotation table
// is built once and shared by all heads.  Each CTA writes an unnormalised
// partial (running max m, sum l, sum p v) per query head; a second kernel,
// launched as a programmatic dependent of the first, merges the slices with
// log-sum-exp weights.
//
// Memory path.  kWarpsPerHead warps per KV head take alternate 8-key steps;
// each streams its head's K and V rows (256 B each per key) through its own
// kStages-deep shared-memory ring with 16-byte cp.async copies (16 lanes per
// row: fully coalesced; keys past the slice end are zero-filled).  The
// 16-byte chunks of a row are XOR-swizzled by the key index so that the
// 8x8 ldmatrix tiles read below are free of bank conflicts.
//
// Arithmetic.  The per-key work runs on the tensor cores (warp-level
// mma.sync, bf16 operands, fp32 accumulation), which leaves the CUDA cores
// only the key rotation and the softmax; issue, not HBM, bounds the plain
// CUDA-core form of this loop.  Precision is kept at fp32 level by splitting
// every operand that is not already bf16 into bf16 hi + lo parts:
//   scores (m16n8k16)  A = the step's 8 keys, corrected by R_{Delta_k} in
//                      fp32 and split (rows 0..7 hi, rows 8..15 lo);
//                      B = the pre-scaled rotated query heads of the KV
//                      head as (hi, lo) column pairs.  The four products of
//                      a (key, head) land in one lane's accumulator.
//   O += P V (m16n8k8) computed as O^T += V^T P^T: A = V^T from transposed
//                      ldmatrix tiles, B = P split as hi + lo (with at most
//                      four query heads per KV head the lo parts fill the
//                      idle columns 4..7).
// The softmax runs in the score fragment (one lane per (key, head)) with
// lazily raised maxima.
//
// Rotation accuracy.  Delta(j) reaches ~1e5, so its angle is reduced in
// double precision once per CTA (first block); later blocks step the base
// by R_{-n} with 0 <= n <= 64 from a per-CTA table, and within a block
// key j0 + t uses base(j0) * R_{-n(t)}.  The R_{-n} table is built from
// R_{-b} and R_{-8a} with the frequency split in two floats so that
// n * omega_hi is exact.
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
constexpr int kStages = 2;      // per-warp ring depth
// Warps sharing a KV head (alternate steps): two while the query fragments
// of a head group fit the 128-register budget of a 512-thread CTA, one for
// eight query heads per KV head.
__host__ __device__ constexpr int warps_per_head(int gq) { return gq <= 4 ? 2 : 1; }
constexpr int kMaxSplits = 512;
constexpr int kMinBlocksPerSplit = 8;  // batched decode: blocks per slice when the batch fills the SMs
constexpr int kStageBytes = kStep * 2 * kD * 2;  // K and V rows of one step
constexpr float kRescaleThreshold = 8.0f;        // log2 units
constexpr int kTabStride = 36;  // float4 per key row of the rotation table (32 + 4 padding)

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

__device__ __forceinline__ float2 neg2(float2 a) { return make_float2(-a.x, -a.y); }

// ---- warp-level tensor-core primitives (bf16 in, fp32 accumulate) ----
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5}, {%6}, "
      "{%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0));
}
// Two floats to bf16x2 (x in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16(float x, float y) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}
// v = hi + lo with hi = bf16(v) and lo = bf16(v - hi): the pair carries
// about 16 significant bits of each element.
__device__ __forceinline__ void split_bf16(float2 v, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(v.x, v.y);
  const float2 r = __ffma2_rn(unpack_bf16(hi), make_float2(-1.f, -1.f), v);
  lo = pack_bf16(r.x, r.y);
}

template <int GQ>
__global__ void __launch_bounds__(warps_per_head(GQ) * 256, 1)
decode_partial_kernel(DecodeKParams p) {
  constexpr int kWarpsPerHead = warps_per_head(GQ);
  constexpr int kNT = (GQ + 3) / 4;                // score n-tiles: 4 heads x {hi, lo} each
  constexpr int kBlockSteps = kBlockKeys / kStep;  // global steps per table block (8)
  // P V columns: with GQ <= 4, column n holds head n & 3, its P hi part for
  // n < 4 and its lo part for n >= 4; with GQ = 8 column n is head n.
  constexpr bool kLoCols = GQ <= 4;
  auto hcol = [](int n) { return kLoCols ? (n & 3) : n; };
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // Region A: the rotated queries during set-up, then the rotation table of
  // the current 64-key block: [key][kTabStride] float4 {cos_i, cos_i+1,
  // sin_i, sin_i+1} for the frequency pair (i, i+1), i = 2 * index.
  float* s_qa = reinterpret_cast<float*>(smem_raw);  // [Hq][128], pre-scaled
  float* s_qr = s_qa + p.Hq * kD;                    // [Hq][128]
  const float4* s_tab = reinterpret_cast<const float4*>(smem_raw);
  float4* s_tab_w = reinterpret_cast<float4*>(smem_raw);
  const int region_a = max(2 * p.Hq * kD * 4, kBlockKeys * kTabStride * 16);
  float2* s_lo = reinterpret_cast<float2*>(smem_raw + region_a);  // [8][64]: R_{-b}
  float2* s_hi = s_lo + 8 * 64;                                   // [9][64]: R_{-8a}
  float2* s_base = s_hi + 9 * 64;                                 // [64]
  unsigned char* s_ring = reinterpret_cast<unsigned char*>(s_base + 64);
  __shared__ float2 s_qcs[2][64];

  // Let the merge kernel (a programmatic dependent) launch early; it waits
  // for this grid's completion before reading the partials.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

  const int tid = threadIdx.x, nthr = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;  // fragment row group / column pair
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
  const int nsteps = (je - js + kStep - 1) / kStep;
  const int nlocal = (nsteps + kWarpsPerHead - 1) / kWarpsPerHead;  // local steps (warp 0 of a head)

  // Stage layout: K rows of the step's 8 keys (256 B each), then V rows.
  // 16-byte chunk c of key row r sits at chunk c ^ (r & 7) of its row, so
  // that the eight rows of an 8x8 ldmatrix tile fall in eight bank groups.
  // Lane roles of the copies: chunk c = lane & 15 of key 2 i + (lane >> 4).
  const long long lane_src = static_cast<long long>(lane >> 4) * row_stride + (lane & 15) * 8;
  // Destination of copy i (key 2 i + (lane >> 4), swizzled chunk), relative to the stage.
  uint32_t lane_dst[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int key = 2 * i + (lane >> 4);
    lane_dst[i] = static_cast<uint32_t>((key * 16 + ((lane & 15) ^ key)) * 16);
  }
  auto issue_step = [&](int u) {
    const int it = kWarpsPerHead * u + par;
    if (it < nsteps) {
      const int jstep = js + it * kStep;
      const uint32_t st = ring + static_cast<uint32_t>((u % kStages) * kStageBytes);
      if (jstep + kStep <= je) {  // full step: no bounds checks
        const __nv_bfloat16* kp = kbase + lane_src + static_cast<long long>(jstep) * row_stride;
        const __nv_bfloat16* vp = vbase + lane_src + static_cast<long long>(jstep) * row_stride;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          cp_async16(st + lane_dst[i], kp + 2 * i * row_stride, 16);
          cp_async16(st + 2048 + lane_dst[i], vp + 2 * i * row_stride, 16);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const bool ok = jstep + 2 * i + (lane >> 4) < je;
          const long long off = ok ? lane_src + static_cast<long long>(jstep + 2 * i) * row_stride : 0;
          cp_async16(st + lane_dst[i], kbase + off, ok ? 16 : 0);
          cp_async16(st + 2048 + lane_dst[i], vbase + off, ok ? 16 : 0);
        }
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
  __syncthreads();
  // Query operands of the score MMA (B, 16 dims x 8 columns per chunk):
  // column n of n-tile nt is head 4 nt + n / 2, hi part (n even) or lo part
  // (n odd) of the pre-scaled rotated query; variant 0 absolute, 1 aliased.
  uint32_t qf[2][kNT][8][2];
#pragma unroll
  for (int v = 0; v < 2; ++v)
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      const int hl = 4 * nt + (g >> 1);
      const float* qrow = (v ? s_qr : s_qa) + (hk * GQ + (hl < GQ ? hl : 0)) * kD;
#pragma unroll
      for (int c = 0; c < 8; ++c)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          uint32_t hi, lo;
          split_bf16(*reinterpret_cast<const float2*>(qrow + 16 * c + 8 * e + 2 * t4), hi, lo);
          qf[v][nt][c][e] = hl < GQ ? ((g & 1) ? lo : hi) : 0u;
        }
    }
  // (The first table build below starts with a barrier, after which the
  // table may overwrite the rotated queries.)

  // O^T accumulators: m-tile mt holds dims 16 mt + g (+8) of heads 2 t4, 2 t4 + 1.
  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[mt][e] = 0.f;
  // Softmax state of head 4 nt + t4 (the same in the 8 lanes of a column).
  float m_run[kNT], l_run[kNT];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
    m_run[nt] = -INFINITY;
    l_run[nt] = 0.f;
  }
  // ldmatrix lane roles: lanes 8 mi .. 8 mi + 7 address rows 0..7 of tile mi.
  const int lm = lane >> 3, lr = lane & 7;

  constexpr int kBlockLocal = kBlockSteps / kWarpsPerHead;  // local steps per table block
  for (int u = 0; u < nlocal; ++u) {
    const int it = kWarpsPerHead * u + par;
    const int blk = u / kBlockLocal;
    const int j0 = js + blk * kBlockKeys;  // table block base
    if ((u % kBlockLocal) == 0) {
      __syncthreads();  // previous table (or the rotated queries) no longer read
      if (bifocal && j0 < first_local) {
        if (blk > 0) {
          const int n = alias_offset(j0 - kBlockKeys, G) - alias_offset(j0, G);  // 0..64
          for (int i = tid; i < 64; i += nthr)
            s_base[i] = compose(compose(s_base[i], s_hi[(n >> 3) * 64 + i]), s_lo[(n & 7) * 64 + i]);
          __syncthreads();
        }
        const int fj0 = alias(j0, G);
        for (int idx = tid; idx < kBlockKeys * 32; idx += nthr) {
          const int t = idx >> 5, pp = idx & 31, i0 = 2 * pp;
          const int n = t - (alias(j0 + t, G) - fj0);  // 0..63
          const float2 c0 =
              compose(compose(s_base[i0], s_hi[(n >> 3) * 64 + i0]), s_lo[(n & 7) * 64 + i0]);
          const float2 c1 = compose(compose(s_base[i0 + 1], s_hi[(n >> 3) * 64 + i0 + 1]),
                                    s_lo[(n & 7) * 64 + i0 + 1]);
          s_tab_w[t * kTabStride + pp] = make_float4(c0.x, c1.x, c0.y, c1.y);
        }
      }
      __syncthreads();
    }
    issue_step(u + kStages - 1);
    cp_async_wait<kStages - 1>();
    __syncwarp();
    if (it >= nsteps) continue;

    const int jstep = js + it * kStep;
    const uint32_t st = ring + static_cast<uint32_t>((u % kStages) * kStageBytes);
    const bool all_local = !bifocal || jstep >= first_local;
    const bool all_remote = bifocal && jstep + kStep - 1 < first_local;

    // Scores z[nt] of (key jstep + g, head 4 nt + t4) in log2 units.
    float z[kNT];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) z[nt] = 0.f;
    if (!all_local) {
      // Aliased scores.  A = the step's 8 keys corrected by R_{f(j) - j},
      // rows 0..7 their bf16 hi parts, rows 8..15 the lo parts; chunk c
      // (dims 16 c ..) and chunk c + 4 (the rotate-half partners) together.
      float acc0[kNT][4], acc1[kNT][4];
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc0[nt][e] = acc1[nt][e] = 0.f;
      const float4* tab = s_tab + (jstep - j0 + g) * kTabStride + t4;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r0, r1, r2, r3;
        const int ch = 2 * c + (lm & 1) + 8 * (lm >> 1);
        ldsm_x4(st + static_cast<uint32_t>(lr * 256 + ((ch ^ lr) << 4)), r0, r1, r2, r3);
        const float4 cs0 = tab[8 * c], cs1 = tab[8 * c + 4];
        const float2 x0 = unpack_bf16(r0), x1 = unpack_bf16(r1), y0 = unpack_bf16(r2), y1 = unpack_bf16(r3);
        const float2 c0 = make_float2(cs0.x, cs0.y), s0 = make_float2(cs0.z, cs0.w);
        const float2 c1 = make_float2(cs1.x, cs1.y), s1 = make_float2(cs1.z, cs1.w);
        // (x, y) -> (x c - y s, y c + x s)
        const float2 nx0 = __ffma2_rn(y0, neg2(s0), __fmul2_rn(x0, c0));
        const float2 ny0 = __ffma2_rn(x0, s0, __fmul2_rn(y0, c0));
        const float2 nx1 = __ffma2_rn(y1, neg2(s1), __fmul2_rn(x1, c1));
        const float2 ny1 = __ffma2_rn(x1, s1, __fmul2_rn(y1, c1));
        uint32_t x0h, x0l, x1h, x1l, y0h, y0l, y1h, y1l;
        split_bf16(nx0, x0h, x0l);
        split_bf16(nx1, x1h, x1l);
        split_bf16(ny0, y0h, y0l);
        split_bf16(ny1, y1h, y1l);
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          mma16816(acc0[nt], x0h, x0l, x1h, x1l, qf[1][nt][c][0], qf[1][nt][c][1]);
          mma16816(acc1[nt], y0h, y0l, y1h, y1l, qf[1][nt][c + 4][0], qf[1][nt][c + 4][1]);
        }
      }
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
        z[nt] = ((acc0[nt][0] + acc0[nt][1]) + (acc0[nt][2] + acc0[nt][3])) +
                ((acc1[nt][0] + acc1[nt][1]) + (acc1[nt][2] + acc1[nt][3]));
    }
    if (!all_remote) {
      // Absolute scores: the cached keys as stored (exact in bf16, lo rows 0).
      float acc0[kNT][4], acc1[kNT][4];
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc0[nt][e] = acc1[nt][e] = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r0, r1, r2, r3;
        const int ch = 2 * c + (lm & 1) + 8 * (lm >> 1);
        ldsm_x4(st + static_cast<uint32_t>(lr * 256 + ((ch ^ lr) << 4)), r0, r1, r2, r3);
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          mma16816(acc0[nt], r0, 0u, r1, 0u, qf[0][nt][c][0], qf[0][nt][c][1]);
          mma16816(acc1[nt], r2, 0u, r3, 0u, qf[0][nt][c + 4][0], qf[0][nt][c + 4][1]);
        }
      }
      const bool local = !bifocal || jstep + g >= first_local;
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        const float za = (acc0[nt][0] + acc0[nt][1]) + (acc1[nt][0] + acc1[nt][1]);
        if (all_local || local) z[nt] = za;
      }
    }

    // Online softmax per head (column); the max used for the exponentials
    // is raised only when it grows by more than kRescaleThreshold.
    bool any_rescale = false;
    float pr[kNT], al[kNT];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      const bool valid = jstep + g < je && 4 * nt + t4 < GQ;
      const float zz = valid ? z[nt] : -INFINITY;
      float bm = zz;
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
      float alpha = 1.f;
      if (bm > m_run[nt] + kRescaleThreshold) {
        alpha = exp2f(m_run[nt] - bm);
        m_run[nt] = bm;
      }
      const float mexp = m_run[nt] == -INFINITY ? 0.f : m_run[nt];
      pr[nt] = exp2f(zz - mexp);
      l_run[nt] = l_run[nt] * alpha + pr[nt];
      al[nt] = alpha;
      any_rescale |= alpha != 1.f;
    }
    any_rescale = __any_sync(0xffffffffu, any_rescale);
    if (any_rescale) {
      // Column n of O^T belongs to head hcol(n); its alpha sits in lane
      // hcol & 3 of n-tile hcol >> 2.
      float ae = 1.f, ao = 1.f;
      const int he = hcol(2 * t4), ho = hcol(2 * t4 + 1);
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        const float x = __shfl_sync(0xffffffffu, al[nt], he & 3);
        const float y = __shfl_sync(0xffffffffu, al[nt], ho & 3);
        if ((he >> 2) == nt) ae = x;
        if ((ho >> 2) == nt) ao = y;
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][0] *= ae;
        o[mt][1] *= ao;
        o[mt][2] *= ae;
        o[mt][3] *= ao;
      }
    }
    // P^T operand (B, 8 keys x 8 columns): keys 2 t4, 2 t4 + 1 of column g,
    // i.e. of head hcol(g), from lanes 4 key + (head & 3) of n-tile head >> 2.
    // P is split as hi + lo in bf16: with GQ <= 4 the lo parts fill columns
    // 4..7, otherwise they go through a second product.
    uint32_t pb_hi, pb_lo;
    {
      const int hh = hcol(g);
      const int src = 8 * t4 + (hh & 3);
      float p0 = 0.f, p1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        const float a = __shfl_sync(0xffffffffu, pr[nt], src);
        const float c = __shfl_sync(0xffffffffu, pr[nt], src + 4);
        if ((hh >> 2) == nt) {
          p0 = a;
          p1 = c;
        }
      }
      uint32_t hi, lo;
      split_bf16(make_float2(p0, p1), hi, lo);
      const bool use = hh < GQ;
      if constexpr (kLoCols) {
        pb_hi = use ? (g < 4 ? hi : lo) : 0u;
        pb_lo = 0u;
      } else {
        pb_hi = use ? hi : 0u;
        pb_lo = use ? lo : 0u;
      }
    }
    // O^T += V^T P^T: four transposed 8x8 loads of V give the A operands of
    // two 16-dim m-tiles each (keys past the slice end have p = 0 and
    // zero-filled rows).
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      uint32_t v0, v1, v2, v3;
      const int ch = 4 * jj + lm;
      ldsm_x4_t(st + static_cast<uint32_t>((kStep + lr) * 256 + ((ch ^ lr) << 4)), v0, v1, v2, v3);
      mma1688(o[2 * jj], v0, v1, pb_hi);
      mma1688(o[2 * jj + 1], v2, v3, pb_hi);
      if constexpr (!kLoCols) {
        mma1688(o[2 * jj], v0, v1, pb_lo);
        mma1688(o[2 * jj + 1], v2, v3, pb_lo);
      }
    }
    __syncwarp();  // the stage is rewritten next step
  }
  cp_async_wait<0>();

  // Per-head statistics of this warp: l summed over the 8 key lanes.
  float lh[kNT];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
    float l = l_run[nt];
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    lh[nt] = l;
  }
  // Each warp leaves its state in its (now idle) ring: o [GQ][128], then
  // (m, l) [GQ][2]; the CTA then merges the warps of each KV head.
  __syncthreads();
  float* hand = reinterpret_cast<float*>(my_ring);
  if constexpr (kLoCols) {
    // Column n + 4 (lane t4 + 2) holds the lo-part product of column n.
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mt][e] += __shfl_xor_sync(0xffffffffu, o[mt][e], 2);
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int d0 = 16 * mt + g;
    const int h0 = 2 * t4, h1 = 2 * t4 + 1;
    if (h0 < GQ) {
      hand[h0 * kD + d0] = o[mt][0];
      hand[h0 * kD + d0 + 8] = o[mt][2];
    }
    if (h1 < GQ) {
      hand[h1 * kD + d0] = o[mt][1];
      hand[h1 * kD + d0 + 8] = o[mt][3];
    }
  }
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
    const int h = 4 * nt + t4;
    if (g == 0 && h < GQ) {
      hand[GQ * kD + 2 * h] = m_run[nt];
      hand[GQ * kD + 2 * h + 1] = lh[nt];
    }
  }
  __syncthreads();
  // Merge: M = max over the head's warps, weights 2^(m_w - M).
  for (int idx = tid; idx < p.Hq * 32; idx += nthr) {
    const int hq = idx >> 5, d4 = idx & 31;
    const int kv = hq / GQ, h = hq % GQ;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarpsPerHead; ++w) {
      const float* src = reinterpret_cast<const float*>(s_ring + (kv + w * p.Hkv) * kStages * kStageBytes);
      M = fmaxf(M, src[GQ * kD + 2 * h]);
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kWarpsPerHead; ++w) {
      const float* src = reinterpret_cast<const float*>(s_ring + (kv + w * p.Hkv) * kStages * kStageBytes);
      const float mw = src[GQ * kD + 2 * h];
      const float a = M == -INFINITY ? 0.f : exp2f(mw - M);
      lsum += a * src[GQ * kD + 2 * h + 1];
      const float4 v = *reinterpret_cast<const float4*>(src + h * kD + 4 * d4);
      acc.x += a * v.x;
      acc.y += a * v.y;
      acc.z += a * v.z;
      acc.w += a * v.w;
    }
    const long long slot = (static_cast<long long>(split) * p.B + b) * p.Hq + hq;
    *reinterpret_cast<float4*>(p.part_o + slot * kD + 4 * d4) = acc;
    if (d4 == 0) {
      p.part_ml[slot * 2] = M;
      p.part_ml[slot * 2 + 1] = lsum;
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
  // Blocks per slice: enough slices for one wave over the SMs for one
  // sequence; with a batch, up to kMinBlocksPerSplit blocks per slice as long
  // as the batch's slices still fill a wave (short sequences would otherwise
  // pay the per-CTA set-up for a single 64-key block).
  const int nblocks = (a.L + kBlockKeys - 1) / kBlockKeys;
  const int target = std::min(num_sms(), kMaxSplits);
  const int fill = static_cast<int>(std::min<long long>(kMinBlocksPerSplit,
                                                         static_cast<long long>(nblocks) * a.B / num_sms()));
  const int bps = std::max((nblocks + target - 1) / target, fill);
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

  const int warps = warps_per_head(GQ) * a.Hkv;
  const size_t region_a = std::max(static_cast<size_t>(2) * a.Hq * kD * sizeof(float),    // q
                                    static_cast<size_t>(kBlockKeys) * kTabStride * 16);     // rotation table
  const size_t smem = region_a + static_cast<size_t>(8 + 9 + 1) * 64 * sizeof(float2) +   // R_-b, R_-8a, base
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
