// Decode: one new query token against an absolute-position KV cache.
//
// Paper digest page, "Method", "KV cache invariant": the cache keeps keys
// rotated at their absolute position j and is never rewritten when G grows;
// a remote key is corrected on the fly by the rotation R_{Delta_k},
// Delta_k = f(j) - j, because R_a R_b = R_{a+b} turns R_j x_j into
// R_{f(j)} x_j, while the query is rotated at f(q) (Delta_q = f(q) - q).
//
// Work split.  The key range [0, L) is cut into `nsplit` contiguous slices of
// whole 16-key steps, one CTA each and about one per SM.  Steps that hold
// remote keys (a prefix of [0, L)) cost more than all-local steps (they
// take the correction rotation), so the slices are balanced by cost: the
// first n_r slices share the remote steps evenly and the rest share the
// local ones.  A CTA covers up to eight KV heads of its slice (more KV
// heads take more CTAs along grid z), so the per-key rotation table is built
// once and shared by all of its heads.  Each CTA writes an unnormalised
// partial (running max m, sum l, sum p v) per query head; a second kernel,
// launched as a programmatic dependent of the first, merges the slices with
// log-sum-exp weights.
//
// Memory path.  One warp per KV head (more when a CTA holds fewer than
// eight heads, taking alternate steps) streams the head's K and V rows (2d
// bytes each per key) through its own two-stage shared-memory ring with
// 16-byte cp.async copies (fully coalesced; keys past the slice end are
// zero-filled).  The query rows and both ring stages are requested before
// any set-up work, so the set-up runs while the first keys are in flight.
// The 16-byte chunks of a row are XOR-swizzled by the key index so that the
// 8x8 ldmatrix tiles read below are free of bank conflicts.
//
// Arithmetic.  A step is 16 keys of one KV head.  The per-key work runs on
// the tensor cores (warp-level mma.sync m16n8k16, bf16 operands, fp32
// accumulation), which leaves the CUDA cores only the key rotation and the
// softmax.  Precision is kept at fp32 level by splitting every operand that
// is not already bf16 into bf16 hi + lo parts:
//   scores   A = the step's 16 keys, corrected by R_{Delta_k} in fp32 and
//            split: one product with the hi parts, one with the lo parts;
//            B = the pre-scaled rotated query heads of the KV head as
//            (hi, lo) column pairs.  The four products of a (key, head) land
//            in one lane's accumulator.  Local keys are exact in bf16 and
//            take one product.
//   O += P V computed as O^T += V^T P^T: A = V^T from transposed ldmatrix
//            tiles (16 dims x 16 keys), B = P split as hi + lo (with at most
//            four query heads per KV head the lo parts fill the idle columns
//            4..7; otherwise a second product).
// The softmax runs in the score fragment (each lane holds two keys of one
// head) with lazily raised maxima.
//
// Correction rotations.  Keys are grouped in 64-key table blocks from the
// slice start j0 = js + 64 b.  Within a block, key j0 + t needs
// R_{Delta(j0+t)} = R_{Delta(j0)} R_{-n(t)}, n(t) = t - (f(j0+t) - f(j0)) in
// [0, 63], and R_{-n} = R_{-8a} R_{-c} (n = 8a + c) comes from two small
// per-CTA tables.  The block base R_{Delta(j0)} is reduced accurately (float
// arithmetic on host-reduced angle tables, no fp64) once per CTA and then
// stepped block to block by R_{-n64},
// n64 = 64 - (f(j0+64) - f(j0)).  Each thread owns one frequency pair of the
// table and keeps that pair's base in registers.  The tables of two blocks
// are double-buffered: while the warps stream block b they build block b+1's
// table, a few entries per step, so one CTA barrier per block suffices.
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>

#include "internal.h"
#include "positions.cuh"
#include "rope_math.cuh"

namespace jl {
namespace {

constexpr int kBlockKeys = 64;  // keys per rotation-table block
constexpr int kStep = 16;       // keys per warp step
constexpr int kStages = 2;      // per-warp ring depth
constexpr int kMaxHeadsPerCta = 8;
constexpr int kMaxWarps = 8;
constexpr int kMaxSplits = 512;
constexpr int kMinStepsPerSplit = 32;  // batched decode: steps per slice when the batch fills the SMs
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr double kRemoteCost = 1.6;        // cost of a step with remote keys / an all-local step
constexpr int kSmallRows = 17;             // R_{-c} (c < 8), then R_{-8a} (a <= 8)

struct DecodeKParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kc;
  const __nv_bfloat16* vc;
  float* part_o;   // [slices, B, Hq, D]
  float* part_ml;  // [slices, B, Hq, 2]
  int* status;     // device status word
  const int* seqlens;  // per-sequence lengths [B] (device) or nullptr: every sequence has length L
  int B, L, Lcap, Hq, Hkv, gq, hpc, wph, w0, G, wp;
  // Slices s < split_r share steps [0, steps_r) evenly, the others share
  // [steps_r, steps_all); with per-sequence lengths, steps past a
  // sequence's end are empty.
  int steps_r, steps_all, split_r;
  float scale_log2;
  AngleTable ang;
};

// 2 pi as three floats: P1 keeps 13 significant bits, so that k * P1 is
// exact for |k| <= 1024.
constexpr float kTwoPiP1 = 6.283203125f;
constexpr float kTwoPiP2 = -1.781781975296326e-05f;
constexpr float kTwoPiP3 = -6.605598229861287e-13f;
constexpr float kInvTwoPiF = 0.15915494309189535f;

// cos and sin of n * omega_i for |n| < 2^30 in float arithmetic only (the
// fp64 pipe is slow on this GPU).  With n = d2 2^20 + d1 2^10 + d0 (10-bit
// digits), n omega = sum_l d_l phi_l mod 2 pi, phi_l from the host's table:
// d_l * hi_l is exact, is reduced by 2 pi = P1 + P2 + P3 (k * P1 exact),
// and the reduced heads are summed without rounding error (two-sum) while
// the small tails (d_l * lo_l, k * P2, k * P3) accumulate separately.  The
// angle handed to sincosf is within about 1.5e-7 rad of the exact one.
// `hi` and `lo` point to the table staged in shared memory ([3][kMaxHalfDim]
// each): kernel parameters indexed differently in every lane serialise.
__device__ __forceinline__ float2 rope_cos_sin_f(long long n, const float* hi, const float* lo, int i) {
  const bool neg = n < 0;
  const unsigned int m = static_cast<unsigned int>(neg ? -n : n);
  float sh = 0.f, sl = 0.f;
#pragma unroll
  for (int l = 0; l < 3; ++l) {
    const float d = static_cast<float>((m >> (10 * l)) & 1023u);
    const float tt = d * hi[l * kMaxHalfDim + i];  // exact
    const float k = rintf(tt * kInvTwoPiF);
    const float rh = fmaf(-k, kTwoPiP1, tt);  // exact
    const float s = sh + rh, bb = s - sh;
    sl += (sh - (s - bb)) + (rh - bb);
    sh = s;
    sl = fmaf(-k, kTwoPiP2, sl);
    sl = fmaf(-k, kTwoPiP3, sl);
    sl = fmaf(d, lo[l * kMaxHalfDim + i], sl);
  }
  const float k = rintf(sh * kInvTwoPiF);
  sh = fmaf(-k, kTwoPiP1, sh);
  sl = fmaf(-k, kTwoPiP2, sl);
  float sn, cs;
  sincosf(sh + sl, &sn, &cs);
  return make_float2(cs, neg ? -sn : sn);
}

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
// Rotates the bf16 pairs (x_i, x_i+1) and (y_i, y_i+1) (rotate-half
// partners) by the table entry t = {cos_i, cos_i+1, sin_i, sin_i+1}:
// (x, y) -> (x c - y s, y c + x s), split into bf16 hi and lo words.
__device__ __forceinline__ void rotate_split(uint32_t xw, uint32_t yw, const float4 t, uint32_t& xh, uint32_t& xl,
                                             uint32_t& yh, uint32_t& yl) {
  const float2 x = unpack_bf16(xw), y = unpack_bf16(yw);
  const float2 c = make_float2(t.x, t.y), s = make_float2(t.z, t.w);
  split_bf16(__ffma2_rn(y, neg2(s), __fmul2_rn(x, c)), xh, xl);
  split_bf16(__ffma2_rn(x, s, __fmul2_rn(y, c)), yh, yl);
}

// Rotations of two frequencies at once: (c, s) = (cos, sin) of frequencies
// (i, i + 1), turned further by the rotation in t = {cos_i, cos_i+1, sin_i,
// sin_i+1} (angles add).
__device__ __forceinline__ void turn2(float2& c, float2& s, const float4 t) {
  const float2 tc = make_float2(t.x, t.y), ts = make_float2(t.z, t.w);
  const float2 nc = __ffma2_rn(s, neg2(ts), __fmul2_rn(c, tc));
  const float2 ns = __ffma2_rn(c, ts, __fmul2_rn(s, tc));
  c = nc;
  s = ns;
}

// floor(a / G) for 0 <= a < G + 64 (a < 128 when G < 64): the quotient is 0
// or 1 once G >= 64; below that (a + 0.5) / G in float is far enough from an
// integer that the float quotient floors exactly.
__device__ __forceinline__ int div_small(int a, int G, float invG) {
  if (G >= 64) return a >= G ? 1 : 0;
  return static_cast<int>(__fmul_rn(static_cast<float>(a) + 0.5f, invG));
}

template <int D, int GQ>
__global__ void __launch_bounds__(kMaxWarps * 32, 1)
decode_partial_kernel(DecodeKParams p) {
  constexpr int kNT = (GQ + 3) / 4;                // score n-tiles: 4 heads x {hi, lo} each
  constexpr int kHalf = D / 2;
  constexpr int kQuads = D / 4;                    // table entries (frequency pairs) per key
  constexpr int kRowChunks = D / 8;                // 16-byte chunks per cache row
  constexpr int kRowsPerCopy = 32 / kRowChunks;    // rows one warp-wide copy covers
  constexpr int kCopies = kStep / kRowsPerCopy;    // copies per step and matrix
  constexpr int kStageBytes = kStep * 2 * D * 2;   // K and V rows of one step
  constexpr int kVOff = kStep * D * 2;             // V rows within a stage
  constexpr int kSC = D / 32;                      // score chunks of 16 dims (+ rotate-half partner)
  constexpr int kMT = D / 16;                      // O^T m-tiles of 16 dims
  constexpr int kBlockSteps = kBlockKeys / kStep;  // global steps per table block (4)
  constexpr int kTabEntries = kBlockKeys * kQuads;
  // P V columns: with GQ <= 4, column n holds head n & 3, its P hi part for
  // n < 4 and its lo part for n >= 4; with GQ = 8 column n is head n.
  constexpr bool kLoCols = GQ <= 4;
  auto hcol = [](int n) { return kLoCols ? (n & 3) : n; };
  const int gq = p.gq;    // query heads per KV head (<= GQ)
  const int wph = p.wph;  // warps per KV head (1, 2 or 4), alternate steps
  const int block_local = kBlockSteps / wph;  // steps per warp per table block

  extern __shared__ __align__(16) unsigned char smem_raw[];
  // Two rotation tables [64 keys][kQuads] float4 {cos_i, cos_i+1, sin_i,
  // sin_i+1}, entry (t, pp) at column pp ^ 4 (t & 1) so that the fragment
  // reads are free of bank conflicts; then the small tables, the first
  // block's base, the query rotations, and the per-warp rings.  The raw
  // query rows are staged in the second table buffer during the set-up.
  float4* s_tab = reinterpret_cast<float4*>(smem_raw);
  float4* s_small = s_tab + 2 * kTabEntries;                                    // [17][kQuads]
  float2* s_base0 = reinterpret_cast<float2*>(s_small + kSmallRows * kQuads);  // [kHalf]
  float2* s_qcs = s_base0 + kHalf;                                              // [2][kHalf]
  unsigned char* s_ring = reinterpret_cast<unsigned char*>(s_qcs + 2 * kHalf);
  const __nv_bfloat16* s_q = reinterpret_cast<const __nv_bfloat16*>(s_tab + kTabEntries);
  __shared__ float s_ang_hi[3 * kMaxHalfDim], s_ang_lo[3 * kMaxHalfDim];  // the angle tables, staged

  // Let the merge kernel (a programmatic dependent) launch early; it waits
  // for this grid's completion before reading the partials.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  // This grid is itself a programmatic dependent of the preceding work on
  // the stream (which may produce q or the cache, or still read the
  // partials): its CTAs may be scheduled while that work finishes, and wait
  // for it here, before touching any memory.
  asm volatile("griddepcontrol.wait;\n" ::: "memory");

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
      if (threadIdx.x == 0 && split == 0 && blockIdx.z == 0) atomicCAS(p.status, 0, 30);
      L = min(max(L, 1), p.Lcap);
    }
    G = static_cast<int>(group_size(L, p.wp));
  }
  long long step0, step1;
  if (split < p.split_r) {
    step0 = static_cast<long long>(p.steps_r) * split / p.split_r;
    step1 = static_cast<long long>(p.steps_r) * (split + 1) / p.split_r;
  } else {
    const long long nl = gridDim.x - p.split_r, sl = split - p.split_r, rest = p.steps_all - p.steps_r;
    step0 = p.steps_r + rest * sl / nl;
    step1 = p.steps_r + rest * (sl + 1) / nl;
  }
  const int js = static_cast<int>(min(static_cast<long long>(L), kStep * step0));
  const int je = static_cast<int>(min(static_cast<long long>(L), kStep * step1));
  const int qpos = L - 1;
  const bool bifocal = G > 1;

  // Warp `par` of KV head hkl takes the global steps it = wph * u + par.
  // KV heads past Hkv (last head group) stream nothing but keep the CTA's
  // barrier count.
  const int hkl = warp % p.hpc, par = warp / p.hpc;
  const int hk0 = blockIdx.z * p.hpc;
  const int hk = hk0 + hkl;
  const bool head_ok = hk < p.Hkv;
  const long long row_stride = static_cast<long long>(p.Hkv) * D;
  const long long cache_off = (static_cast<long long>(b) * p.Lcap * p.Hkv + (head_ok ? hk : 0)) * D;
  const __nv_bfloat16* kbase = p.kc + cache_off;
  const __nv_bfloat16* vbase = p.vc + cache_off;
  unsigned char* my_ring = s_ring + warp * kStages * kStageBytes;
  const uint32_t ring = static_cast<uint32_t>(__cvta_generic_to_shared(my_ring));
  const int nsteps_all = (je - js + kStep - 1) / kStep;
  const int nsteps = head_ok ? nsteps_all : 0;
  const int nlocal = (nsteps_all + wph - 1) / wph;  // same for every warp

  // The CTA's raw query rows (query heads hk0 * gq ..), one cp.async group.
  {
    const int nh = min(p.hpc, p.Hkv - hk0) * gq;
    const __nv_bfloat16* qsrc = p.q + (static_cast<long long>(b) * p.Hq + hk0 * gq) * D;
    const uint32_t qdst = static_cast<uint32_t>(__cvta_generic_to_shared(s_q));
    for (int c = tid; c < nh * (D / 8); c += nthr) cp_async16(qdst + 16 * c, qsrc + 8 * c, 16);
    cp_async_commit();
  }

  // Stage layout: K rows of the step's 16 keys (2D bytes each), then V rows.
  // 16-byte chunk c of key row r sits at chunk c ^ (r & 7) of its row, so
  // that the eight rows of an 8x8 ldmatrix tile fall in eight bank groups.
  const int crow = lane / kRowChunks, cchunk = lane % kRowChunks;
  const long long lane_src = crow * row_stride + cchunk * 8;
  const long long copy_stride = kRowsPerCopy * row_stride;
  uint32_t lane_dst[kCopies];
#pragma unroll
  for (int i = 0; i < kCopies; ++i) {
    const int key = kRowsPerCopy * i + crow;
    lane_dst[i] = static_cast<uint32_t>((key * kRowChunks + (cchunk ^ (key & 7))) * 16);
  }
  auto issue_step = [&](int u) {
    const int it = wph * u + par;
    if (it < nsteps) {
      const int jstep = js + it * kStep;
      const uint32_t st = ring + static_cast<uint32_t>((u & (kStages - 1)) * kStageBytes);
      const __nv_bfloat16* kp = kbase + lane_src + static_cast<long long>(jstep) * row_stride;
      const __nv_bfloat16* vp = vbase + lane_src + static_cast<long long>(jstep) * row_stride;
      if (jstep + kStep <= je) {  // full step: no bounds checks
#pragma unroll
        for (int i = 0; i < kCopies; ++i) {
          cp_async16(st + lane_dst[i], kp + i * copy_stride, 16);
          cp_async16(st + kVOff + lane_dst[i], vp + i * copy_stride, 16);
        }
      } else {
#pragma unroll
        for (int i = 0; i < kCopies; ++i) {
          const bool ok = jstep + kRowsPerCopy * i + crow < je;
          cp_async16(st + lane_dst[i], ok ? kp + i * copy_stride : kbase, ok ? 16 : 0);
          cp_async16(st + kVOff + lane_dst[i], ok ? vp + i * copy_stride : vbase, ok ? 16 : 0);
        }
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int s = 0; s < kStages; ++s) issue_step(s);
  for (int i = tid; i < 3 * kHalf; i += nthr) {
    const int l = i / kHalf, f = i % kHalf;
    s_ang_hi[l * kMaxHalfDim + f] = p.ang.hi[l][f];
    s_ang_lo[l * kMaxHalfDim + f] = p.ang.lo[l][f];
  }
  __syncthreads();

  // ---- Set-up, while the query rows and the first two steps are in flight ----
  // Query rotations R_{L-1} and R_{f(L-1)}, the first block's base
  // R_{Delta(js)} (angles reduced in double), and the small tables R_{-c}
  // (c < 8) and R_{-8a} (a <= 8) with omega = hi + lo, hi holding 17
  // significant bits so that n * hi is exact in float for n <= 64.
  const bool any_remote = bifocal && js < je && !is_local(qpos, js, p.w0);
  for (int i = tid; i < kHalf * (any_remote ? 3 : 2); i += nthr) {
    const int which = i / kHalf, f = i % kHalf;
    const long long pos = which == 0 ? qpos : which == 1 ? alias(qpos, G) : alias_offset(js, G);
    const float2 cs = rope_cos_sin_f(pos, s_ang_hi, s_ang_lo, f);
    if (which < 2)
      s_qcs[which * kHalf + f] = cs;
    else
      s_base0[f] = cs;
  }
  if (any_remote) {
    for (int idx = tid; idx < kSmallRows * kQuads; idx += nthr) {
      const int r = idx / kQuads, pp = idx % kQuads;
      const int n = r < 8 ? r : 8 * (r - 8);
      const float2 cs[2] = {rope_cos_sin_f(n, s_ang_hi, s_ang_lo, 2 * pp),
                            rope_cos_sin_f(n, s_ang_hi, s_ang_lo, 2 * pp + 1)};
      s_small[idx] = make_float4(cs[0].x, cs[1].x, -cs[0].y, -cs[1].y);  // R_{-n}
    }
  }
  cp_async_wait<kStages>();  // the query rows (the oldest group) have landed
  __syncthreads();

  // Query operands of the score MMA (B, 16 dims x 8 columns per chunk):
  // column n of n-tile nt is head 4 nt + n / 2, hi part (n even) or lo part
  // (n odd) of the pre-scaled rotated query; variant 0 absolute, 1 aliased.
  // Chunk c < kSC holds the first-half dims 16 c + 8 e + 2 t4 (+1) and chunk
  // c + kSC their rotate-half partners, so each lane rotates its own pairs.
  uint32_t qf[2][kNT][kMT][2];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
    const int hl = 4 * nt + (g >> 1);
    const bool valid = head_ok && hl < gq;
    const __nv_bfloat16* qrow = s_q + (valid ? hkl * gq + hl : 0) * D;
#pragma unroll
    for (int c = 0; c < kSC; ++c)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int i = 16 * c + 8 * e + 2 * t4;
        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(qrow + i));
        const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(qrow + kHalf + i));
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          const float2 c0 = s_qcs[v * kHalf + i], c1 = s_qcs[v * kHalf + i + 1];
          const float2 cc = make_float2(c0.x, c1.x), ss = make_float2(c0.y, c1.y);
          const float2 sc = make_float2(p.scale_log2, p.scale_log2);
          const float2 rx = __fmul2_rn(__ffma2_rn(y, neg2(ss), __fmul2_rn(x, cc)), sc);
          const float2 ry = __fmul2_rn(__ffma2_rn(x, ss, __fmul2_rn(y, cc)), sc);
          uint32_t hi, lo;
          split_bf16(rx, hi, lo);
          qf[v][nt][c][e] = valid ? ((g & 1) ? lo : hi) : 0u;
          split_bf16(ry, hi, lo);
          qf[v][nt][c + kSC][e] = valid ? ((g & 1) ? lo : hi) : 0u;
        }
      }
  }

  // Rotation-table state of this thread: frequency pair pp (fixed, since
  // nthr is a multiple of 32 >= kQuads), the base of the block being built,
  // and j0 mod G of that block.
  const int pp = tid % kQuads;
  const int entries_per_thread = (kTabEntries + nthr - 1) / nthr;
  const int per_step = (entries_per_thread + block_local - 1) / block_local;
  const float invG = 1.0f / static_cast<float>(G);
  float2 bc = make_float2(1.f, 1.f), bs = make_float2(0.f, 0.f);
  int r0 = 0;
  auto build_entries = [&](int buf, int k0, int k1) {
    float4* tab = s_tab + buf * kTabEntries;
    for (int k = k0; k < k1; ++k) {
      const int e = tid + nthr * k;
      if (e >= kTabEntries) break;
      const int t = e / kQuads;
      const int n = t - div_small(r0 + t, G, invG);  // 0..63
      float2 c = bc, s = bs;
      turn2(c, s, s_small[(8 + (n >> 3)) * kQuads + pp]);
      turn2(c, s, s_small[(n & 7) * kQuads + pp]);
      tab[t * kQuads + (pp ^ ((t & 1) << 2))] = make_float4(c.x, c.y, s.x, s.y);
    }
  };
  if (any_remote) {
    const float2 b0 = s_base0[2 * pp], b1 = s_base0[2 * pp + 1];
    bc = make_float2(b0.x, b1.x);
    bs = make_float2(b0.y, b1.y);
    r0 = js % G;
  }
  __syncthreads();  // query rows read; their buffer becomes table 1
  if (any_remote) build_entries(0, 0, entries_per_thread);
  __syncthreads();  // table of block 0 complete

  // O^T accumulators: m-tile mt holds dims 16 mt + g (+8) of heads 2 t4, 2 t4 + 1.
  float o[kMT][4];
#pragma unroll
  for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[mt][e] = 0.f;
  // Softmax state of head 4 nt + t4 (the same in the 8 lanes of a column).
  float m_run[kNT], l_run[kNT];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
    m_run[nt] = -INFINITY;
    l_run[nt] = 0.f;
  }
  // ldmatrix lane roles.  Scores (A, 16 keys x 16 dims): lane l addresses key
  // (l & 7) + 8 ((l >> 3) & 1) at chunk 2 c + (l >> 4).  P V (A = V^T, 16
  // dims x 16 keys, transposed): key (l & 7) + 8 (l >> 4) at chunk 2 mt +
  // ((l >> 3) & 1).  Offsets relative to the stage, per chunk index.
  const int ka = (lane & 7) + 8 * ((lane >> 3) & 1), kb = (lane & 7) + 8 * (lane >> 4);
  const uint32_t a_row = static_cast<uint32_t>(ka * 2 * D), b_row = static_cast<uint32_t>(kVOff + kb * 2 * D);
  const int a_sw = ka & 7, b_sw = kb & 7, a_hi = lane >> 4, b_hi = (lane >> 3) & 1;
  const int sw = (g & 1) << 2;  // table column swizzle of this lane's keys (g and g + 8)

  for (int u = 0; u < nlocal; ++u) {
    const int it = wph * u + par;
    const int blk = u / block_local, ub = u - blk * block_local;
    const int j0 = js + blk * kBlockKeys;  // table block base
    // Block blk's table was built during block blk - 1 (or the set-up);
    // after this barrier nobody reads block blk - 1's buffer any more.
    if (ub == 0 && blk > 0) __syncthreads();
    // Part of the next block's table (remote keys form a prefix of [0, L)).
    if (bifocal && j0 + kBlockKeys < je && !is_local(qpos, j0 + kBlockKeys, p.w0)) {
      if (ub == 0) {  // base and residue of block blk + 1
        const int q64 = div_small(r0 + kBlockKeys, G, invG);
        const int n = kBlockKeys - q64;  // 0..64
        turn2(bc, bs, s_small[(8 + (n >> 3)) * kQuads + pp]);
        turn2(bc, bs, s_small[(n & 7) * kQuads + pp]);
        r0 += kBlockKeys - q64 * G;
      }
      build_entries((blk + 1) & 1, ub * per_step, min((ub + 1) * per_step, entries_per_thread));
    }
    cp_async_wait<kStages - 1>();
    __syncwarp();
    if (it < nsteps) {
      const int jstep = js + it * kStep;
      const uint32_t st = ring + static_cast<uint32_t>((u & (kStages - 1)) * kStageBytes);
      const bool all_local = !bifocal || is_local(qpos, jstep, p.w0);
      const bool all_remote = bifocal && !is_local(qpos, jstep + kStep - 1, p.w0);

      // Scores z[nt][r] of (key jstep + g + 8 r, head 4 nt + t4), log2 units.
      float z[kNT][2];
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) z[nt][0] = z[nt][1] = 0.f;
      if (!all_local) {
        // Aliased scores.  A = the step's 16 keys corrected by R_{f(j) - j},
        // once with their bf16 hi parts and once with the lo parts; chunk c
        // (dims 16 c ..) and chunk c + kSC (the rotate-half partners).
        float acc[kNT][4];
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
        const float4* tab0 = s_tab + (blk & 1) * kTabEntries + (jstep - j0 + g) * kQuads;
        const float4* tab1 = tab0 + 8 * kQuads;
#pragma unroll
        for (int c = 0; c < kSC; ++c) {
          uint32_t x0, x1, x2, x3, y0, y1, y2, y3;
          ldsm_x4(st + a_row + static_cast<uint32_t>(((2 * c + a_hi) ^ a_sw) << 4), x0, x1, x2, x3);
          ldsm_x4(st + a_row + static_cast<uint32_t>(((D / 16 + 2 * c + a_hi) ^ a_sw) << 4), y0, y1, y2, y3);
          // x0/y0: key g, dims 16 c + 2 t4 (+1); x1/y1: key g + 8, same dims;
          // x2/y2: key g, dims 16 c + 8 + 2 t4; x3/y3: key g + 8, those dims.
          uint32_t h[8], l[8];
          rotate_split(x0, y0, tab0[(8 * c + t4) ^ sw], h[0], l[0], h[4], l[4]);
          rotate_split(x1, y1, tab1[(8 * c + t4) ^ sw], h[1], l[1], h[5], l[5]);
          rotate_split(x2, y2, tab0[(8 * c + 4 + t4) ^ sw], h[2], l[2], h[6], l[6]);
          rotate_split(x3, y3, tab1[(8 * c + 4 + t4) ^ sw], h[3], l[3], h[7], l[7]);
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            mma16816(acc[nt], h[0], h[1], h[2], h[3], qf[1][nt][c][0], qf[1][nt][c][1]);
            mma16816(acc[nt], l[0], l[1], l[2], l[3], qf[1][nt][c][0], qf[1][nt][c][1]);
            mma16816(acc[nt], h[4], h[5], h[6], h[7], qf[1][nt][c + kSC][0], qf[1][nt][c + kSC][1]);
            mma16816(acc[nt], l[4], l[5], l[6], l[7], qf[1][nt][c + kSC][0], qf[1][nt][c + kSC][1]);
          }
        }
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          z[nt][0] = acc[nt][0] + acc[nt][1];
          z[nt][1] = acc[nt][2] + acc[nt][3];
        }
      }
      if (!all_remote) {
        // Absolute scores: the cached keys as stored (exact in bf16).
        float acc[kNT][4];
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
#pragma unroll
        for (int c = 0; c < kSC; ++c) {
          uint32_t x0, x1, x2, x3, y0, y1, y2, y3;
          ldsm_x4(st + a_row + static_cast<uint32_t>(((2 * c + a_hi) ^ a_sw) << 4), x0, x1, x2, x3);
          ldsm_x4(st + a_row + static_cast<uint32_t>(((D / 16 + 2 * c + a_hi) ^ a_sw) << 4), y0, y1, y2, y3);
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            mma16816(acc[nt], x0, x1, x2, x3, qf[0][nt][c][0], qf[0][nt][c][1]);
            mma16816(acc[nt], y0, y1, y2, y3, qf[0][nt][c + kSC][0], qf[0][nt][c + kSC][1]);
          }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const bool local = all_local || is_local(qpos, jstep + g + 8 * r, p.w0);
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt)
            if (local) z[nt][r] = acc[nt][2 * r] + acc[nt][2 * r + 1];
        }
      }

      // Online softmax per head (column); the max used for the exponentials
      // is raised only when it grows by more than kRescaleThreshold.
      bool any_rescale = false;
      float pr[kNT][2], al[kNT];
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        const bool hv = 4 * nt + t4 < gq;
        const float z0 = hv && jstep + g < je ? z[nt][0] : -INFINITY;
        const float z1 = hv && jstep + g + 8 < je ? z[nt][1] : -INFINITY;
        float bm = fmaxf(z0, z1);
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
        float alpha = 1.f;
        if (bm > m_run[nt] + kRescaleThreshold) {
          alpha = exp2f(m_run[nt] - bm);
          m_run[nt] = bm;
        }
        const float mexp = m_run[nt] == -INFINITY ? 0.f : m_run[nt];
        pr[nt][0] = exp2f(z0 - mexp);
        pr[nt][1] = exp2f(z1 - mexp);
        l_run[nt] = l_run[nt] * alpha + (pr[nt][0] + pr[nt][1]);
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
        for (int mt = 0; mt < kMT; ++mt) {
          o[mt][0] *= ae;
          o[mt][1] *= ao;
          o[mt][2] *= ae;
          o[mt][3] *= ao;
        }
      }
      // P^T operand (B, 16 keys x 8 columns): keys 2 t4, 2 t4 + 1 (b0) and
      // 2 t4 + 8, 2 t4 + 9 (b1) of column g, i.e. of head hcol(g); key k < 8
      // of head hh sits in lane 4 k + (hh & 3), key k + 8 in the same lane's
      // second slot.  P is split as hi + lo in bf16: with GQ <= 4 the lo
      // parts fill columns 4..7, otherwise they go through a second product.
      uint32_t pb_hi[2], pb_lo[2];
      {
        const int hh = hcol(g);
        const int src = 8 * t4 + (hh & 3);
        float pv[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const float a = __shfl_sync(0xffffffffu, pr[nt][r], src);
            const float c = __shfl_sync(0xffffffffu, pr[nt][r], src + 4);
            if ((hh >> 2) == nt) {
              pv[r][0] = a;
              pv[r][1] = c;
            }
          }
        const bool use = hh < gq;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          uint32_t hi, lo;
          split_bf16(make_float2(pv[r][0], pv[r][1]), hi, lo);
          if constexpr (kLoCols) {
            pb_hi[r] = use ? (g < 4 ? hi : lo) : 0u;
            pb_lo[r] = 0u;
          } else {
            pb_hi[r] = use ? hi : 0u;
            pb_lo[r] = use ? lo : 0u;
          }
        }
      }
      // O^T += V^T P^T: one transposed x4 load of V per 16-dim m-tile (keys
      // past the slice end have p = 0 and zero-filled rows).
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        uint32_t v0, v1, v2, v3;
        ldsm_x4_t(st + b_row + static_cast<uint32_t>(((2 * mt + b_hi) ^ b_sw) << 4), v0, v1, v2, v3);
        mma16816(o[mt], v0, v1, v2, v3, pb_hi[0], pb_hi[1]);
        if constexpr (!kLoCols) mma16816(o[mt], v0, v1, v2, v3, pb_lo[0], pb_lo[1]);
      }
    }
    __syncwarp();  // the stage is rewritten next
    issue_step(u + kStages);
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
  if constexpr (kLoCols) {
    // Column n + 4 (lane t4 + 2) holds the lo-part product of column n.
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mt][e] += __shfl_xor_sync(0xffffffffu, o[mt][e], 2);
  }
  if (wph == 1) {
    // One warp per KV head: its state is the CTA's partial for the head.
    if (!head_ok) return;
    const long long slot0 = (static_cast<long long>(split) * p.B + b) * p.Hq + hk * gq;
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) {
      const int d0 = 16 * mt + g;
      const int h0 = 2 * t4, h1 = 2 * t4 + 1;
      if (h0 < gq) {
        p.part_o[(slot0 + h0) * D + d0] = o[mt][0];
        p.part_o[(slot0 + h0) * D + d0 + 8] = o[mt][2];
      }
      if (h1 < gq) {
        p.part_o[(slot0 + h1) * D + d0] = o[mt][1];
        p.part_o[(slot0 + h1) * D + d0 + 8] = o[mt][3];
      }
    }
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      const int h = 4 * nt + t4;
      if (g == 0 && h < gq) *reinterpret_cast<float2*>(p.part_ml + (slot0 + h) * 2) = make_float2(m_run[nt], lh[nt]);
    }
    return;
  }
  // Several warps per KV head: each leaves its state in its (now idle)
  // ring, o [gq][D] then (m, l) [gq][2], and the CTA merges them.
  __syncthreads();
  float* hand = reinterpret_cast<float*>(my_ring);
#pragma unroll
  for (int mt = 0; mt < kMT; ++mt) {
    const int d0 = 16 * mt + g;
    const int h0 = 2 * t4, h1 = 2 * t4 + 1;
    if (h0 < gq) {
      hand[h0 * D + d0] = o[mt][0];
      hand[h0 * D + d0 + 8] = o[mt][2];
    }
    if (h1 < gq) {
      hand[h1 * D + d0] = o[mt][1];
      hand[h1 * D + d0 + 8] = o[mt][3];
    }
  }
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
    const int h = 4 * nt + t4;
    if (g == 0 && h < gq) {
      hand[gq * D + 2 * h] = m_run[nt];
      hand[gq * D + 2 * h + 1] = lh[nt];
    }
  }
  __syncthreads();
  // Merge: M = max over the head's warps, weights 2^(m_w - M).
  for (int idx = tid; idx < p.hpc * gq * kQuads; idx += nthr) {
    const int hql = idx / kQuads, d4 = idx % kQuads;
    const int kvl = hql / gq, h = hql % gq;
    const int kv = hk0 + kvl;
    if (kv >= p.Hkv) continue;
    float M = -INFINITY;
    for (int w = 0; w < wph; ++w) {
      const float* src = reinterpret_cast<const float*>(s_ring + (kvl + w * p.hpc) * kStages * kStageBytes);
      M = fmaxf(M, src[gq * D + 2 * h]);
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lsum = 0.f;
    for (int w = 0; w < wph; ++w) {
      const float* src = reinterpret_cast<const float*>(s_ring + (kvl + w * p.hpc) * kStages * kStageBytes);
      const float mw = src[gq * D + 2 * h];
      const float a = M == -INFINITY ? 0.f : exp2f(mw - M);
      lsum += a * src[gq * D + 2 * h + 1];
      const float4 v = *reinterpret_cast<const float4*>(src + h * D + 4 * d4);
      acc.x += a * v.x;
      acc.y += a * v.y;
      acc.z += a * v.z;
      acc.w += a * v.w;
    }
    const long long slot = (static_cast<long long>(split) * p.B + b) * p.Hq + kv * gq + h;
    *reinterpret_cast<float4*>(p.part_o + slot * D + 4 * d4) = acc;
    if (d4 == 0) *reinterpret_cast<float2*>(p.part_ml + slot * 2) = make_float2(M, lsum);
  }
}

// Merge the per-slice partials of one (batch, query head) with log-sum-exp
// weights: out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s, M = max m_s.
// Each warp takes the slices s = warp (mod 16) and requests up to kBatch of
// them at once (one round trip to L2 for up to 160 slices), folding them
// into a running (max, sum, vector); the warps then combine in shared
// memory.  A lane owns D / 32 output elements.
constexpr int kMergeWarps = 16;
constexpr int kMergeBatch = 10;

template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32)
decode_merge_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                    int nsplit, int BH, __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  constexpr int kV = D / 32;
  __shared__ float s_m[kMergeWarps], s_l[kMergeWarps];
  __shared__ __align__(16) float s_acc[kMergeWarps][D];
  // The next grid on the stream may be scheduled now (a programmatic
  // dependent such as the next decode's partial kernel waits for this grid
  // before touching memory).
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  // The partials are written by the preceding grid.
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  const int bh = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float M = -INFINITY, Lsum = 0.f;
  float acc[kV];
#pragma unroll
  for (int v = 0; v < kV; ++v) acc[v] = 0.f;
  for (int s0 = warp; s0 < nsplit; s0 += kMergeWarps * kMergeBatch) {
    float2 ml[kMergeBatch];
    float os[kMergeBatch][kV];
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) {
      const int s = s0 + kMergeWarps * k;
      if (s < nsplit) {
        const long long slot = static_cast<long long>(s) * BH + bh;
        ml[k] = *reinterpret_cast<const float2*>(part_ml + slot * 2);
        if constexpr (kV == 4) {
          const float4 t = *reinterpret_cast<const float4*>(part_o + slot * D + 4 * lane);
          os[k][0] = t.x; os[k][1] = t.y; os[k][2] = t.z; os[k][3] = t.w;
        } else {
          const float2 t = *reinterpret_cast<const float2*>(part_o + slot * D + 2 * lane);
          os[k][0] = t.x; os[k][1] = t.y;
        }
      } else {
        ml[k] = make_float2(-INFINITY, 0.f);
#pragma unroll
        for (int v = 0; v < kV; ++v) os[k][v] = 0.f;
      }
    }
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) {
      const float Mn = fmaxf(M, ml[k].x);
      if (Mn == -INFINITY) continue;
      const float a = exp2f(M - Mn), w = exp2f(ml[k].x - Mn);
      Lsum = Lsum * a + ml[k].y * w;
#pragma unroll
      for (int v = 0; v < kV; ++v) acc[v] = acc[v] * a + os[k][v] * w;
      M = Mn;
    }
  }
#pragma unroll
  for (int v = 0; v < kV; ++v) s_acc[warp][kV * lane + v] = acc[v];
  if (lane == 0) {
    s_m[warp] = M;
    s_l[warp] = Lsum;
  }
  __syncthreads();
  if (warp == 0) {
    float Mt = s_m[0];
#pragma unroll
    for (int w = 1; w < kMergeWarps; ++w) Mt = fmaxf(Mt, s_m[w]);
    float Dn = 0.f;
    float t[kV];
#pragma unroll
    for (int v = 0; v < kV; ++v) t[v] = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) {
      const float a = s_m[w] == -INFINITY ? 0.f : exp2f(s_m[w] - Mt);
      Dn += a * s_l[w];
#pragma unroll
      for (int v = 0; v < kV; ++v) t[v] += a * s_acc[w][kV * lane + v];
    }
    const float inv = 1.f / Dn;
    __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(out + static_cast<long long>(bh) * D + kV * lane);
#pragma unroll
    for (int v = 0; v < kV; v += 2) dst[v / 2] = __floats2bfloat162_rn(t[v] * inv, t[v + 1] * inv);
    if (lse != nullptr && lane == 0) lse[bh] = (Mt + log2f(Dn)) * 0.69314718055994531f;
  }
}

// Streaming multiprocessors of the current device (cached per device).
int num_sms() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

// Capacity of the query-head template for gq query heads per KV head.
int gq_capacity(int gq) { return gq <= 1 ? 1 : gq <= 2 ? 2 : gq <= 4 ? 4 : gq <= 8 ? 8 : 0; }

template <int D, int GQ>
cudaError_t launch_partial(const dim3& grid, int warps, size_t smem, const DecodeKParams& p, cudaStream_t stream) {
  cudaError_t err = cudaFuncSetAttribute(decode_partial_kernel<D, GQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  // A programmatic dependent of the preceding work on the stream (the kernel
  // waits for it before touching memory), so that its launch overlaps that
  // work's tail.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(32 * warps);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_partial_kernel<D, GQ>, p);
}

}  // namespace

int decode_max_splits() { return kMaxSplits; }

int decode_slice_cap() { return std::min(num_sms(), kMaxSplits); }

size_t decode_workspace_bytes(int B, int Hq, int d, int Lcap) {
  (void)Lcap;
  return static_cast<size_t>(kMaxSplits) * B * Hq * (d + 2) * sizeof(float);
}

size_t decode_scratch_bytes(int B, int Hq, int d) {
  return static_cast<size_t>(decode_slice_cap()) * B * Hq * (d + 2) * sizeof(float);
}

bool decode_supported(int Hq, int Hkv, int d) {
  return (d == 64 || d == 128) && Hkv >= 1 && Hq % Hkv == 0 && gq_capacity(Hq / Hkv) != 0;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (!decode_supported(a.Hq, a.Hkv, a.d)) return cudaErrorInvalidValue;
  const int gq = a.Hq / a.Hkv, cap = gq_capacity(gq);
  const int ngroups = (a.Hkv + kMaxHeadsPerCta - 1) / kMaxHeadsPerCta;
  const int hpc = (a.Hkv + ngroups - 1) / ngroups;
  const int wph = std::min(4, kMaxWarps / hpc);  // 1, 2 or 4: a table block is 4 steps
  // Slices: one wave over the SMs for one sequence, in whole 16-key steps
  // spread evenly; with a batch, up to kMinStepsPerSplit steps per slice as
  // long as the batch's slices still fill a wave (short sequences would
  // otherwise pay the per-CTA set-up for a few steps).
  const int nsm = num_sms();
  const int slice_cap = decode_slice_cap();
  const long long S = (static_cast<long long>(a.L) + kStep - 1) / kStep;
  const long long target = std::max(1, std::min(slice_cap, nsm / ngroups));
  const long long fill = std::min<long long>(kMinStepsPerSplit, S * a.B * ngroups / nsm);
  const long long sps = std::max((S + target - 1) / target, std::max(fill, 1LL));
  const int nsplit = static_cast<int>((S + sps - 1) / sps);

  DecodeKParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.kc = static_cast<const __nv_bfloat16*>(a.k_cache);
  p.vc = static_cast<const __nv_bfloat16*>(a.v_cache);
  p.part_o = a.part;
  p.part_ml = a.part + static_cast<size_t>(slice_cap) * a.B * a.Hq * a.d;
  p.B = a.B; p.L = a.L; p.Lcap = a.Lcap; p.Hq = a.Hq; p.Hkv = a.Hkv;
  p.gq = gq; p.hpc = hpc; p.wph = wph;
  p.w0 = a.w0; p.G = a.G; p.wp = a.wp;
  // Cost split: steps holding a remote key cost about kRemoteCost times an
  // all-local step (correction rotation and hi/lo split of every element,
  // measured on B300 at L = 32769).  Batched decode with per-sequence
  // lengths keeps the even split (each sequence has its own G and window).
  long long steps_r = S;
  if (a.seqlens == nullptr) {
    const long long first_local = first_local_key(a.L - 1, a.w0);  // keys >= first_local are local
    steps_r = a.G > 1 ? std::min(S, std::max(0LL, (first_local + kStep - 1) / kStep)) : 0;
  }
  int split_r = nsplit;
  if (steps_r < S) {
    const double wr = kRemoteCost * static_cast<double>(steps_r), wl = static_cast<double>(S - steps_r);
    split_r = static_cast<int>(std::lround(nsplit * wr / (wr + wl)));
    split_r = std::max(steps_r > 0 ? 1 : 0, std::min(split_r, nsplit - 1));
  }
  // One region when either side gets no slice (e.g. a single slice).
  if (split_r >= nsplit) {
    split_r = nsplit;
    steps_r = S;
  } else if (split_r <= 0) {
    split_r = 0;
    steps_r = 0;
  }
  p.steps_r = static_cast<int>(steps_r);
  p.steps_all = static_cast<int>(S);
  p.split_r = split_r;
  p.seqlens = a.seqlens;
  p.status = device_status_ptr();
  if (p.status == nullptr) return cudaErrorInvalidSymbol;
  p.scale_log2 = a.scale_log2;
  p.ang = a.ang;

  const int warps = hpc * wph;
  const size_t stage_bytes = static_cast<size_t>(kStep) * 2 * a.d * 2;
  const size_t smem = static_cast<size_t>(2 * kBlockKeys + kSmallRows) * (a.d / 4) * 16 +  // tables
                      static_cast<size_t>(3) * (a.d / 2) * sizeof(float2) +               // base, query rotations
                      static_cast<size_t>(warps) * kStages * stage_bytes;                 // rings
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  const dim3 grid(nsplit, a.B, ngroups);
  cudaError_t err = cudaErrorInvalidValue;
#define JL_DECODE_CASE(DV, GQV) \
  if (a.d == DV && cap == GQV) err = launch_partial<DV, GQV>(grid, warps, smem, p, stream);
  JL_DECODE_CASE(128, 1)
  JL_DECODE_CASE(128, 2)
  JL_DECODE_CASE(128, 4)
  JL_DECODE_CASE(128, 8)
  JL_DECODE_CASE(64, 1)
  JL_DECODE_CASE(64, 2)
  JL_DECODE_CASE(64, 4)
  JL_DECODE_CASE(64, 8)
#undef JL_DECODE_CASE
  if (err != cudaSuccess) return err;

  // The merge waits on the partial kernel through griddepcontrol.wait, so it
  // may be launched before that kernel finishes.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B * a.Hq);
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.d == 128)
    return cudaLaunchKernelEx(&cfg, decode_merge_kernel<128>, static_cast<const float*>(p.part_o),
                              static_cast<const float*>(p.part_ml), nsplit, a.B * a.Hq,
                              static_cast<__nv_bfloat16*>(a.o), a.lse);
  return cudaLaunchKernelEx(&cfg, decode_merge_kernel<64>, static_cast<const float*>(p.part_o),
                            static_cast<const float*>(p.part_ml), nsplit, a.B * a.Hq,
                            static_cast<__nv_bfloat16*>(a.o), a.lse);
}

}  // namespace jl
