// Causal bifocal attention over pre-rotated operands on the sm_100-family
// tensor cores (tcgen05.mma, accumulators in tensor memory, TMA-fed
// shared-memory ring, warp-specialised roles).
//
// Routing (paper digest page, "Method", Eq. 1).  A CTA owns two 128-row query
// tiles of one head (rows q0 .. q0+255) and walks the key tiles in two
// phases: first the "remote" visits, key tiles that hold pairs with
// q - k > w0, scored with Q_rem K_rem^T (both rotated at aliased positions
// f(x) = floor(x / G)); then the "local" visits, key tiles that hold pairs
// with 0 <= q - k <= w0, scored with Q_abs K_abs^T.  A key tile that straddles
// the q - k = w0 band is visited once in each phase, each visit masked to its
// own pairs, so every causal pair is scored exactly once with the right
// rotation and only straddling tiles pay for two score sets.  The online
// softmax makes the order of visits irrelevant.  Only one rotation of Q is
// resident at a time: after the last remote visit the Q tiles are reloaded
// with the absolute rotation.  In window-only mode (the local views A and C
// of the three-pass form, Eq. 7) the remote phase is skipped, and the qa/ka
// operands are whichever rotation the caller passes.
//
// Roles (10 warps):
//   warps 0-3  softmax of query tile 0 (thread = row = TMEM lane)
//   warps 4-7  softmax of query tile 1
//   warp  8    tensor-core issue (the whole warp runs the loop, one elected
//              lane issues each MMA and commit) and TMEM allocation
//   warp  9    TMA producer (one thread)
// Tensor memory (512 columns): S_0, S_1 (fp32 scores, 128 columns each),
// O_0, O_1 (fp32 outputs); P_t (bf16 probabilities) overwrites the first 64
// columns of S_t and feeds the PV product straight from tensor memory.
// Per visit the issue order is PV(t, v-1) then QK(t, v) for t = 0, 1, so the
// tensor core works on one tile while the softmax warps work on the other.
//
// Softmax: base-2 exponentials with scale * log2(e) folded in; the running
// max is raised only when it grows by more than 8 (log2 units), so O is
// rescaled in tensor memory rarely.  The row log-sum-exp is exported in
// natural log.  Every barrier wait is bounded (and suspends the thread rather
// than spinning): on expiry the CTA records a status code, drains its bulk
// copies and tensor-core work and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>

#include "internal.h"
#include "positions.cuh"
#include "sm100.cuh"

namespace jl {
namespace {

using namespace sm100;

constexpr int kBM = 128;                    // rows per query tile
constexpr int kBN = 128;                    // keys per key tile
constexpr int kBoxBytes = 128 * 64 * 2;     // one 128-row x 64-column swizzled box
constexpr int kSlots = 5;                   // K/V ring depth
constexpr int kThreads = 320;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr long long kWaitLimit = 4000000000ll;  // clock cycles (~2 s)
constexpr float kRescaleThreshold = 8.0f;       // log2 units

// Per head dim D: a tile is D/64 boxes of 128 rows x 64 columns.
template <int D>
struct Cfg {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kSmemBytes = 2 * kTileBytes + kSlots * kTileBytes + 1024;  // + alignment slack
  // Matrix descriptor strides of the value tile read as an MN-major B
  // operand: LBO = distance between 64-column boxes, SBO = 8 key rows.
  static constexpr uint32_t kVLbo = kBoxBytes;
  static constexpr uint32_t kVSbo = 1024;
};

struct TcParams {
  int B, Lq, q_base, Hq, Hkv, w0, G, npairs;
  int pair_block;  // query-tile pairs per scheduling block (about one wave per KV head)
  int window_only;  // skip the remote phase (local views of the three-pass form)
  long long wait_limit;  // clock cycles a pipeline wait may take before the CTA gives up
  float scale_log2;
  __nv_bfloat16* o;
  float* lse;
  int* status;
};

// The visits of one CTA: v < nr are remote visits of key tile v; the rest
// are local visits of key tiles jl0 .. jmax.
struct Plan {
  int nr, jl0, jmax, nv;
};

// q0: position of the CTA's first query row; qend: one past the last query
// position of the call.  window_only: no remote visits.
__device__ __forceinline__ Plan make_plan(int q0, int qend, int w0, bool window_only) {
  Plan p;
  const int qlast = min(q0 + 2 * kBM - 1, qend - 1);
  p.jmax = qlast / kBN;
  p.nr = window_only ? 0 : min(remote_tile_count(qlast, w0, kBN), p.jmax + 1);
  p.jl0 = first_local_tile(q0, w0, kBN);
  p.nv = p.nr + (p.jmax - p.jl0 + 1);
  return p;
}

__device__ __forceinline__ void visit_of(const Plan& p, int v, int& j, bool& remote) {
  remote = v < p.nr;
  j = remote ? v : p.jl0 + (v - p.nr);
}

struct Bars {
  uint64_t q_full, q_empty, mma_final;
  uint64_t full[kSlots], empty[kSlots];
  uint64_t s_full[2], p_full[2], pv_done[2];
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_qa, const __grid_constant__ CUtensorMap tm_qr,
                  const __grid_constant__ CUtensorMap tm_ka, const __grid_constant__ CUtensorMap tm_kr,
                  const __grid_constant__ CUtensorMap tm_v, TcParams prm) {
  constexpr int kTileBytes = Cfg<D>::kTileBytes;
  constexpr int kBoxes = D / 64;
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) Bars bars;
  __shared__ uint32_t s_tmem_base;
  __shared__ volatile int s_abort;

  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = smem_base;                  // 2 query tiles
  const uint32_t sRing = smem_base + 2 * kTileBytes;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Grid order: blocks of pair_block query-tile pairs, longest rows first;
  // within a block, batch, then KV head, then pair, then the query heads of
  // the KV head.  A resident wave (about one CTA per SM) is then the query
  // heads of one KV head over adjacent tile pairs, which walk the same K/V
  // tiles at about the same time, so most K/V reads are served from L2.
  const int gqh = prm.Hq / prm.Hkv;
  const int u = blockIdx.x;
  const int per_block = prm.pair_block * prm.B * prm.Hq;  // CTAs of a full block
  const int blk = u / per_block, rin = u % per_block;
  const int p_hi = prm.npairs - 1 - blk * prm.pair_block;  // longest pair of the block
  const int nb = min(prm.pair_block, p_hi + 1);            // pairs in this block
  const int hq_in = rin % gqh, pi = (rin / gqh) % nb, bk = rin / (gqh * nb);
  const int b = bk / prm.Hkv, hk = bk % prm.Hkv;
  const int pair = p_hi - pi;
  const int h = hk * gqh + hq_in;
  const int row0 = pair * 2 * kBM;        // first query row of the CTA (local)
  const int q0 = prm.q_base + row0;       // its position
  const Plan plan = make_plan(q0, prm.q_base + prm.Lq, prm.w0, prm.window_only != 0);

  auto bar = [](uint64_t& x) { return smem_u32(&x); };

  if (tid == 0) {
    s_abort = 0;
    mbar_init(bar(bars.q_full), 1);
    mbar_init(bar(bars.q_empty), 1);
    mbar_init(bar(bars.mma_final), 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar(bars.full[s]), 1);
      mbar_init(bar(bars.empty[s]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(bars.s_full[t]), 1);
      mbar_init(bar(bars.p_full[t]), 4 * 32);
      mbar_init(bar(bars.pv_done[t]), 1);
    }
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&s_tmem_base), 512);
    tmem_relinquish();
  }
  if (warp == kLoadWarp && lane == 0) {
    prefetch_tensormap(&tm_qa);
    prefetch_tensormap(&tm_qr);
    prefetch_tensormap(&tm_ka);
    prefetch_tensormap(&tm_kr);
    prefetch_tensormap(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem_base;

  auto fail = [&](int code) {
    s_abort = 1;
    atomicCAS(prm.status, 0, code);
  };

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      auto load_q = [&](const CUtensorMap* m) {
        mbar_arrive_expect_tx(bar(bars.q_full), 2 * kTileBytes);
        for (int t = 0; t < 2; ++t)
          for (int c = 0; c < kBoxes; ++c)
            tma_load_4d(sQ + t * kTileBytes + c * kBoxBytes, m, bar(bars.q_full), 64 * c, h, row0 + t * kBM, b);
      };
      load_q(plan.nr > 0 ? &tm_qr : &tm_qa);
      int qloads = 1;
      bool ok = true;
      int idx = 0;
      for (int v = 0; v < plan.nv && ok; ++v) {
        int j;
        bool remote;
        visit_of(plan, v, j, remote);
        if (v == plan.nr && v > 0) {  // switch the resident Q rotation
          if (!(ok = mbar_wait(bar(bars.q_empty), 0, &s_abort, prm.wait_limit))) { fail(1); break; }
          load_q(&tm_qa);
          ++qloads;
        }
        for (int part = 0; part < 2 && ok; ++part, ++idx) {  // K then V
          const int s = idx % kSlots, use = idx / kSlots;
          if (use > 0 && !(ok = mbar_wait(bar(bars.empty[s]), (use - 1) & 1, &s_abort, prm.wait_limit))) {
            fail(2);
            break;
          }
          const uint32_t dst = sRing + s * kTileBytes;
          mbar_arrive_expect_tx(bar(bars.full[s]), kTileBytes);
          for (int c = 0; c < kBoxes; ++c) {
            tma_load_4d(dst + c * kBoxBytes, part == 0 ? (remote ? &tm_kr : &tm_ka) : &tm_v, bar(bars.full[s]),
                        64 * c, hk, j * kBN, b);
          }
        }
      }
      // Drain: every bulk copy this thread started has landed before the CTA
      // may exit (on the normal path these waits return at once).  The
      // latest arming of each ring slot is among the last kSlots loads; the
      // waits use the full limit and ignore the abort flag.
      const volatile int never = 0;
      bool drained = true;
      for (int i = max(0, idx - kSlots); i < idx; ++i)
        drained &= mbar_wait(bar(bars.full[i % kSlots]), (i / kSlots) & 1, &never, kWaitLimit);
      drained &= mbar_wait(bar(bars.q_full), (qloads - 1) & 1, &never, kWaitLimit);
      if (!drained) atomicCAS(prm.status, 0, 11);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ tensor-core issue
    // The whole warp runs the loop, so the descriptors and addresses are
    // warp-uniform (uniform registers); one elected lane issues each
    // operation.  Wait outcomes are made warp-uniform.
    const uint32_t id_qk = idesc_bf16_f32(kBM, kBN, false);
    const uint32_t id_pv = idesc_bf16_f32(kBM, D, true);
    const uint64_t qdesc[2] = {desc_sw128(sQ, 16, 1024), desc_sw128(sQ + kTileBytes, 16, 1024)};
    auto wait = [&](uint32_t b, uint32_t parity, int code) {
      const bool r = __all_sync(0xffffffffu, mbar_wait(b, parity, &s_abort, prm.wait_limit));
      if (!r && lane == 0) fail(code);
      return r;
    };
    auto wait_slot = [&](int idx) {
      if (!wait(bar(bars.full[idx % kSlots]), (idx / kSlots) & 1, 4)) return false;
      tc_fence_after();
      return true;
    };
    auto pv = [&](int t, int vprev) {  // O_t += P_t V(vprev)
      if (!wait(bar(bars.p_full[t]), vprev & 1, 5)) return false;
      tc_fence_after();
      const uint64_t vdesc = desc_sw128(sRing + ((2 * vprev + 1) % kSlots) * kTileBytes, Cfg<D>::kVLbo, Cfg<D>::kVSbo);
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk)  // 16 keys = 2048 bytes per step
        mma_ts_elect(tmem + 256 + t * 128, tmem + t * 128 + kk * 8, vdesc + (kk * 2048 >> 4), id_pv,
                     (vprev > 0 || kk > 0) ? 1u : 0u);
      mma_commit_elect(bar(bars.pv_done[t]));
      return true;
    };
    bool ok = wait(bar(bars.q_full), 0, 3);
    for (int v = 0; v < plan.nv && ok; ++v) {
      if (v > 0 && !(ok = wait_slot(2 * (v - 1) + 1))) break;  // V of the previous visit
      if (!(ok = wait_slot(2 * v))) break;                     // K of this visit
      // Descriptors advance by their start-address field (bytes >> 4).
      const uint64_t kdesc = desc_sw128(sRing + ((2 * v) % kSlots) * kTileBytes, 16, 1024);
      for (int t = 0; t < 2 && ok; ++t) {
        if (v > 0) {
          if (!(ok = pv(t, v - 1))) break;
          if (t == 1) mma_commit_elect(bar(bars.empty[(2 * (v - 1) + 1) % kSlots]));
        }
        if (t == 0 && v == plan.nr && v > 0) {  // first local visit: Q_abs resident?
          if (!(ok = wait(bar(bars.q_full), 1, 6))) break;
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
          mma_ss_elect(tmem + t * 128, qdesc[t] + off, kdesc + off, id_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit_elect(bar(bars.s_full[t]));
      }
      if (!ok) break;
      mma_commit_elect(bar(bars.empty[(2 * v) % kSlots]));
      if (v == plan.nr - 1 && plan.nr < plan.nv) mma_commit_elect(bar(bars.q_empty));
    }
    if (ok) {
      const int vl = plan.nv - 1;
      ok = wait_slot(2 * vl + 1);
      for (int t = 0; t < 2 && ok; ++t) ok = pv(t, vl);
      if (ok) mma_commit_elect(bar(bars.empty[(2 * vl + 1) % kSlots]));
    }
    // Drain: every MMA issued by this warp completes before TMEM is freed.
    mma_commit_elect(bar(bars.mma_final));
    const volatile int never = 0;
    if (!__all_sync(0xffffffffu, mbar_wait(bar(bars.mma_final), 0, &never, kWaitLimit)) && lane == 0)
      atomicCAS(prm.status, 0, 7);
  } else {
    // ------------------------------------------------------------ softmax warps
    const int t = warp >> 2;           // query tile
    const int r = (warp & 3) * 32 + lane;  // row in tile = TMEM lane
    const int q = q0 + t * kBM + r;        // query position
    const int qrow = row0 + t * kBM + r;   // output row
    const int q0t = q0 + t * kBM;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * 128;
    const uint32_t tO = tmem + lane_base + 256 + t * 128;  // D columns
    const float sc = prm.scale_log2;
    const int w0 = prm.w0;
    float m_used = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int v = 0; v < plan.nv; ++v) {
      int j;
      bool remote;
      visit_of(plan, v, j, remote);
      const int k0 = j * kBN;
      // Every lane waits; the outcome is made warp-uniform, since the
      // tensor-memory accesses that follow are warp-collective.
      ok = __all_sync(0xffffffffu, mbar_wait(bar(bars.s_full[t]), v & 1, &s_abort, prm.wait_limit));
      if (!ok) { fail(8); break; }
      tc_fence_after();
      uint32_t a0[32], a1[32], a2[32], a3[32];
      tmem_ld32(tS + 0, a0);
      tmem_ld32(tS + 32, a1);
      tmem_ld32(tS + 64, a2);
      tmem_ld32(tS + 96, a3);
      tmem_ld_wait(a0);
      tmem_ld_wait(a1);
      tmem_ld_wait(a2);
      tmem_ld_wait(a3);
      float s[128];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        s[i] = __uint_as_float(a0[i]);
        s[32 + i] = __uint_as_float(a1[i]);
        s[64 + i] = __uint_as_float(a2[i]);
        s[96 + i] = __uint_as_float(a3[i]);
      }
      // Masks are needed only on tiles at the window band or the diagonal.
      const bool need_mask = remote ? remote_visit_needs_mask(q0t, kBM, k0, kBN, w0)
                                    : local_visit_needs_mask(q0t, kBM, k0, kBN, w0);
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (!visit_keeps(remote, q, k0 + c, w0)) s[c] = -INFINITY;
      }
      // Row max and row sum as 8-way trees (independent chains).
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = s[k];
#pragma unroll
      for (int c = 8; c < 128; c += 8)
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(mx8[k], s[c + k]);
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const float m_new = fmaxf(m_used, mx * sc);
      float factor = 1.f;
      if (m_new > m_used + kRescaleThreshold) {
        factor = ex2_approx(m_used - m_new);  // 0 when m_used is -inf
        m_used = m_new;
      }
      const float m_exp = (m_used == -INFINITY) ? 0.f : m_used;
      const float2 sc2 = make_float2(sc, sc), nm2 = make_float2(-m_exp, -m_exp);
      float2 sum2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
      // P columns 0..63 (bf16 pairs) over S columns already read, stored 16
      // columns at a time so that few packed registers are live next to S.
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = 32 * q4 + 2 * i;
          const float2 a = __ffma2_rn(make_float2(s[c], s[c + 1]), sc2, nm2);
          const float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
          sum2[i & 3] = __fadd2_rn(sum2[i & 3], e);
          pk[i] = pack_bf16x2(e.x, e.y);
        }
        tmem_st16(tS + 16 * q4, pk);
      }
      const float2 t2 = __fadd2_rn(__fadd2_rn(sum2[0], sum2[1]), __fadd2_rn(sum2[2], sum2[3]));
      const float rowsum = t2.x + t2.y;
      l_run = l_run * factor + rowsum;
      // Rescale O_t in tensor memory when any row of this warp raised its max.
      if (v > 0 && __any_sync(0xffffffffu, factor != 1.f)) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(bars.pv_done[t]), (v - 1) & 1, &s_abort, prm.wait_limit));
        if (!ok) { fail(9); break; }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * factor);
          tmem_st32(tO + c * 32, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(bars.p_full[t]));
    }
    // P stores of an iteration that gave up may still be in flight.
    tmem_st_wait();
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(bars.pv_done[t]), (plan.nv - 1) & 1, &s_abort, prm.wait_limit));
    if (ok) {
      tc_fence_after();
      const float inv = 1.f / l_run;
      __nv_bfloat16* orow = prm.o + ((static_cast<long long>(b) * prm.Lq + qrow) * prm.Hq + h) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_ld_wait(o);
        if (qrow < prm.Lq) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[8 * i + 0]) * inv, __uint_as_float(o[8 * i + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(o[8 * i + 2]) * inv, __uint_as_float(o[8 * i + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(o[8 * i + 4]) * inv, __uint_as_float(o[8 * i + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(o[8 * i + 6]) * inv, __uint_as_float(o[8 * i + 7]) * inv);
            dst[i] = w;
          }
        }
      }
      if (qrow < prm.Lq && prm.lse != nullptr)
        prm.lse[(static_cast<long long>(b) * prm.Hq + h) * prm.Lq + qrow] =
            (m_used + log2f(l_run)) * 0.69314718055994531f;
    } else {
      fail(10);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// 4-D map (d, head, row, batch) over a TensorView, boxes of 64 columns x
// `rows` rows of one head.
bool make_view_map(CUtensorMap* m, const TensorView& t, int d, int heads, int B, int rows) {
  const uint64_t dims[4] = {static_cast<uint64_t>(d), static_cast<uint64_t>(heads),
                            static_cast<uint64_t>(t.rows), static_cast<uint64_t>(B)};
  const uint64_t strides[3] = {static_cast<uint64_t>(t.sh) * 2, static_cast<uint64_t>(t.sr) * 2,
                               static_cast<uint64_t>(t.sb) * 2};
  const uint32_t box[4] = {64, 1, static_cast<uint32_t>(rows), 1};
  return make_tmap_bf16(m, t.base, 4, dims, strides, box, true);
}

template <int D>
cudaError_t launch_tc(const PrefillArgs& a, int* status, cudaStream_t stream) {
  CUtensorMap tqa, tqr, tka, tkr, tv;
  if (!make_view_map(&tqa, a.qa, D, a.Hq, a.B, kBM) || !make_view_map(&tqr, a.qr, D, a.Hq, a.B, kBM) ||
      !make_view_map(&tka, a.ka, D, a.Hkv, a.B, kBN) || !make_view_map(&tkr, a.kr, D, a.Hkv, a.B, kBN) ||
      !make_view_map(&tv, a.v, D, a.Hkv, a.B, kBN))
    return cudaErrorInvalidValue;
  TcParams p;
  p.B = a.B;
  p.Lq = a.Lq;
  p.q_base = a.q_base;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  // One G for the call; with G == 1 both rotations coincide, so every pair
  // is scored in the local phase (no window).
  // A window-only call keeps its window (clamped so that position
  // arithmetic cannot overflow).
  p.w0 = a.window_only ? std::min(a.w0, 1 << 30) : ((a.G == 1 || a.w0 >= a.Lk) ? (1 << 30) : a.w0);
  p.window_only = a.window_only ? 1 : 0;
  p.wait_limit = a.wait_limit > 0 ? a.wait_limit : kWaitLimit;
  p.G = a.G;
  p.npairs = (a.Lq + 2 * kBM - 1) / (2 * kBM);
  {
    int dev = 0, nsm = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    p.pair_block = std::max(1, std::min(p.npairs, nsm / (a.Hq / a.Hkv)));
  }
  p.scale_log2 = a.scale_log2;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.status = status;
  constexpr int smem = Cfg<D>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long blocks = static_cast<long long>(p.npairs) * a.B * a.Hq;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  prefill_tc_kernel<D><<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(tqa, tqr, tka, tkr, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_attention(const PrefillArgs& a, cudaStream_t stream) {
  int* status = device_status_ptr();
  if (status == nullptr) return cudaErrorInvalidSymbol;
  if (a.d == 128 && a.cta_pair) return launch_prefill_attention_pair(a, status, stream);
  if (a.d == 128) return launch_tc<128>(a, status, stream);
  if (a.d == 64) return launch_tc<64>(a, status, stream);
  return cudaErrorInvalidValue;
}

}  // namespace jl
