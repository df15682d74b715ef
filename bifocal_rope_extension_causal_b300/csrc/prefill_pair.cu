// Causal bifocal attention over pre-rotated operands, head dim 128, on CTA
// pairs: a cluster of two CTAs runs each tensor-core operation together
// (tcgen05.mma.cta_group::2, M = 256), so the pair shares every K/V tile while
// each CTA keeps only one 128-row query tile and its own accumulators.
//
// Routing (paper digest page, "Method", Eq. 1) is the one of the single-CTA
// kernel: the pair's 256 query rows walk the key tiles that hold remote pairs
// (q - k > w0) with Q_rem K_rem^T, then the key tiles that hold local pairs
// with Q_abs K_abs^T; a key tile that straddles the q - k = w0 band is
// visited in both phases, each visit masked to its own pairs.  Only one Q
// rotation is resident: it is reloaded once, between the phases.
//
// Why pairs.  With two 128-row query tiles in one CTA, the two score tiles
// and the two output tiles fill all 512 tensor-memory columns, so the score
// tile cannot be double-buffered and each tile's softmax sits on the
// tensor core's critical path between its QK^T and its PV.  In a pair, each
// CTA holds one query tile: S is double-buffered (2 x 128 columns) next to
// O (128 columns), the softmax of visit v overlaps QK^T of visit v+1 and PV
// of visit v-1, and each K/V tile still serves 256 query rows.  Each CTA
// loads half of every K/V tile into its own shared memory: 64 of the 128 key
// rows of K (the B operand of QK^T is split by its N = key columns) and 64
// of the 128 dims of V (the B operand of PV is split by its N = dims).
//
// Roles (10 warps per CTA):
//   warps 0-7  softmax of the CTA's query tile: warp w reads TMEM lanes
//              32 (w % 4) .. +31 (one row per thread) and key columns
//              64 (w / 4) .. +63; the two warps of a row exchange row maxima
//              and sums through shared memory
//   warp  8    rank 0: tensor-core issue (one thread); rank 1: forwards the
//              completion of its own TMA loads to rank 0; both: tensor
//              memory allocation for the pair
//   warp  9    TMA producer of the CTA's own Q tile and K/V halves
// Tensor memory per CTA: S_0, S_1 (fp32 scores, columns 0 and 128), O (fp32,
// column 256); P (bf16) overwrites the first 64 columns of its S buffer and
// feeds PV straight from tensor memory.
//
// Every barrier wait is bounded; on expiry the CTA records a status code,
// tells its peer, drains its copies and tensor-core work and exits.
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

constexpr int kD = 128;
constexpr int kBM = 128;                  // query rows per CTA; a pair covers 256
constexpr int kBN = 128;                  // keys per key tile
constexpr int kQBox = 128 * 64 * 2;       // Q box: 128 rows x 64 columns (16 KB)
constexpr int kKBox = 64 * 64 * 2;        // K half box: 64 rows x 64 columns (8 KB)
constexpr int kQBytes = 2 * kQBox;        // one query tile
constexpr int kSlotBytes = 16384;         // a K half (two 64-row boxes) or a V half (one 128-row box)
constexpr int kSlots = 10;                // K/V ring depth
constexpr int kSmemBytes = kQBytes + kSlots * kSlotBytes + 1024;  // + alignment slack
constexpr int kThreads = 320;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr int kColO = 256;                       // O in tensor memory
constexpr long long kWaitLimit = 4000000000ll;  // clock cycles (~2 s)
constexpr float kRescaleThreshold = 8.0f;       // log2 units

struct PairParams {
  int B, Lq, q_base, Hq, Hkv, w0, G, npairs;
  int pair_block;   // query-tile pairs per scheduling block (about one wave per KV head)
  int window_only;  // skip the remote phase (local views of the three-pass form)
  long long wait_limit;
  float scale_log2;
  __nv_bfloat16* o;
  float* lse;
  int* status;
};

struct Plan {
  int nr, jl0, jmax, nv;
};

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

// Barriers.  l*: completion of this CTA's own TMA loads; p*: rank 1's loads,
// forwarded to rank 0 (used on rank 0 only).  empty, q_empty, s_full,
// pv_done and mma_final are signalled in both CTAs by the tensor-core
// commits of rank 0; p_full (rank 0 only) collects the 16 softmax warps of
// the pair.
struct Bars {
  uint64_t lq_full, pq_full, q_empty, mma_final;
  uint64_t lfull[kSlots], pfull[kSlots], empty[kSlots];
  uint64_t s_full[2], p_full[2], pv_done[2];
};

__global__ void __launch_bounds__(kThreads, 1)
prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_qa, const __grid_constant__ CUtensorMap tm_qr,
                    const __grid_constant__ CUtensorMap tm_ka, const __grid_constant__ CUtensorMap tm_kr,
                    const __grid_constant__ CUtensorMap tm_v, PairParams prm) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) Bars bars;
  __shared__ uint32_t s_tmem_base;
  __shared__ volatile int s_abort;
  __shared__ float s_xmax[2][8][32];  // row-max halves, by visit parity
  __shared__ int s_xok[2][8][32];
  __shared__ float s_xsum[8][32];    // epilogue: row-sum halves
  __shared__ int s_xeok[8][32];

  // Identical layout in both CTAs: the tensor core reads each CTA's operands
  // at the same shared-memory offsets.
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = smem_base;
  const uint32_t sRing = smem_base + kQBytes;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const uint32_t peer = rank ^ 1u;
  // Grid order (per pair): blocks of pair_block query-tile pairs, longest
  // rows first; within a block, batch, then KV head, then pair, then the
  // query heads of the KV head, so that the pairs resident at one time walk
  // the same K/V tiles.
  const int gqh = prm.Hq / prm.Hkv;
  const int u = blockIdx.x >> 1;
  const int per_block = prm.pair_block * prm.B * prm.Hq;
  const int blk = u / per_block, rin = u % per_block;
  const int p_hi = prm.npairs - 1 - blk * prm.pair_block;
  const int nb = min(prm.pair_block, p_hi + 1);
  const int hq_in = rin % gqh, pi = (rin / gqh) % nb, bk = rin / (gqh * nb);
  const int b = bk / prm.Hkv, hk = bk % prm.Hkv;
  const int pair = p_hi - pi;
  const int h = hk * gqh + hq_in;
  const int row0 = pair * 2 * kBM;   // first query row of the pair (local)
  const int q0 = prm.q_base + row0;  // its position
  const int my_row0 = row0 + static_cast<int>(rank) * kBM;
  const Plan plan = make_plan(q0, prm.q_base + prm.Lq, prm.w0, prm.window_only != 0);

  auto bar = [](uint64_t& x) { return smem_u32(&x); };

  if (tid == 0) {
    s_abort = 0;
    mbar_init(bar(bars.lq_full), 1);
    mbar_init(bar(bars.pq_full), 1);
    mbar_init(bar(bars.q_empty), 1);
    mbar_init(bar(bars.mma_final), 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar(bars.lfull[s]), 1);
      mbar_init(bar(bars.pfull[s]), 1);
      mbar_init(bar(bars.empty[s]), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(bars.s_full[x]), 1);
      mbar_init(bar(bars.p_full[x]), 16);
      mbar_init(bar(bars.pv_done[x]), 1);
    }
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc_pair(smem_u32(&s_tmem_base), 512);
    tmem_relinquish_pair();
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
  cluster_sync();  // the peer's barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = s_tmem_base;
  const uint32_t peer_abort = map_to_rank(smem_u32(const_cast<int*>(&s_abort)), peer);

  auto fail = [&](int code) {
    s_abort = 1;
    st_cluster_u32(peer_abort, 1u);
    atomicCAS(prm.status, 0, code);
  };

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      auto load_q = [&](const CUtensorMap* m) {
        mbar_arrive_expect_tx(bar(bars.lq_full), kQBytes);
        for (int c = 0; c < 2; ++c) tma_load_4d(sQ + c * kQBox, m, bar(bars.lq_full), 64 * c, h, my_row0, b);
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
        for (int part = 0; part < 2 && ok; ++part, ++idx) {  // K half, then V half
          const int s = idx % kSlots, use = idx / kSlots;
          if (use > 0 && !(ok = mbar_wait(bar(bars.empty[s]), (use - 1) & 1, &s_abort, prm.wait_limit))) {
            fail(2);
            break;
          }
          const uint32_t dst = sRing + s * kSlotBytes;
          mbar_arrive_expect_tx(bar(bars.lfull[s]), kSlotBytes);
          if (part == 0) {
            const CUtensorMap* km = remote ? &tm_kr : &tm_ka;
            for (int c = 0; c < 2; ++c)
              tma_load_4d(dst + c * kKBox, km, bar(bars.lfull[s]), 64 * c, hk, j * kBN + static_cast<int>(rank) * 64, b);
          } else {
            tma_load_4d(dst, &tm_v, bar(bars.lfull[s]), 64 * static_cast<int>(rank), hk, j * kBN, b);
          }
        }
      }
      // Drain: every bulk copy this thread started has landed before the CTA
      // may exit (the waits ignore the abort flag).
      const volatile int never = 0;
      bool drained = true;
      for (int i = max(0, idx - kSlots); i < idx; ++i)
        drained &= mbar_wait(bar(bars.lfull[i % kSlots]), (i / kSlots) & 1, &never, kWaitLimit);
      drained &= mbar_wait(bar(bars.lq_full), (qloads - 1) & 1, &never, kWaitLimit);
      if (!drained) atomicCAS(prm.status, 0, 11);
    }
  } else if (warp == kMmaWarp && rank == 1) {
    // ------------------------------------------------------------ rank 1: forward load completions
    if (lane == 0) {
      auto forward = [&](uint64_t& local, uint32_t parity, uint64_t& remote) {
        if (!mbar_wait(bar(local), parity, &s_abort, prm.wait_limit)) return false;
        mbar_arrive_cluster(map_to_rank(bar(remote), 0));
        return true;
      };
      bool ok = forward(bars.lq_full, 0, bars.pq_full);
      int idx = 0;
      for (int v = 0; v < plan.nv && ok; ++v) {
        if (v == plan.nr && v > 0) ok = forward(bars.lq_full, 1, bars.pq_full);
        for (int part = 0; part < 2 && ok; ++part, ++idx) {
          const int s = idx % kSlots;
          ok = forward(bars.lfull[s], (idx / kSlots) & 1, bars.pfull[s]);
        }
      }
      if (!ok) fail(12);
      // The last commit of rank 0 reaches this CTA too; after it, no
      // tensor-core operation of the pair touches this CTA's memory.
      const volatile int never = 0;
      if (!mbar_wait(bar(bars.mma_final), 0, &never, kWaitLimit)) atomicCAS(prm.status, 0, 7);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ rank 0: tensor-core issue
    // The whole warp runs the loop (warp-uniform descriptors in uniform
    // registers); one elected lane issues each operation.
    const uint32_t id_qk = idesc_bf16_f32(2 * kBM, kBN, false);
    const uint32_t id_pv = idesc_bf16_f32(2 * kBM, kD, true);
    const uint64_t qdesc = desc_sw128(sQ, 16, 1024);
    auto wait = [&](uint64_t& b, uint32_t parity, int code) {
      const bool r = __all_sync(0xffffffffu, mbar_wait(bar(b), parity, &s_abort, prm.wait_limit));
      if (!r && lane == 0) fail(code);
      return r;
    };
    auto wait_both = [&](uint64_t& l, uint64_t& p, uint32_t parity, int code) {
      if (!wait(l, parity, code) || !wait(p, parity, code)) return false;
      tc_fence_after();
      return true;
    };
    auto wait_item = [&](int idx) {
      const int s = idx % kSlots;
      return wait_both(bars.lfull[s], bars.pfull[s], (idx / kSlots) & 1, 4);
    };
    // O += P(w) V(w): P from the S buffer of visit w, V half from the ring.
    auto pv = [&](int w) {
      const int x = w & 1;
      if (!wait(bars.p_full[x], (w >> 1) & 1, 5)) return false;
      tc_fence_after();
      if (!wait_item(2 * w + 1)) return false;
      const uint64_t vdesc = desc_sw128(sRing + ((2 * w + 1) % kSlots) * kSlotBytes, kQBox, 1024);
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk)  // 16 keys = 2048 bytes per step
        mma_ts_pair_elect(tmem + kColO, tmem + x * 128 + kk * 8, vdesc + (kk * 2048 >> 4), id_pv,
                          (w > 0 || kk > 0) ? 1u : 0u);
      mma_commit_pair_elect(bar(bars.pv_done[x]));
      mma_commit_pair_elect(bar(bars.empty[(2 * w + 1) % kSlots]));
      return true;
    };
    bool ok = wait_both(bars.lq_full, bars.pq_full, 0, 3);
    for (int v = 0; v < plan.nv && ok; ++v) {
      if (v == plan.nr && v > 0 && !(ok = wait_both(bars.lq_full, bars.pq_full, 1, 6))) break;
      if (!(ok = wait_item(2 * v))) break;
      // S(v) = Q K^T into buffer v & 1; its previous P was consumed by
      // PV(v - 2), issued earlier (the tensor core runs in issue order).
      // Descriptors advance by their start-address field (bytes >> 4).
      const uint64_t kdesc = desc_sw128(sRing + ((2 * v) % kSlots) * kSlotBytes, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        const uint32_t qoff = (kk >> 2) * kQBox + (kk & 3) * 32;
        const uint32_t koff = (kk >> 2) * kKBox + (kk & 3) * 32;
        mma_ss_pair_elect(tmem + (v & 1) * 128, qdesc + (qoff >> 4), kdesc + (koff >> 4), id_qk, kk > 0 ? 1u : 0u);
      }
      mma_commit_pair_elect(bar(bars.s_full[v & 1]));
      mma_commit_pair_elect(bar(bars.empty[(2 * v) % kSlots]));
      if (v == plan.nr - 1 && plan.nr < plan.nv) mma_commit_pair_elect(bar(bars.q_empty));
      if (v > 0 && !(ok = pv(v - 1))) break;
    }
    if (ok) pv(plan.nv - 1);
    // Drain: every MMA issued by this warp completes before TMEM is freed
    // and before either CTA may exit (the cluster barrier below).
    mma_commit_pair_elect(bar(bars.mma_final));
    const volatile int never = 0;
    if (!__all_sync(0xffffffffu, mbar_wait(bar(bars.mma_final), 0, &never, kWaitLimit)) && lane == 0)
      atomicCAS(prm.status, 0, 7);
  } else {
    // ------------------------------------------------------------ softmax warps (both CTAs)
    const int qd = warp & 3, hf = warp >> 2;  // lane quarter (rows), key-column half
    const int r = qd * 32 + lane;             // row in the tile = TMEM lane
    const int q0t = q0 + static_cast<int>(rank) * kBM;
    const int q = q0t + r;                    // query position
    const int qrow = my_row0 + r;             // output row
    const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
    const uint32_t p_full_addr[2] = {map_to_rank(bar(bars.p_full[0]), 0), map_to_rank(bar(bars.p_full[1]), 0)};
    const float sc = prm.scale_log2;
    const int w0 = prm.w0;
    const int partner = warp ^ 4;
    float m_used = -INFINITY, l_run = 0.f;
    bool ok = true;
    // The two warps of a row take the same branches: every visit both reach
    // the exchange below (named barrier 1 + qd, 64 threads) and leave the
    // loop together when either of them failed.
    for (int v = 0; v < plan.nv; ++v) {
      int j;
      bool remote;
      visit_of(plan, v, j, remote);
      const int kh = j * kBN + hf * 64;  // first key of this warp's columns
      const int x = v & 1;
      const bool wok = ok && __all_sync(0xffffffffu, mbar_wait(bar(bars.s_full[x]), (v >> 1) & 1, &s_abort, prm.wait_limit));
      // The scores are loaded even when the wait gave up (the values are
      // then unused: both warps of the row leave at the exchange below), so
      // that they have a single definition.
      tc_fence_after();
      uint32_t a0[32], a1[32];
      tmem_ld32(tmem + lane_base + x * 128 + hf * 64, a0);
      tmem_ld32(tmem + lane_base + x * 128 + hf * 64 + 32, a1);
      tmem_ld_wait(a0);
      tmem_ld_wait(a1);
      float s[64];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        s[i] = __uint_as_float(a0[i]);
        s[32 + i] = __uint_as_float(a1[i]);
      }
      const bool need_mask = remote ? remote_visit_needs_mask(q0t, kBM, kh, 64, w0)
                                    : local_visit_needs_mask(q0t, kBM, kh, 64, w0);
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (!visit_keeps(remote, q, kh + c, w0)) s[c] = -INFINITY;
      }
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = s[k];
#pragma unroll
      for (int c = 8; c < 64; c += 8)
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(mx8[k], s[c + k]);
      float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      // Row max over both halves.
      s_xmax[x][warp][lane] = mx;
      s_xok[x][warp][lane] = wok ? 1 : 0;
      asm volatile("bar.sync %0, 64;\n" ::"r"(1 + qd) : "memory");
      mx = fmaxf(mx, s_xmax[x][partner][lane]);
      const bool both = wok && s_xok[x][partner][lane] != 0;  // uniform over the warp and its partner
      if (!both) {
        ok = false;
        break;
      }
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
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float2 a = __ffma2_rn(make_float2(s[2 * i], s[2 * i + 1]), sc2, nm2);
        const float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
        sum2[i & 3] = __fadd2_rn(sum2[i & 3], e);
        pk[i] = pack_bf16x2(e.x, e.y);
      }
      // P columns 32 hf .. +31 of the buffer: over S columns that both
      // warps of the row have read before the exchange.
      tmem_st32(tmem + lane_base + x * 128 + hf * 32, pk);
      const float2 t2 = __fadd2_rn(__fadd2_rn(sum2[0], sum2[1]), __fadd2_rn(sum2[2], sum2[3]));
      l_run = l_run * factor + (t2.x + t2.y);
      // Rescale this warp's half of O (dims 64 hf ..) when a row raised its max.
      if (v > 0 && __any_sync(0xffffffffu, factor != 1.f)) {
        const int w = v - 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(bars.pv_done[w & 1]), (w >> 1) & 1, &s_abort, prm.wait_limit))) {
          ok = false;  // the partner learns it at the next exchange
          tmem_st_wait();
          continue;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t o[32];
          const uint32_t ta = tmem + lane_base + kColO + hf * 64 + c * 32;
          tmem_ld32(ta, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * factor);
          tmem_st32(ta, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(bar(bars.p_full[x]));
        else
          mbar_arrive_cluster(p_full_addr[x]);
      }
    }
    tmem_st_wait();
    // Epilogue: wait for the last PV, add the two halves' row sums, write
    // this warp's 64 dims of every row.
    bool eok = ok;
    if (eok) {
      const int w = plan.nv - 1;
      eok = __all_sync(0xffffffffu, mbar_wait(bar(bars.pv_done[w & 1]), (w >> 1) & 1, &s_abort, prm.wait_limit));
    }
    s_xsum[warp][lane] = l_run;
    s_xeok[warp][lane] = eok ? 1 : 0;
    asm volatile("bar.sync %0, 64;\n" ::"r"(1 + qd) : "memory");
    const float l_row = l_run + s_xsum[partner][lane];
    eok = eok && s_xeok[partner][lane] != 0;
    if (eok) {
      tc_fence_after();
      const float inv = 1.f / l_row;
      __nv_bfloat16* orow = prm.o + ((static_cast<long long>(b) * prm.Lq + qrow) * prm.Hq + h) * kD + hf * 64;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_base + kColO + hf * 64 + c * 32, o);
        tmem_ld_wait(o);
        if (qrow < prm.Lq) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 wv;
            wv.x = pack_bf16x2(__uint_as_float(o[8 * i + 0]) * inv, __uint_as_float(o[8 * i + 1]) * inv);
            wv.y = pack_bf16x2(__uint_as_float(o[8 * i + 2]) * inv, __uint_as_float(o[8 * i + 3]) * inv);
            wv.z = pack_bf16x2(__uint_as_float(o[8 * i + 4]) * inv, __uint_as_float(o[8 * i + 5]) * inv);
            wv.w = pack_bf16x2(__uint_as_float(o[8 * i + 6]) * inv, __uint_as_float(o[8 * i + 7]) * inv);
            dst[i] = wv;
          }
        }
      }
      if (hf == 0 && qrow < prm.Lq && prm.lse != nullptr)
        prm.lse[(static_cast<long long>(b) * prm.Hq + h) * prm.Lq + qrow] = (m_used + log2f(l_row)) * 0.69314718055994531f;
    } else if (hf == 0 && lane == 0) {
      fail(10);
    }
  }

  // Both CTAs stay resident until the pair's last tensor-core operation and
  // every remote arrival have completed; then the pair frees its tensor memory.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// 4-D map (d, head, row, batch) over a TensorView, boxes of 64 columns x
// `rows` rows of one head.
bool make_pair_map(CUtensorMap* m, const TensorView& t, int heads, int B, int rows) {
  const uint64_t dims[4] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(heads), static_cast<uint64_t>(t.rows),
                            static_cast<uint64_t>(B)};
  const uint64_t strides[3] = {static_cast<uint64_t>(t.sh) * 2, static_cast<uint64_t>(t.sr) * 2,
                               static_cast<uint64_t>(t.sb) * 2};
  const uint32_t box[4] = {64, 1, static_cast<uint32_t>(rows), 1};
  return make_tmap_bf16(m, t.base, 4, dims, strides, box, true);
}

}  // namespace

cudaError_t launch_prefill_attention_pair(const PrefillArgs& a, int* status, cudaStream_t stream) {
  if (a.d != kD) return cudaErrorInvalidValue;
  CUtensorMap tqa, tqr, tka, tkr, tv;
  if (!make_pair_map(&tqa, a.qa, a.Hq, a.B, kBM) || !make_pair_map(&tqr, a.qr, a.Hq, a.B, kBM) ||
      !make_pair_map(&tka, a.ka, a.Hkv, a.B, 64) || !make_pair_map(&tkr, a.kr, a.Hkv, a.B, 64) ||
      !make_pair_map(&tv, a.v, a.Hkv, a.B, kBN))
    return cudaErrorInvalidValue;
  PairParams p;
  p.B = a.B;
  p.Lq = a.Lq;
  p.q_base = a.q_base;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  // One G for the call; with G == 1 both rotations coincide and every pair
  // is scored in the local phase.  A window-only call keeps its window
  // (clamped so that position arithmetic cannot overflow).
  p.w0 = a.window_only ? std::min(a.w0, 1 << 30) : ((a.G == 1 || a.w0 >= a.Lk) ? (1 << 30) : a.w0);
  p.window_only = a.window_only ? 1 : 0;
  p.wait_limit = a.wait_limit > 0 ? a.wait_limit : kWaitLimit;
  p.G = a.G;
  p.npairs = (a.Lq + 2 * kBM - 1) / (2 * kBM);
  {
    int dev = 0, nsm = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    p.pair_block = std::max(1, std::min(p.npairs, (nsm / 2) / (a.Hq / a.Hkv)));
  }
  p.scale_log2 = a.scale_log2;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.status = status;
  cudaError_t e = cudaFuncSetAttribute(prefill_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long units = static_cast<long long>(p.npairs) * a.B * a.Hq;
  if (units == 0) return cudaSuccess;
  if (2 * units > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * units));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_pair_kernel, tqa, tqr, tka, tkr, tv, p);
}

}  // namespace jl
