// Causal bifocal attention over pre-rotated operands, warp-level MMA version.
//
// One CTA = 64 query rows of one head (4 warps x 16 rows); key tiles of 64
// stream through a two-stage cp.async ring.  Each (query tile, key tile)
// block is routed by its distance range (paper digest page, "Method", Eq. 1):
// local blocks score Q_abs K_abs^T only, remote blocks Q_rem K_rem^T only,
// and only blocks that straddle the q - k = w0 band compute both and select
// per element.  The softmax is the usual online one (fp32 running max and
// sum per row, base-2 exponentials with the scale folded in), and the row
// log-sum-exp is exported in natural log.
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"
#include "positions.cuh"

namespace jl {
namespace {

constexpr int kBM = 64;
constexpr int kBN = 64;
constexpr int kWarps = 4;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global -> shared; src_bytes == 0 zero-fills.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Row-major tile of 64 rows x D bf16 with the 16-byte chunks of each row
// XOR-swizzled by (row & 7) so that ldmatrix reads are bank-conflict free.
template <int D>
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int row, int chunk) {
  return base + static_cast<uint32_t>(row * D * 2 + ((chunk ^ (row & 7)) << 4));
}

// Copy rows [r0, r0 + 64) of a row-major matrix with row stride `stride`
// elements into a swizzled tile; rows >= nrows are zero-filled.
template <int D>
__device__ __forceinline__ void load_tile(uint32_t dst, const __nv_bfloat16* src, long long stride,
                                          int r0, int nrows) {
  constexpr int kChunks = D / 8;
  for (int idx = threadIdx.x; idx < kBM * kChunks; idx += kWarps * 32) {
    const int r = idx / kChunks, c = idx % kChunks;
    const int gr = r0 + r;
    const bool ok = gr < nrows;
    const __nv_bfloat16* g = src + (ok ? gr : 0) * stride + c * 8;
    cp_async16(tile_addr<D>(dst, r, c), g, ok ? 16 : 0);
  }
}

// S = Q K^T for this warp's 16 rows and the 64 keys of the tile.
template <int D>
__device__ __forceinline__ void qk_tile(float (&s)[kBN / 8][4], uint32_t sq, uint32_t sk, int warp,
                                        int lane) {
#pragma unroll
  for (int nb = 0; nb < kBN / 8; ++nb)
#pragma unroll
    for (int e = 0; e < 4; ++e) s[nb][e] = 0.f;
#pragma unroll
  for (int kb = 0; kb < D / 16; ++kb) {
    uint32_t a[4];
    ldsm_x4(a, tile_addr<D>(sq, warp * 16 + (lane & 15), 2 * kb + (lane >> 4)));
#pragma unroll
    for (int np = 0; np < kBN / 16; ++np) {
      uint32_t b[4];
      ldsm_x4(b, tile_addr<D>(sk, np * 16 + (lane >> 4) * 8 + (lane & 7), 2 * kb + ((lane >> 3) & 1)));
      mma_bf16(s[2 * np], a, b[0], b[1]);
      mma_bf16(s[2 * np + 1], a, b[2], b[3]);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
prefill_mma_kernel(PrefillArgs p) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int kTileBytes = kBM * D * 2;
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sQa = s_base, sQr = s_base + kTileBytes;
  // stage s: K_abs, K_rem, V
  auto sKa = [&](int st) { return s_base + (2 + 3 * st) * kTileBytes; };
  auto sKr = [&](int st) { return s_base + (3 + 3 * st) * kTileBytes; };
  auto sV = [&](int st) { return s_base + (4 + 3 * st) * kTileBytes; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int nqt = (p.L + kBM - 1) / kBM;
  const int qt = nqt - 1 - static_cast<int>(blockIdx.x);  // longest rows first
  const int h = blockIdx.y, b = blockIdx.z;
  const int hk = h / (p.Hq / p.Hkv);
  const int q0 = qt * kBM;
  const bool bifocal = p.G > 1;

  const auto* qa = static_cast<const __nv_bfloat16*>(p.qa) + (static_cast<long long>(b) * p.Hq + h) * p.L * D;
  const auto* qr = static_cast<const __nv_bfloat16*>(p.qr) + (static_cast<long long>(b) * p.Hq + h) * p.L * D;
  const auto* ka = static_cast<const __nv_bfloat16*>(p.ka) + (static_cast<long long>(b) * p.Hkv + hk) * p.L * D;
  const auto* kr = static_cast<const __nv_bfloat16*>(p.kr) + (static_cast<long long>(b) * p.Hkv + hk) * p.L * D;
  const auto* vv = static_cast<const __nv_bfloat16*>(p.v) + (static_cast<long long>(b) * p.L * p.Hkv + hk) * D;
  const long long v_stride = static_cast<long long>(p.Hkv) * D;

  const int q_last = min(q0 + kBM - 1, p.L - 1);
  const int n_kv = q_last / kBN + 1;

  auto tile_class = [&](int j) {
    const int c = classify_tile(q0, kBM, j * kBN, kBN, p.w0);
    return bifocal ? c : static_cast<int>(kTileLocal);
  };
  auto issue = [&](int j) {
    const int st = j & 1, c = tile_class(j);
    if (c != kTileRemote) load_tile<D>(sKa(st), ka, D, j * kBN, p.L);
    if (c != kTileLocal) load_tile<D>(sKr(st), kr, D, j * kBN, p.L);
    load_tile<D>(sV(st), vv, v_stride, j * kBN, p.L);
  };

  load_tile<D>(sQa, qa, D, q0, p.L);
  if (bifocal) load_tile<D>(sQr, qr, D, q0, p.L);
  issue(0);
  cp_async_commit();

  float o[D / 8][4];
#pragma unroll
  for (int nb = 0; nb < D / 8; ++nb)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[nb][e] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  const int row0 = q0 + warp * 16 + g;  // rows row0 and row0 + 8

  for (int j = 0; j < n_kv; ++j) {
    if (j + 1 < n_kv) issue(j + 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    const int st = j & 1, c = tile_class(j), k0 = j * kBN;
    float s[kBN / 8][4];
    if (c == kTileRemote) {
      qk_tile<D>(s, sQr, sKr(st), warp, lane);
    } else {
      qk_tile<D>(s, sQa, sKa(st), warp, lane);
      if (c == kTileStraddle) {
        float sr[kBN / 8][4];
        qk_tile<D>(sr, sQr, sKr(st), warp, lane);
#pragma unroll
        for (int nb = 0; nb < kBN / 8; ++nb)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = row0 + ((e & 2) ? 8 : 0);
            const int col = k0 + nb * 8 + 2 * t + (e & 1);
            if (!is_local(r, col, p.w0)) s[nb][e] = sr[nb][e];
          }
      }
    }
    const bool diag = tile_needs_causal_mask(q0, k0, kBN);
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nb = 0; nb < kBN / 8; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float val = s[nb][e] * p.scale_log2;
        if (diag) {
          const int r = row0 + ((e & 2) ? 8 : 0);
          const int col = k0 + nb * 8 + 2 * t + (e & 1);
          if (col > r) val = -INFINITY;
        }
        s[nb][e] = val;
        mx[e >> 1] = fmaxf(mx[e >> 1], val);
      }
    float alpha[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
      const float m_new = fmaxf(m_run[i], mx[i]);
      alpha[i] = exp2f(m_run[i] - m_new);
      m_run[i] = m_new;
      l_run[i] *= alpha[i];
    }
#pragma unroll
    for (int nb = 0; nb < kBN / 8; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float pe = exp2f(s[nb][e] - m_run[e >> 1]);
        s[nb][e] = pe;
        l_run[e >> 1] += pe;
      }
#pragma unroll
    for (int nb = 0; nb < D / 8; ++nb) {
      o[nb][0] *= alpha[0];
      o[nb][1] *= alpha[0];
      o[nb][2] *= alpha[1];
      o[nb][3] *= alpha[1];
    }
    // O += P V
#pragma unroll
    for (int kb = 0; kb < kBN / 16; ++kb) {
      uint32_t a[4];
      a[0] = pack_bf16(s[2 * kb][0], s[2 * kb][1]);
      a[1] = pack_bf16(s[2 * kb][2], s[2 * kb][3]);
      a[2] = pack_bf16(s[2 * kb + 1][0], s[2 * kb + 1][1]);
      a[3] = pack_bf16(s[2 * kb + 1][2], s[2 * kb + 1][3]);
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        uint32_t bb[4];
        ldsm_x4_t(bb, tile_addr<D>(sV(st), kb * 16 + ((lane >> 3) & 1) * 8 + (lane & 7), 2 * np + (lane >> 4)));
        mma_bf16(o[2 * np], a, bb[0], bb[1]);
        mma_bf16(o[2 * np + 1], a, bb[2], bb[3]);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  // Epilogue: normalise, write O (bf16, [B, L, Hq, D]) and the natural-log LSE.
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], 1);
    l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], 2);
  }
  auto* out = static_cast<__nv_bfloat16*>(p.o);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = row0 + 8 * i;
    if (r >= p.L) continue;
    const float inv = 1.f / l_run[i];
    __nv_bfloat16* orow = out + ((static_cast<long long>(b) * p.L + r) * p.Hq + h) * D;
#pragma unroll
    for (int nb = 0; nb < D / 8; ++nb) {
      *reinterpret_cast<__nv_bfloat162*>(orow + nb * 8 + 2 * t) =
          __floats2bfloat162_rn(o[nb][2 * i] * inv, o[nb][2 * i + 1] * inv);
    }
    if (p.lse != nullptr && t == 0)
      p.lse[(static_cast<long long>(b) * p.Hq + h) * p.L + r] =
          (m_run[i] + log2f(l_run[i])) * 0.69314718055994531f;
  }
}

}  // namespace

cudaError_t launch_prefill_attention(const PrefillArgs& a, cudaStream_t stream) {
  const int nqt = (a.L + kBM - 1) / kBM;
  const dim3 grid(nqt, a.Hq, a.B), block(kWarps * 32);
  if (a.d == 128) {
    const int smem = 8 * kBM * 128 * 2;
    cudaFuncSetAttribute(prefill_mma_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    prefill_mma_kernel<128><<<grid, block, smem, stream>>>(a);
  } else if (a.d == 64) {
    const int smem = 8 * kBM * 64 * 2;
    cudaFuncSetAttribute(prefill_mma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    prefill_mma_kernel<64><<<grid, block, smem, stream>>>(a);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace jl
