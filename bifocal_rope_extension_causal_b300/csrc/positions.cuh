// Position mapping of dynamic bifocal RoPE, in one place for host and device.
//
// "Jet-Long: Efficient Long-Context Extension with Dynamic Bifocal RoPE",
// paper digest page, section "Method": the bifocal score routes a pair by its
// distance q - k against the local window w0 (Eq. 1); remote pairs use the
// aliased positions f(x) = floor(x / G) with G = max(1, ceil(L / w_pretrained))
// (Eqs. 2-3); the KV-cache correction uses Delta(x) = f(x) - x.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define JL_HD __host__ __device__ __forceinline__
#else
#define JL_HD inline
#endif

namespace jl {

// G = max(1, ceil(L / w_pretrained)) for L >= 0, w_pretrained >= 1.
JL_HD int64_t group_size(int64_t L, int64_t w_pretrained) {
  return L <= 0 ? 1 : (L + w_pretrained - 1) / w_pretrained;
}

// f(x) = floor(x / G); positions are non-negative so C division is floor.
JL_HD int alias(int x, int G) { return x / G; }

// Delta(x) = f(x) - x <= 0.
JL_HD int alias_offset(int x, int G) { return x / G - x; }

// Eq. 1 routing: q - k == w0 is still local.
JL_HD bool is_local(int qpos, int kpos, int w0) { return qpos - kpos <= w0; }

// Routing class of a (query tile, key tile) block of the causal score matrix.
enum TileClass : int {
  kTileSkip = 0,      // every key after every query: fully masked
  kTileLocal = 1,     // every causal pair has q - k <= w0
  kTileRemote = 2,    // every pair has q - k > w0
  kTileStraddle = 3,  // both kinds: both score sets, select per element
};

// Query rows [q0, q0 + bm), key columns [k0, k0 + bn).
JL_HD int classify_tile(int q0, int bm, int k0, int bn, int w0) {
  const int dmax = (q0 + bm - 1) - k0;  // largest q - k in the block
  const int dmin = q0 - (k0 + bn - 1);  // smallest q - k in the block
  if (dmax < 0) return kTileSkip;
  if (dmax <= w0) return kTileLocal;
  if (dmin > w0) return kTileRemote;
  return kTileStraddle;
}

// Does the block contain pairs with k > q (needs the causal mask)?
JL_HD bool tile_needs_causal_mask(int q0, int k0, int bn) { return k0 + bn - 1 > q0; }

}  // namespace jl
