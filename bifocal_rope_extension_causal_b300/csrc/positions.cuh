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

// Eq. 1 routing: a pair is local when q - k <= w0 (q - k == w0 is still
// local), remote otherwise.  Every local/remote decision of the kernels goes
// through the functions below.
JL_HD bool is_local(int qpos, int kpos, int w0) { return qpos - kpos <= w0; }

// For one query position the remote keys form a prefix: keys k >= the value
// below are local, earlier keys remote.
JL_HD int first_local_key(int qpos, int w0) { return qpos - w0; }

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

// Visit plan of query rows [q0, qlast] over key tiles of width bn: tiles
// 0 .. remote_tile_count - 1 hold a pair with q - k > w0 (for qlast; the
// caller caps the count at the causal limit), and tiles from
// first_local_tile on hold a pair with q - k <= w0 (for q0).
JL_HD int remote_tile_count(int qlast, int w0, int bn) {
  const int t = qlast - w0 - 1;  // tile j has a remote pair iff bn * j <= t
  return t >= 0 ? t / bn + 1 : 0;
}
JL_HD int first_local_tile(int q0, int w0, int bn) {
  const int u = q0 - (bn - 1) - w0;  // tile j has a local pair iff bn * j >= u
  return u <= 0 ? 0 : (u + bn - 1) / bn;
}

// A visit scores the block with one rotation and keeps only its own pairs:
// the remote visit needs a mask unless every pair is remote, the local
// visit unless every pair is local and causal.
JL_HD bool remote_visit_needs_mask(int q0, int bm, int k0, int bn, int w0) {
  return classify_tile(q0, bm, k0, bn, w0) != kTileRemote;
}
JL_HD bool local_visit_needs_mask(int q0, int bm, int k0, int bn, int w0) {
  return classify_tile(q0, bm, k0, bn, w0) != kTileLocal || tile_needs_causal_mask(q0, k0, bn);
}
JL_HD bool visit_keeps(bool remote_visit, int q, int k, int w0) {
  return remote_visit ? !is_local(q, k, w0) : (k <= q && is_local(q, k, w0));
}

}  // namespace jl
