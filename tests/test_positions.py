"""The position and routing helpers every kernel uses (csrc/positions.cuh),
compiled for the host with g++ and checked by brute force over small
shapes: the dynamic group size, the alias map, the tile classes and the
visit plan of the routed prefill (which key tiles get a remote and a local
visit, which visits need a mask, which pairs each visit keeps) must score
every causal pair exactly once, with the rotation Eq. 1 routes it to."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "bifocal_rope_extension_causal_b300", "csrc", "positions.cuh")

PROGRAM = r"""
#include <stdio.h>
#include "positions.cuh"
using namespace jl;
static int fails = 0;
#define CHECK(c) do { if (!(c)) { if (fails++ < 10) printf("fail line %d\n", __LINE__); } } while (0)
int main() {
  // G: smallest g >= 1 with (L - 1) / g < w
  for (int w = 1; w <= 40; ++w)
    for (int L = 0; L <= 300; ++L) {
      long long g = 1;
      if (L > 0) while ((L - 1) / g >= w) ++g;
      CHECK(group_size(L, w) == g);
    }
  for (int G = 1; G <= 9; ++G)
    for (int x = 0; x < 500; ++x) {
      CHECK(alias(x, G) * G <= x && x < (alias(x, G) + 1) * G);
      CHECK(alias_offset(x, G) == alias(x, G) - x);
    }
  // Visit plan of query rows [q0, qlast] over key tiles of width bn: each
  // causal pair is kept by exactly one visit, the remote visit iff
  // q - k > w0; visits that need no mask keep every pair of their block.
  const int bns[] = {4, 8, 16};
  for (int bn : bns)
    for (int w0 = 0; w0 <= 70; w0 += 3)
      for (int q0 = 0; q0 <= 96; q0 += bn) {
        const int bm = bn, qlast = q0 + 2 * bm - 1;
        const int jmax = qlast / bn;
        const int nr = remote_tile_count(qlast, w0, bn) < jmax + 1 ? remote_tile_count(qlast, w0, bn) : jmax + 1;
        const int jl0 = first_local_tile(q0, w0, bn);
        for (int q = q0; q <= qlast; ++q)
          for (int k = 0; k <= q; ++k) {
            const int j = k / bn;
            const bool remote_pair = !is_local(q, k, w0);
            CHECK(remote_pair == (q - k > w0));
            CHECK(is_local(q, k, w0) == (k >= first_local_key(q, w0)));
            int kept = 0;
            if (j < nr && visit_keeps(true, q, k, w0)) { ++kept; CHECK(remote_pair); }
            if (j >= jl0 && j <= jmax && visit_keeps(false, q, k, w0)) { ++kept; CHECK(!remote_pair); }
            CHECK(kept == 1);
          }
        // Tiles outside the plan hold no pair of that kind.
        for (int j = 0; j <= jmax; ++j)
          for (int q = q0; q <= qlast; ++q)
            for (int k = j * bn; k < (j + 1) * bn && k <= q; ++k) {
              if (j >= nr) CHECK(is_local(q, k, w0));
              if (j < jl0) CHECK(!is_local(q, k, w0));
            }
        // A visit that needs no mask keeps every pair of its block (per query tile).
        for (int t = 0; t < 2; ++t) {
          const int q0t = q0 + t * bm;
          for (int j = 0; j <= jmax; ++j) {
            const int k0 = j * bn;
            const int cls = classify_tile(q0t, bm, k0, bn, w0);
            bool any_remote = false, any_local = false, any_acausal = false;
            for (int q = q0t; q < q0t + bm; ++q)
              for (int k = k0; k < k0 + bn; ++k) {
                if (k > q) any_acausal = true;
                else if (is_local(q, k, w0)) any_local = true;
                else any_remote = true;
              }
            CHECK(cls == (!any_remote && !any_local ? kTileSkip
                          : any_remote && any_local ? kTileStraddle
                          : any_remote ? (any_acausal ? kTileStraddle : kTileRemote) : kTileLocal));
            if (!remote_visit_needs_mask(q0t, bm, k0, bn, w0)) CHECK(!any_local && !any_acausal);
            if (!local_visit_needs_mask(q0t, bm, k0, bn, w0)) CHECK(!any_remote && !any_acausal);
            CHECK(tile_needs_causal_mask(q0t, k0, bn) == any_acausal);
          }
        }
      }
  printf("%d failures\n", fails);
  return fails != 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_routing_helpers_brute_force(tmp_path):
    src = tmp_path / "positions_check.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "positions_check"
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout
