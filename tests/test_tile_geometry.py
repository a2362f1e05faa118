"""CPU: the tile-geometry header compiled as host C++ and checked by brute force.

The kernels and the host planner share pa_tiles.cuh.  This test compiles it
with g++ (no CUDA needed) and checks, over many unit positions, window and
sink sizes and sequence layouts: that the tiles of every unit visit exactly
the key blocks some row of the unit sees under the sink/window mask, each
once; that `needs_mask` is set exactly where some row of the unit misses some
key of the tile; that `visible_columns` matches the mask key by key; and that
the cheap `tile_width` used by the MMA issuer equals `tile_geom`'s width.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "..", "windowed_prefill_attention_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <cstdlib>
#include <initializer_list>
#include "pa_tiles.cuh"
using namespace pa;
// the mask, written out: key j visible to query token t
static bool sees(int t, int j, int S, int W) {
  if (j > t) return false;
  if (W <= 0) return true;
  const int lo = imax(0, t / kPage + 1 - W);
  return j / kPage < S || j / kPage >= lo;
}
int main() {
  long checked = 0;
  for (int G : {1, 2, 4, 8, 16}) for (int TQ : {kRows / G, kUnitRows / G}) {
    for (int S : {0, 1, 2, 5}) for (int W : {0, 1, 3, 4, 7, 16}) for (int q_start : {0, 5, 48, 300}) for (int n_q : {1, 17, 130, 333}) {
      SeqGeom sg{};
      sg.q_start = q_start; sg.n_q = n_q; sg.n_ctx = q_start + n_q;
      seq_geom_fill(sg, S, W);
      for (int t0 = (q_start / TQ) * TQ; t0 < q_start + n_q; t0 += TQ) {
        const UnitGeom u = unit_geom(t0, TQ, sg, S, W);
        const int ta = imax(t0, q_start), tb = imin(t0 + TQ, q_start + n_q) - 1;
        const int nkb = u.qb + 1;
        int* visits = (int*)calloc(nkb, sizeof(int));
        for (int i = 0; i < u.n_tiles; ++i) {
          const TileGeom tg = tile_geom(u, i, S, W);
          if (tile_width(u, i) != tg.nb || tg.nb < 1 || tg.nb > kTileBlocks) { printf("FAIL width %d %d\n", tile_width(u, i), tg.nb); return 1; }
          bool any_hidden = false;
          for (int b = tg.kb0; b < tg.kb0 + tg.nb; ++b) ++visits[b];
          for (int t = ta; t <= tb; ++t) {
            const unsigned long long vh[2] = {visible_columns(tg, t, S, W, 0), visible_columns(tg, t, S, W, 1)};
            for (int c = 0; c < kTileKeys; ++c) {
              const unsigned long long v = vh[c / 64];
              const int j = tg.kb0 * kPage + c;
              const bool in_tile = c < tg.nb * kPage;
              const bool want = in_tile && sees(t, j, S, W);
              if (in_tile && !sees(t, j, S, W)) any_hidden = true;
              const bool got = (v >> (c % 64)) & 1ull;
              if (tg.needs_mask && got != want) { printf("FAIL cols t=%d j=%d\n", t, j); return 1; }
              if (!tg.needs_mask && in_tile && !want) { printf("FAIL unmasked t=%d j=%d\n", t, j); return 1; }
              ++checked;
            }
          }
          if (any_hidden != tg.needs_mask) { printf("FAIL needs_mask %d %d\n", (int)any_hidden, (int)tg.needs_mask); return 1; }
        }
        for (int b = 0; b < nkb; ++b) {
          bool seen = false;
          for (int t = ta; t <= tb && !seen; ++t)
            for (int j = b * kPage; j < (b + 1) * kPage && !seen; ++j) seen = sees(t, j, S, W);
          if (visits[b] != (seen ? 1 : 0)) { printf("FAIL visits b=%d %d %d\n", b, visits[b], (int)seen); return 1; }
        }
        free(visits);
      }
    }
  }
  printf("OK %ld\n", checked);
  return 0;
}
"""


def test_tile_geometry_against_the_mask(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    src = tmp_path / "geom.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "geom"
    subprocess.run([gxx, "-O2", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0 and out.stdout.startswith("OK"), out.stdout + out.stderr
