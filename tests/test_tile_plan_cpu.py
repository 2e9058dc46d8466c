"""The GEMM schedule planner (flce_plan_tiles), on the CPU.

The expected plans are derived by hand from the stated policy; each case gives the
derivation. GB300 holds 36 clusters of four CTAs or 76 CTA pairs at once, and tiles
are 256 x 256.
- Two pairs share an operand along an even tile dimension (else along the longer one)
  unless that needs more than 6 % more rounds of tiles.
- Raster groups keep the revisited operand's panels within 40 MiB of L2.
- When fewer panels than a square-ish resident set fit that budget, the group is that
  square (side g with g^2 <= capacity) and both operands take the normal L2 policy.
"""
import pytest

from linear_cross_entropy_forward_gb300 import _binding as B

MiB = 1 << 20
NORMAL, EVICT_FIRST, EVICT_LAST = 0, 1, 2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from linear_cross_entropy_forward_gb300.build import build
    build()


CASES = [
    # Llama-3 head forward: 32 x 501 tiles, hidden panels 256 x 4096 x 2 B = 2 MiB.
    # M even -> share B; 8016 cluster tiles take ceil(8016/36) = 223 rounds against
    # ceil(16032/76) = 211 for pairs: 223 <= 1.06 * 211, so share.  A shared panel is
    # 4 MiB: 10 fit 40 MiB, >= the square side 6 (36 clusters) -> group 10, hints kept.
    ("llama3_forward", (32, 501, 0, 2 * MiB, 256, EVICT_LAST, NORMAL), (1, 10, EVICT_LAST, NORMAL)),
    # Llama-3 dlogits, first 65536-column chunk: 32 x 256 tiles; 114 rounds against 108
    # (<= 6 % more) -> share; group 10 as above.
    ("llama3_dlogits", (32, 256, 0, 2 * MiB, 256, EVICT_LAST, NORMAL), (1, 10, EVICT_LAST, NORMAL)),
    # Llama-3 dweight [H,V], first chunk: 16 x 256 tiles, hidden^T panels 256 x 8192 x 2 B =
    # 4 MiB; 57 rounds against 54 -> share.  Shared panels of 8 MiB: 5 fit, fewer than
    # the square side 6 and than the 8 fast cluster tiles -> lockstep group 6, normal hints.
    ("llama3_dweight", (16, 256, 0, 4 * MiB, 256, EVICT_LAST, NORMAL), (1, 6, NORMAL, NORMAL)),
    # Llama-3 dhidden, first chunk: 32 x 16 tiles, N fastest, weight panels 256 x 65536 x
    # 2 B = 32 MiB.  Sharing: 8 rounds of clusters against 7 of pairs (+14 %) -> none.
    # One panel fits; square side for 76 pairs is 8 -> lockstep group 8, normal hints.
    ("llama3_dhidden", (32, 16, 1, 32 * MiB, 256, NORMAL, EVICT_LAST), (0, 8, NORMAL, NORMAL)),
    # Gemma-2 dweight [H,V], first 131072-column chunk: 9 x 512 tiles.  M odd, N even ->
    # share A along N; 64 rounds against 61 (<= 6 %).  The fast M dimension is not the
    # shared one: panels 256 x 4096 x 2 B = 2 MiB, 20 fit, capped at the 9 M tiles.
    ("gemma_dweight", (9, 512, 0, 2 * MiB, 256, EVICT_LAST, NORMAL), (2, 9, EVICT_LAST, NORMAL)),
    # Both counts odd: share along the longer dimension (N); 1 round either way.
    ("odd_counts", (3, 5, 0, 1 * MiB, 256, NORMAL, NORMAL), (2, 3, NORMAL, NORMAL)),
    # One tile: nothing to share.
    ("single_tile", (1, 1, 0, 1 * MiB, 256, NORMAL, NORMAL), (0, 1, NORMAL, NORMAL)),
    # 2 x 76 tiles: 2 rounds of pairs against 3 of clusters (+50 %) -> no sharing.
    ("quantised", (2, 76, 1, 1 * MiB, 256, NORMAL, NORMAL), (0, 40, NORMAL, NORMAL)),
    # 128-column tiles never share (clusters of four are built for 256-column tiles).
    ("narrow_tiles", (32, 64, 0, 1 * MiB, 128, NORMAL, NORMAL), (0, 32, NORMAL, NORMAL)),
]


@pytest.mark.parametrize("name,args,want", CASES, ids=[c[0] for c in CASES])
def test_plan_matches_the_policy(name, args, want):
    m, n, raster, panel, tn, ah, bh = args
    assert B.plan_tiles(m, n, raster, panel, tn, ah, bh, 36, 76) == want


def test_plan_without_clusters_of_four_never_shares():
    # a GPU that fits no cluster of four (capacity 0) keeps one pair per cluster
    assert B.plan_tiles(32, 501, 0, 2 * MiB, 256, EVICT_LAST, NORMAL, 0, 76)[0] == 0


@pytest.mark.parametrize("bad", [dict(m=0), dict(n=0), dict(raster=2), dict(ah=3), dict(c2=0)])
def test_plan_rejects_bad_arguments(bad):
    a = dict(m=4, n=4, raster=0, ah=0, c2=76)
    a.update(bad)
    with pytest.raises(B.FlceError) as ei:
        B.plan_tiles(a["m"], a["n"], a["raster"], MiB, 256, a["ah"], 0, 36, a["c2"])
    assert ei.value.code == 1


TILE_ORDER_CHECK = r"""
#include <cstdio>
#include <vector>
#include "flce_gemm.cuh"
using namespace flce;

// Every output tile is visited exactly once over all cluster tiles and pairs; a tile
// past the end appears only for the spare half of a cluster tile along an odd shared
// dimension.
static int check(int m, int n, int share, int raster, int group) {
  GemmShape sh{};
  sh.m_tiles = m; sh.n_tiles = n; sh.share = share; sh.raster = raster; sh.group = group;
  const int total = cluster_m_tiles(sh) * cluster_n_tiles(sh);
  const int pairs = share ? 2 : 1;
  std::vector<int> hits(static_cast<size_t>(m) * n, 0);
  int spare = 0;
  for (int t = 0; t < total; ++t)
    for (int p = 0; p < pairs; ++p) {
      int mt, nt;
      tile_coords(t, sh, p, mt, nt);
      if (mt < 0 || nt < 0) return 1;
      if (mt >= m || nt >= n) {
        const bool ok = (share == 1 && (m & 1) && mt == m && nt < n) ||
                        (share == 2 && (n & 1) && nt == n && mt < m);
        if (!ok) return 2;
        ++spare;
        continue;
      }
      ++hits[static_cast<size_t>(mt) * n + nt];
    }
  for (int h : hits)
    if (h != 1) return 3;
  const int want_spare = share == 1 ? (m & 1) * n : share == 2 ? (n & 1) * m : 0;
  return spare == want_spare ? 0 : 4;
}

int main() {
  const int dims[] = {1, 2, 3, 5, 8, 13, 16, 32, 37};
  const int groups[] = {1, 2, 3, 6, 8, 10, 1 << 30};
  long cases = 0;
  for (int m : dims)
    for (int n : dims)
      for (int share = 0; share < 3; ++share)
        for (int raster = 0; raster < 2; ++raster)
          for (int g : groups) {
            const int rc = check(m, n, share, raster, g);
            if (rc) {
              std::printf("FAIL %d m=%d n=%d share=%d raster=%d group=%d\n", rc, m, n, share,
                          raster, g);
              return 1;
            }
            ++cases;
          }
  std::printf("OK %ld\n", cases);
  return 0;
}
"""


def test_tile_order_covers_every_tile_once(tmp_path):
    """The persistent schedule's tile order (tile_coords, compiled for the host with
    nvcc): every output tile exactly once for every share, raster and group choice,
    including ragged groups and odd shared dimensions."""
    import os
    import subprocess
    from linear_cross_entropy_forward_gb300.build import CSRC, ROOT, nvcc_path
    try:
        nvcc = nvcc_path()
    except RuntimeError:
        pytest.skip("nvcc not available")
    src = tmp_path / "tile_order_check.cu"
    src.write_text(TILE_ORDER_CHECK)
    exe = tmp_path / "tile_order_check"
    r = subprocess.run([nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
                        "-I" + CSRC, "-I" + os.path.join(ROOT, "include"), str(src), "-o",
                        str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.startswith("OK"), out.stdout + out.stderr
