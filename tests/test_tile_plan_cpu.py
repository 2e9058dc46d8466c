"""The GEMM schedule planner (flce_plan_tiles), on the CPU.

The expected plans are derived by hand from the stated policy; each case gives the
derivation.  GB300 holds 76 CTA pairs at once (one pair per cluster), tiles are
256 x 256, and the square side of a resident set of 76 tiles is 8 (8^2 <= 76 < 9^2).
- Raster groups keep the revisited operand's panels within 40 MiB of L2.
- When fewer panels than the square side fit that budget (and fewer than the fast
  dimension has), the group is that square side (capped at the fast dimension) and
  both operands take the normal L2 policy.
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
    # Llama-3 head forward: 32 x 501 tiles, M fastest, hidden panels 256 x 4096 x 2 B =
    # 2 MiB: 20 fit 40 MiB, fewer than the 32 M tiles but not fewer than the square
    # side 8 -> group 20, hints kept.
    ("llama3_forward", (32, 501, 0, 2 * MiB, EVICT_LAST, NORMAL), (20, EVICT_LAST, NORMAL)),
    # Llama-3-shaped dlogits over a 65536-column vocabulary chunk: 32 x 256 tiles, same
    # panels -> 20.
    ("llama3_dlogits", (32, 256, 0, 2 * MiB, EVICT_LAST, NORMAL), (20, EVICT_LAST, NORMAL)),
    # Llama-3 dweight [H,V], first chunk: 16 x 256 tiles, hidden^T panels 256 x 8192 x
    # 2 B = 4 MiB: 10 fit, >= 8 -> group 10, hints kept.
    ("llama3_dweight", (16, 256, 0, 4 * MiB, EVICT_LAST, NORMAL), (10, EVICT_LAST, NORMAL)),
    # Llama-3 dhidden, first chunk: 32 x 16 tiles, N fastest, weight panels 256 x 65536 x
    # 2 B = 32 MiB: one fits, fewer than 8 and than the 16 N tiles -> lockstep group 8,
    # normal hints.
    ("llama3_dhidden", (32, 16, 1, 32 * MiB, NORMAL, EVICT_LAST), (8, NORMAL, NORMAL)),
    # Gemma-2 dweight [H,V], first 131072-column chunk: 9 x 512 tiles, M fastest, panels
    # 256 x 4096 x 2 B = 2 MiB: 20 fit, capped at the 9 M tiles.
    ("gemma_dweight", (9, 512, 0, 2 * MiB, EVICT_LAST, NORMAL), (9, EVICT_LAST, NORMAL)),
    # Small odd counts: 40 panels fit, capped at the 3 M tiles.
    ("odd_counts", (3, 5, 0, 1 * MiB, NORMAL, NORMAL), (3, NORMAL, NORMAL)),
    # One tile.
    ("single_tile", (1, 1, 0, 1 * MiB, NORMAL, NORMAL), (1, NORMAL, NORMAL)),
    # N fastest over 76 tiles with 1 MiB panels: 40 fit, >= 8 -> group 40.
    ("wide_fast_dimension", (2, 76, 1, 1 * MiB, NORMAL, NORMAL), (40, NORMAL, NORMAL)),
    # 40 MiB panels: one fits, fewer than the square side and than the 3 fast tiles ->
    # the square side capped at the fast dimension, 3; normal hints.
    ("few_fast_tiles", (4, 3, 1, 40 * MiB, NORMAL, EVICT_LAST), (3, NORMAL, NORMAL)),
    # No revisited operand (panel 0): one group over the whole fast dimension.
    ("no_panel", (32, 501, 0, 0, EVICT_LAST, NORMAL), (32, EVICT_LAST, NORMAL)),
]


@pytest.mark.parametrize("name,args,want", CASES, ids=[c[0] for c in CASES])
def test_plan_matches_the_policy(name, args, want):
    m, n, raster, panel, ah, bh = args
    assert B.plan_tiles(m, n, raster, panel, ah, bh, 76) == want


def test_plan_with_one_pair_keeps_the_budget_group():
    # one resident pair: the square side is 1, never above the budget group, so the
    # budget group (1 here) and the requested hints stand
    assert B.plan_tiles(32, 16, 1, 32 * MiB, NORMAL, EVICT_LAST, 1) == (1, NORMAL, EVICT_LAST)


@pytest.mark.parametrize("bad", [dict(m=0), dict(n=0), dict(raster=2), dict(ah=3), dict(pairs=0)])
def test_plan_rejects_bad_arguments(bad):
    a = dict(m=4, n=4, raster=0, ah=0, pairs=76)
    a.update(bad)
    with pytest.raises(B.FlceError) as ei:
        B.plan_tiles(a["m"], a["n"], a["raster"], MiB, a["ah"], 0, a["pairs"])
    assert ei.value.code == 1


TILE_ORDER_CHECK = r"""
#include <cstdio>
#include <vector>
#include "flce_gemm.cuh"
using namespace flce;

// Every output tile is visited exactly once over the schedule's tile indices.
static int check(int m, int n, int raster, int group) {
  GemmShape sh{};
  sh.m_tiles = m; sh.n_tiles = n; sh.raster = raster; sh.group = group;
  const int total = m * n;
  std::vector<int> hits(static_cast<size_t>(m) * n, 0);
  for (int t = 0; t < total; ++t) {
    int mt, nt;
    tile_coords(t, sh, mt, nt);
    if (mt < 0 || nt < 0 || mt >= m || nt >= n) return 1;
    ++hits[static_cast<size_t>(mt) * n + nt];
  }
  for (int h : hits)
    if (h != 1) return 2;
  return 0;
}

int main() {
  const int dims[] = {1, 2, 3, 5, 8, 13, 16, 32, 37};
  const int groups[] = {1, 2, 3, 6, 8, 10, 1 << 30};
  long cases = 0;
  for (int m : dims)
    for (int n : dims)
      for (int raster = 0; raster < 2; ++raster)
        for (int g : groups) {
          const int rc = check(m, n, raster, g);
          if (rc) {
            std::printf("FAIL %d m=%d n=%d raster=%d group=%d\\n", rc, m, n, raster, g);
            return 1;
          }
          ++cases;
        }
  std::printf("OK %ld\\n", cases);
  return 0;
}
"""


def test_tile_order_covers_every_tile_once(tmp_path):
    """The persistent schedule's tile order (tile_coords, compiled for the host with
    nvcc): every output tile exactly once for every raster and group choice,
    including ragged groups."""
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


DESC_CHECK = r"""
#include <cstdio>
#include "flce_gemm.cuh"
using namespace flce;

// The UMMA thread builds each stage's descriptors by adding (stage bytes >> 4) and
// (k-slice offset >> 4) to the stage-0, k-slice-0 descriptor: that must equal building
// them from the addresses, for every stage and k-slice, at every shared-memory base the
// kernel's operand rings can have (1 KB aligned, the ring inside the 2^18-byte window).
template <bool MN, int BYTES>
static int check(const GemmShape& sh) {
  constexpr int STAGES = PairCfg<256, 4>::STAGES;
  constexpr uint64_t kK = (MN ? UK * 128 : UK * 2) >> 4;
  for (uint32_t base = 0; base + STAGES * BYTES <= (1u << 18); base += 1024) {
    const uint64_t d0 = operand_desc<MN>(base, 0, sh);
    for (int s = 0; s < STAGES; ++s)
      for (int kk = 0; kk < BK / UK; ++kk)
        if (operand_desc<MN>(base + s * BYTES, kk, sh) !=
            d0 + static_cast<uint64_t>(s) * (BYTES >> 4) + kk * kK)
          return 1;
  }
  return 0;
}

int main() {
  GemmShape sh{};
  sh.mn_lbo = MN_ATOM_BYTES;
  sh.mn_sbo = 1024;
  using C = PairCfg<256, 4>;
  const int rc = check<false, C::A_BYTES>(sh) | check<true, C::A_BYTES>(sh) |
                 check<false, C::B_BYTES>(sh) | check<true, C::B_BYTES>(sh);
  std::printf(rc ? "FAIL\n" : "OK\n");
  return rc;
}
"""


def test_incremental_descriptors_equal_rebuilt_ones(tmp_path):
    """The shared-memory descriptors the UMMA thread advances by stage and k-slice equal
    the ones built from the operand addresses (compiled for the host with nvcc)."""
    import os
    import subprocess
    from linear_cross_entropy_forward_gb300.build import CSRC, ROOT, nvcc_path
    try:
        nvcc = nvcc_path()
    except RuntimeError:
        pytest.skip("nvcc not available")
    src = tmp_path / "desc_check.cu"
    src.write_text(DESC_CHECK)
    exe = tmp_path / "desc_check"
    r = subprocess.run([nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
                        "-I" + CSRC, "-I" + os.path.join(ROOT, "include"), str(src), "-o",
                        str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.startswith("OK"), out.stdout + out.stderr
