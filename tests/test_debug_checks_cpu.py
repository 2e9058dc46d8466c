"""The in-kernel bounds checks of the FLCE_DEBUG build, on the CPU.

The predicates the debug kernels call before every TMA load and epilogue store are
plain host/device functions (csrc/flce_check.cuh).  Here they are compiled for the
host with nvcc and run on accesses the GEMMs make -- which must pass -- and on
planted mistakes -- which must fail: a box a whole tile past the padded edge, a
negative coordinate, an x off the 16-byte grid, a store run past its row, a part
index past the statistics arrays, a TMEM read from another warp's lane quadrant.
The debug library itself must load without a GPU and export the same C ABI.
"""
import ctypes
import os
import subprocess

import pytest

from linear_cross_entropy_forward_gb300 import _binding as B

CHECK = r"""
#include <cstdio>
#include "flce_check.cuh"
using namespace flce;

static int fails = 0;
#define EXPECT(c) do { if (!(c)) { std::printf("FAIL line %d: %s\n", __LINE__, #c); ++fails; } } while (0)

int main() {
  // Llama-3 head forward, hidden [8192, 4096] K-major: k blocks of 64, pair rows of 256
  EXPECT(tma_box_ok(0, 0, 4096, 8192));
  EXPECT(tma_box_ok(4096 - 64, 8192 - 64, 4096, 8192));
  // ragged N = 300: the peer CTA of the last pair starts at row 384 (zero fill), legal
  EXPECT(tma_box_ok(0, 384 + 64, 200, 300));
  // weight [H=4096, V=128100] MN-major: the last n-tile's second half starts at
  // column 128192, past V (zero fill), still inside the padded 128256
  EXPECT(tma_box_ok(128000 + 128 + 64, 4032, 128100, 4096));
  // planted mistakes
  EXPECT(!tma_box_ok(0, 512, 200, 300));          // a whole pair tile past the padded rows
  EXPECT(!tma_box_ok(-64, 0, 4096, 8192));        // negative x
  EXPECT(!tma_box_ok(0, -1, 4096, 8192));         // negative y
  EXPECT(!tma_box_ok(4, 0, 4096, 8192));          // x off the 16-byte grid
  EXPECT(!tma_box_ok(128256 + 256, 0, 128256, 4096));
  // epilogue stores: a chunk of 32 columns inside a row of the dlogits chunk
  EXPECT(row_run_ok(65536 - 32, 32, 65536));
  EXPECT(!row_run_ok(65536 - 16, 32, 65536));     // runs past the row
  EXPECT(!row_run_ok(-8, 8, 64));
  EXPECT(index_ok(500, 501) && !index_ok(501, 501) && !index_ok(-1, 501));
  // TMEM: two 256-column accumulators, warp 5 reads quadrant 1
  EXPECT(tmem_ok(256 + 128, 128, 1, 5));
  EXPECT(!tmem_ok(256 + 256, 32, 1, 5));          // past the 512 allocated columns
  EXPECT(!tmem_ok(0, 32, 2, 5));                  // another warp's lane quadrant
  if (fails) return 1;
  std::printf("OK\n");
  return 0;
}
"""


def test_bounds_predicates_pass_real_accesses_and_fail_planted_mistakes(tmp_path):
    from linear_cross_entropy_forward_gb300.build import CSRC, nvcc_path
    try:
        nvcc = nvcc_path()
    except RuntimeError:
        pytest.skip("nvcc not available")
    src = tmp_path / "check.cu"
    src.write_text(CHECK)
    exe = tmp_path / "check"
    r = subprocess.run([nvcc, "-std=c++17", "-I" + CSRC, str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0 and out.stdout.startswith("OK"), out.stdout + out.stderr


def test_debug_library_builds_and_exports_the_same_abi():
    from linear_cross_entropy_forward_gb300.build import DEBUG_LIB_PATH, build
    path = build(debug=True)
    assert path == DEBUG_LIB_PATH and os.path.exists(path)
    lib = ctypes.CDLL(path)
    for name in B.EXPORTED:
        assert hasattr(lib, name), name
    lib.flce_strerror.restype = ctypes.c_char_p
    assert b"bounds" in lib.flce_strerror(10)
