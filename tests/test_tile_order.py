"""The persistent GEMM's tile order (grouped rows, upper triangle for symmetric
products) must visit every output tile exactly once: the header's tile_coords
compiled for the host and checked for every grid up to 64 x 64 tiles (sides up
to 8192)."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r'''
#include <cstdio>
#include <set>
#include <utility>
#include "gemm_tc.cuh"
using namespace precond;
int main() {
  long bad = 0;
  for (int tm = 1; tm <= 64; ++tm)
    for (int tn = 1; tn <= 64; ++tn)
      for (int sym = 0; sym < 2; ++sym) {
        if (sym && tm != tn) continue;
        const int total = sym ? tn * (tn + 1) / 2 : tm * tn;
        std::set<std::pair<int, int>> seen;
        for (int t = 0; t < total; ++t) {
          int ti, tj;
          tile_coords(t, tm, tn, sym, ti, tj);
          if (ti < 0 || ti >= tm || tj < 0 || tj >= tn || (sym && ti > tj) || !seen.insert({ti, tj}).second) ++bad;
        }
        if ((int)seen.size() != total) ++bad;
      }
  printf("%ld\n", bad);
  return bad != 0;
}
'''


def test_tile_order_is_a_bijection():
    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else None)
    if nvcc is None:
        pytest.skip("nvcc not available")
    csrc = os.path.join(ROOT, "shampoo_roots_gb300", "csrc")
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "tile_order.cu")
        exe = os.path.join(d, "tile_order")
        with open(src, "w") as f:
            f.write(PROGRAM)
        subprocess.run([nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-I", csrc, "-o", exe, src],
                       check=True, capture_output=True)
        out = subprocess.run([exe], capture_output=True, text=True)
        assert out.returncode == 0 and out.stdout.strip() == "0", out.stdout
