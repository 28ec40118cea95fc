"""Host check of the update kernel's operand tile layout (optile_idx in common.cuh).

The tf32 halves of U, Vbar and W are stored as the shared-memory image of the
update's 128 x 16 K-major operand tiles so that one tile is one contiguous bulk
copy.  Every writer (the streaming kernel's drain, the W reduction, the split
kernel) and the reader agree through optile_idx alone; this test compiles that
function for the host and checks the properties the kernels rely on: a
permutation of the padded buffer, tiles contiguous, 16-byte groups kept together
and aligned, and the 64-byte swizzle inside a tile (row r at 64 r bytes, its
16-byte piece q at q ^ ((r / 2) mod 4)), which is the layout the MMA's
shared-memory descriptor reads.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "..", "rank_orthonormalized_optimizer_03_b300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <vector>
#include "common.cuh"
using dion::optile_idx;
int check(long long rows, long long rp) {
  const long long padded = (rows + 127) / 128 * 128;
  std::vector<int> seen(padded * rp, 0);
  for (long long row = 0; row < padded; ++row)
    for (long long k = 0; k < rp; ++k) {
      const long long o = optile_idx(row, k, rp);
      if (o < 0 || o >= padded * rp) { printf("out of range %lld %lld\n", row, k); return 1; }
      if (seen[o]++) { printf("collision %lld %lld\n", row, k); return 1; }
      // the tile of (row, k) is the contiguous block t * 2048 .. t * 2048 + 2047
      const long long t = (row / 128) * (rp / 16) + k / 16;
      if (o / 2048 != t) { printf("tile %lld %lld\n", row, k); return 1; }
      // 64-byte swizzle inside the tile
      const long long r = row % 128, kk = k % 16, q = kk / 4;
      const long long bytes = r * 64 + ((q ^ ((r >> 1) & 3)) << 4) + 4 * (kk & 3);
      if ((o - t * 2048) * 4 != bytes) { printf("swizzle %lld %lld\n", row, k); return 1; }
      // a group of four consecutive k (k % 4 == 0) is one aligned 16-byte piece
      if (k % 4 == 0) {
        if (o % 4) { printf("alignment %lld %lld\n", row, k); return 1; }
        for (int e = 1; e < 4; ++e)
          if (optile_idx(row, k + e, rp) != o + e) { printf("group %lld %lld\n", row, k); return 1; }
      }
    }
  return 0;
}
int main() {
  const long long cases[][2] = {{128, 32}, {256, 192}, {300, 64}, {1000, 256}, {129, 768}};
  for (auto& c : cases)
    if (check(c[0], c[1])) return 1;
  printf("ok\n");
  return 0;
}
"""


def _nvcc():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


def test_operand_tile_layout(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not available")
    src = tmp_path / "layout.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "layout"
    res = subprocess.run([nvcc, "-std=c++17", "-O1", "-I", CSRC, "-o", str(exe), str(src)],
                         capture_output=True, text=True)
    assert res.returncode == 0, res.stderr[-2000:]
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.strip().endswith("ok"), run.stdout + run.stderr
