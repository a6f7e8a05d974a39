"""Host checks of the integer partitions the kernels use (``csrc/partition.h``),
compiled with the host C++ compiler (no GPU):

* o_proj's rows over its CTAs: the shares tile [0, hidden) in CTA order, each
  row exactly once, for even splits and for a grid whose first CTAs take a
  larger share, the shapes the batch-1 launcher makes included;
* the cluster merge of decode attention: every output unit has exactly one
  owner, each rank owns a contiguous range, the senders' slots fit the
  receive area, and the bytes a rank receives equal what its merge barrier
  expects (the kernel's expect-tx count).
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "decode_attention_block_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <initializer_list>
#include "partition.h"
using namespace spark;

static int fails = 0;
#define CHECK(c, ...) do { if (!(c)) { std::printf(__VA_ARGS__); std::printf("\n"); ++fails; } } while (0)

static void check_share(int hidden, int grid, int early, int early_rows) {
  int next = 0;
  for (int i = 0; i < grid; ++i) {
    int r0, r1;
    oproj_share(hidden, grid, early, early_rows, i, r0, r1);
    CHECK(r0 == next && r1 >= r0 && r1 <= hidden, "share hidden %d grid %d early %d x %d: CTA %d [%d, %d) after %d",
          hidden, grid, early, early_rows, i, r0, r1, next);
    if (early > 0 && early < grid && i < early)
      CHECK(r1 - r0 == early_rows, "early CTA %d holds %d rows, not %d", i, r1 - r0, early_rows);
    next = r1;
  }
  CHECK(next == hidden, "share hidden %d grid %d early %d x %d ends at %d", hidden, grid, early, early_rows, next);
}

int main() {
  // even splits
  for (int hidden : {1, 7, 100, 2560, 4096})
    for (int grid = 1; grid <= 160; ++grid)
      if (grid <= hidden) check_share(hidden, grid, 0, 0);
  // the first CTAs with a larger share (the batch-1 launcher: 152 SMs, the
  // free ones taking up to 25 rows of 2560)
  for (int grid : {2, 64, 152})
    for (int early = 1; early < grid; ++early)
      for (int rows : {1, 3, 17, 25, 32})
        if ((long)early * rows <= 2560) check_share(2560, grid, early, rows);
  check_share(2560, 152, 88, 25);
  // the cluster merge
  CHECK(merge_recv_bytes_max() % 16 == 0, "receive area not 16-byte sized");
  for (int cl = 1; cl <= kMergeMaxCluster; ++cl) {
    const int sf = merge_slot_floats(cl);
    CHECK(sf % 4 == 0, "cl %d: slot of %d floats breaks float4 alignment", cl, sf);
    if (cl >= 2) CHECK(cl * sf * 4 <= merge_recv_bytes_max(), "cl %d: slots exceed the receive area", cl);
    int got[kMergeMaxCluster] = {0};
    for (int u = 0; u < kMergeUnits; ++u) {
      const int q = merge_owner(u, cl);
      CHECK(q >= 0 && q < cl && merge_unit0(q, cl) <= u && u < merge_unit0(q + 1, cl),
            "cl %d: unit %d owner %d", cl, u, q);
      for (int r = 0; r < cl; ++r)  // sender r's unit u lands in q's slot r
        if (r != q) {
          const int off = r * sf + 8 + 8 * (u - merge_unit0(q, cl));
          CHECK(off + 8 <= cl * sf, "cl %d: unit %d from %d past the slots", cl, u, r);
          got[q] += 32;
        }
    }
    for (int q = 0; q < cl; ++q) {
      const int units = merge_unit0(q + 1, cl) - merge_unit0(q, cl);
      CHECK(units >= 1 && 8 + 8 * units <= sf, "cl %d: rank %d owns %d units", cl, q, units);
      got[q] += 32 * (cl - 1);  // m and l from every other rank
      CHECK(got[q] == (cl - 1) * 32 * (1 + units), "cl %d: rank %d receives %d bytes, expects %d", cl, q, got[q],
            (cl - 1) * 32 * (1 + units));
    }
    CHECK(merge_unit0(0, cl) == 0 && merge_unit0(cl, cl) == kMergeUnits, "cl %d: units not covered", cl);
  }
  std::printf("%d failures\n", fails);
  return fails != 0;
}
"""


def test_partitions_cover_every_row_and_unit_once(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    src = tmp_path / "partition_check.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "partition_check"
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True)
    assert res.returncode == 0, res.stdout + res.stderr
    assert res.stdout.strip().endswith("0 failures")
