// partition.h -- integer partitions shared by the kernels and their host
// launchers (plain C++: the host-side tests compile it without CUDA).
//   * o_proj's rows over its CTAs, when the first CTAs of the grid take a
//     larger share (they start on SMs the previous kernel leaves free);
//   * the cluster merge of decode attention: which rank owns which units of
//     a group's output and where the other ranks' slices land in its
//     shared memory.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define SPARK_HD __host__ __device__
#else
#define SPARK_HD
#endif

namespace spark {

// Rows [r0, r1) of `hidden` computed by CTA i of `grid`.  early > 0 (and
// early * early_rows <= hidden): the first `early` CTAs take early_rows
// rows each and the others share the remaining rows evenly; early == 0 or
// early >= grid: an even split.
SPARK_HD inline void oproj_share(int hidden, int grid, int early, int early_rows, int i, int& r0, int& r1) {
  if (early <= 0 || early >= grid) {
    r0 = (int)((int64_t)hidden * i / grid);
    r1 = (int)((int64_t)hidden * (i + 1) / grid);
    return;
  }
  if (i < early) {
    r0 = i * early_rows;
    r1 = r0 + early_rows;
    return;
  }
  const int base = early * early_rows, late = grid - early;
  r0 = base + (int)((int64_t)(hidden - base) * (i - early) / late);
  r1 = base + (int)((int64_t)(hidden - base) * (i - early + 1) / late);
}

// The cluster merge: a group's output o[4][256] is 128 units of 8 floats
// (one lane's dims of one head).  Rank r of a cluster of cl owns units
// [merge_unit0(r, cl), merge_unit0(r + 1, cl)); it receives from every other
// rank q, in slot q of its receive area (merge_slot_floats(cl) floats), that
// rank's m[4], l[4] and its values of the owned units.
constexpr int kMergeUnits = 128;
constexpr int kMergeMaxCluster = 16;

SPARK_HD constexpr int merge_unit0(int r, int cl) { return kMergeUnits * r / cl; }

SPARK_HD constexpr int merge_slot_floats(int cl) { return 8 + 8 * ((kMergeUnits + cl - 1) / cl); }

// the rank that owns unit u
SPARK_HD inline int merge_owner(int u, int cl) {
  int q = u * cl / kMergeUnits;
  while (q + 1 < cl && merge_unit0(q + 1, cl) <= u) ++q;
  while (merge_unit0(q, cl) > u) --q;
  return q;
}

// bytes of the receive area for any cluster of up to kMergeMaxCluster ranks
constexpr int merge_recv_bytes_max() {
  int most = 0;
  for (int cl = 2; cl <= kMergeMaxCluster; ++cl)
    if (cl * merge_slot_floats(cl) * 4 > most) most = cl * merge_slot_floats(cl) * 4;
  return most;
}

}  // namespace spark
