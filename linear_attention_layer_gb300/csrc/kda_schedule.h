// kda_schedule.h -- a host-built schedule of (sequence, head) units for the
// kernels whose CTAs walk a unit list (CTA b runs list[b], list[b + grid],
// ...): the units, longest first, each go to the CTA with the least work so
// far.  Dealing longest-first units round-robin instead leaves the busiest CTA
// several percent above the mean on a batch of mixed lengths.
#pragma once

#include <stdint.h>

#include <algorithm>
#include <functional>
#include <queue>
#include <utility>
#include <vector>

namespace kda {

// by_len: the sequences, longest first; cost(seq): the work of one of its
// units (> 0).  Writes list[k * grid + b] = seq * H + head for CTA b's k-th
// unit, -1 where a CTA has none, and returns the list length (a multiple of
// grid), or 0 when it would exceed cap (the caller keeps its plain order).
template <class Cost>
int build_unit_schedule(const std::vector<int>& by_len, int H, int grid, Cost cost, int* list,
                        int cap) {
  if (grid <= 0 || H <= 0) return 0;
  std::vector<std::vector<int>> mine(grid);
  using Slot = std::pair<long long, int>;  // (work so far, CTA)
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> least;
  for (int b = 0; b < grid; ++b) least.push({0, b});
  for (int seq : by_len) {
    const long long c = std::max<long long>(1, cost(seq));
    for (int h = 0; h < H; ++h) {
      const Slot sl = least.top();
      least.pop();
      mine[sl.second].push_back(seq * H + h);
      least.push({sl.first + c, sl.second});
    }
  }
  size_t depth = 0;
  for (const auto& m : mine) depth = std::max(depth, m.size());
  if (depth * (size_t)grid > (size_t)cap) return 0;
  for (size_t k = 0; k < depth; ++k)
    for (int b = 0; b < grid; ++b) list[k * grid + b] = k < mine[b].size() ? mine[b][k] : -1;
  return (int)(depth * grid);
}

}  // namespace kda
