// Host test driver for kda_schedule.h: reads "H grid cap" and a list of
// sequence lengths (tokens) on stdin, builds the schedule of (sequence,
// head) units with cost = 64-token chunks, and prints the list length, then
// one line per CTA: its units in order.
#include <cstdio>
#include <numeric>
#include <vector>

#include "kda_schedule.h"

int main() {
  int H, grid, cap;
  if (std::scanf("%d %d %d", &H, &grid, &cap) != 3) return 2;
  std::vector<int> len;
  int x;
  while (std::scanf("%d", &x) == 1) len.push_back(x);
  std::vector<int> idx(len.size());
  std::iota(idx.begin(), idx.end(), 0);
  std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) { return len[a] > len[b]; });
  std::vector<int> list(cap > 0 ? cap : 1, -7);
  auto chunks = [&](int s) { return (long long)((len[s] + 63) / 64); };
  const int n = kda::build_unit_schedule(idx, H, grid, chunks, list.data(), cap);
  std::printf("%d\n", n);
  if (n <= 0) return 0;
  for (int b = 0; b < grid; ++b) {
    for (int k = b; k < n; k += grid) std::printf("%d ", list[k]);
    std::printf("\n");
  }
  return 0;
}
