// Host test driver for the long-sequence split planner of kda_chunk_tc.cu:
// reads "H sms" and the sequence lengths (tokens) on stdin, prints the plan
// and the entries of its two passes.  Nothing here touches a GPU.
#include <cstdio>

#include "kda_chunk_tc.cu"

namespace kda {
// the affine-summary fold lives in another translation unit of the library
cudaError_t launch_state_fold(int, int, int, const float*, const float*, const float*, float*,
                              long long, const FoldEntry*, int, cudaStream_t) {
  return cudaSuccess;
}
}  // namespace kda

int main() {
  int H, sms;
  if (std::scanf("%d %d", &H, &sms) != 2) return 2;
  std::vector<int32_t> cu{0};
  int x;
  while (std::scanf("%d", &x) == 1) cu.push_back(cu.back() + x);
  kda::Problem p{};
  p.num_seqs = (int)cu.size() - 1;
  p.total_tokens = cu.back();
  p.num_heads = H;
  p.dk = p.dv = 128;
  p.io_bf16 = true;
  const kda::tcp::SplitPlan pl = kda::tcp::plan_split_search(p, cu.data(), sms, ~(size_t)0);
  std::printf("plan %d %d %d %d %d\n", pl.use ? 1 : 0, pl.seg0_len, pl.seg_len, pl.s0_at, pl.E);
  if (!pl.use) return 0;
  for (int n = 0; n < p.num_seqs; ++n) std::printf("seq %d %d %d\n", n, pl.nseg[n], pl.base[n]);
  for (const auto& e : kda::tcp::pass1_entries(pl, cu.data(), p.num_seqs))
    std::printf("p1 %d %d %d %d %d %d\n", e.n, e.tb, e.te, e.in, e.out, e.flags);
  for (const auto& e : kda::tcp::pass2_entries(pl, cu.data(), p.num_seqs))
    std::printf("p2 %d %d %d %d %d %d\n", e.n, e.tb, e.te, e.in, e.out, e.flags);
  return 0;
}
