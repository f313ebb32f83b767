// kda_chunk_simt_dk64.cu -- instantiates the CUDA-core chunked prefill for dk = 64.
#include "kda_chunk_simt.cuh"

namespace kda {
namespace simt {
cudaError_t launch_dk64(const Problem& p, const Args& a, cudaStream_t st) {
  return launch_dk<64>(p, a, st);
}
}  // namespace simt
}  // namespace kda
