// kda_chunk_simt_dk128.cu -- instantiates the CUDA-core chunked prefill for dk = 128.
#include "kda_chunk_simt.cuh"

namespace kda {
namespace simt {
cudaError_t launch_dk128(const Problem& p, const Args& a, cudaStream_t st) {
  return launch_dk<128>(p, a, st);
}
}  // namespace simt
}  // namespace kda
