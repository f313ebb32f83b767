// kda_chunk_simt_dk32.cu -- instantiates the CUDA-core chunked prefill for dk = 32.
#include "kda_chunk_simt.cuh"

namespace kda {
namespace simt {
cudaError_t launch_dk32(const Problem& p, const Args& a, cudaStream_t st) {
  return launch_dk<32>(p, a, st);
}
}  // namespace simt
}  // namespace kda
