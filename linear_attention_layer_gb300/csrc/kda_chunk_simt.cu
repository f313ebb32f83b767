// kda_chunk_simt.cu -- dispatch of the CUDA-core chunked prefill by key width.
#include "kda_chunk_simt.cuh"

namespace kda {

cudaError_t launch_chunk_simt(const Problem& p, const Args& a, cudaStream_t st) {
  if (p.num_seqs == 0) return cudaSuccess;
  switch (p.dk) {
    case 32: return simt::launch_dk32(p, a, st);
    case 64: return simt::launch_dk64(p, a, st);
    case 128: return simt::launch_dk128(p, a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kda
