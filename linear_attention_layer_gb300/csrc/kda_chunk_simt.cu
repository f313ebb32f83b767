// kda_chunk_simt.cu -- dispatch of the CUDA-core prefill: the warp-per-unit
// token loop for small states (dv = 32, dk <= 64), else the chunked kernel by
// key width.
#include "kda_chunk_simt.cuh"

namespace kda {

cudaError_t launch_chunk_simt(const Problem& p, const Args& a, cudaStream_t st) {
  if (p.num_seqs == 0) return cudaSuccess;
  // small states: the warp-per-unit token loop beats 16-token chunks here
  if (recurrent_small_supported(p)) return launch_recurrent_small(p, a, st);
  switch (p.dk) {
    case 32: return simt::launch_dk32(p, a, st);
    case 64: return simt::launch_dk64(p, a, st);
    case 128: return simt::launch_dk128(p, a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kda
