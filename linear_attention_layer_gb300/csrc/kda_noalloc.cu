// kda_noalloc.cu -- kda_chunk_fwd_noalloc: the chunked prefill for callers
// that cannot allocate device memory.
//
// kda_chunk_fwd splits a few long sequences across SMs only when the caller
// hands it scratch (desc->workspace).  Some callers cannot obtain that
// scratch with cudaMalloc: their device memory belongs to a host framework
// that reserved the whole HBM up front, or they run inside a plugin that is
// not allowed to allocate, or inside a latency-critical loop where the
// implicit device synchronisation of cudaMalloc is unacceptable.  This entry
// point serves them from a fixed scratch array that lives in this library's
// module instead: nothing is allocated or freed at call time.
#include <cuda_runtime.h>

#include "../../include/kda.h"
#include "kda_launch.h"

namespace {

// The scratch every call of kda_chunk_fwd_noalloc shares.  Every GPU that
// loads this library holds it until the process exits.  In host code this
// name is only a stand-in for the device array: the device address comes
// from cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device, or null.  It is
// looked up on every call (a cheap host query): a cached address would go
// stale if the context were torn down and the module loaded again.
void* scratch_on_current_device() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
    cudaGetLastError();  // clear this thread's last-error state
    return nullptr;
  }
  return p;
}

}  // namespace

extern "C" kda_status_t kda_chunk_fwd_noalloc(const kda_desc_t* desc, const void* q,
                                              const void* k, const void* v, const float* z,
                                              const float* beta, const float* initial_state,
                                              const int32_t* cu_seqlens, void* out,
                                              float* final_state, kda_stream_t stream) {
  kda::Args a;
  kda::Problem p;
  const kda_status_t s = kda::validate_prefill(desc, q, k, v, z, beta, initial_state, cu_seqlens,
                                               out, final_state, a, p);
  if (s != KDA_OK) return s;
  if (!kda::chunk_tc_supported(p, a)) {
    // the CUDA-core path never uses scratch
    return kda::launch_chunk_simt(p, a, (cudaStream_t)stream) == cudaSuccess ? KDA_OK
                                                                             : KDA_ERR_CUDA;
  }
  // Any split plan at all?  The launcher then takes the best one whose
  // segment summaries fit in the array, or runs unsplit when none fits.
  void* ws = nullptr;
  if (kda::chunk_tc_workspace_bytes(p, desc->cu_seqlens_host) > 0) {
    ws = scratch_on_current_device();
    if (!ws) return KDA_ERR_CUDA;
  }
  const cudaError_t e = kda::launch_chunk_tc(p, a, desc->cu_seqlens_host, ws,
                                             ws ? (size_t)KDA_NOALLOC_SCRATCH_BYTES : 0,
                                             (cudaStream_t)stream);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
