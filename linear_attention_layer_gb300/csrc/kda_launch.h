// kda_launch.h -- internal launchers behind the C ABI (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

namespace kda {

// Function attributes (such as the dynamic shared-memory limit) belong to a
// device's context, so a launcher that sets them must do so on every device
// it launches on.  run(fn) calls fn once per device -- the current one --
// and remembers success; a failure is returned and retried on the next call.
class PerDeviceInit {
 public:
  template <class F>
  cudaError_t run(F&& fn) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return fn();  // beyond the table: every call
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev]) return cudaSuccess;
    e = fn();
    if (e == cudaSuccess) done_[dev] = true;
    return e;
  }

 private:
  static constexpr int kMaxDevices = 64;
  std::mutex mu_;
  bool done_[kMaxDevices] = {};
};

struct Problem {
  int num_seqs;
  int total_tokens;
  int num_heads;
  int dk;
  int dv;
  int io_bf16;  // 0 = fp32 q/k/v/out, 1 = bf16
};

struct Args {
  const void* q;
  const void* k;
  const void* v;
  const float* z;
  const float* beta;
  const float* initial_state;  // may be null (zeros)
  const int32_t* cu_seqlens;   // device
  void* out;
  float* final_state;  // may be null
  int* err;            // device error word
  const float* a_log;  // per-head gate log-scale [H], may be null (A = 0)
  float* ckpt;               // state checkpoints (null: none)
  const int32_t* ckpt_off;   // device [N + 1] prefix sums of checkpoints per sequence
  int ckpt_every;            // tokens between checkpoints (0: none)
  int gate_per_head;         // 1: z is [T, H], one gate per head (scalar alpha)
  // fused short convolution of q and k (tensor-core path; conv_w = 0: none):
  // taps [H][dk][W], incoming states [N][H][dk][W-1] (null: zeros)
  int conv_w = 0;
  const float* conv_wq = nullptr;
  const float* conv_wk = nullptr;
  const float* conv_sq = nullptr;
  const float* conv_sk = nullptr;
};

// One work item of a chunked launch: a (sequence, head) pair, processed
// over tokens [tok_begin, tok_end) of that sequence (relative to its start).
// A negative tok_end means "to the end of the sequence".
struct WorkItem {
  int32_t seq;
  int32_t head;
};

// Decode: one token per (request, head), state updated in place.
cudaError_t launch_decode(const Problem& p, const void* q, const void* k, const void* v,
                          const float* z, const float* beta, const float* a_log, int gate_per_head,
                          float* state, void* out, int* err, cudaStream_t stream);

// Speculative decoding (inputs of a window: [B*W, H, .]).  rp: a window
// whose first accept[b] tokens are applied again and the state written
// (rp.accept == nullptr: none); wn: a window whose W outputs are computed
// from the (replayed) state, which it does not write (W == 0: none).
struct WinInputs {
  const void* q = nullptr;
  const void* k = nullptr;
  const void* v = nullptr;
  const float* z = nullptr;
  const float* beta = nullptr;
  int W = 0;
  const int32_t* accept = nullptr;
};
// Optional fused pre- and post-processing of the decode-side calls
// (kda_fusion_t): width 0 = no convolution, onw null = no output norm.
struct FusionArgs {
  int width;
  const float* wq;
  const float* wk;
  float* sq;
  float* sk;
  const float* onw;
  float eps;
};
cudaError_t launch_window(const Problem& p, const WinInputs& rp, const WinInputs& wn,
                          const float* a_log, int gate_per_head, float* state, void* out,
                          int* err, cudaStream_t stream, const FusionArgs* fusion = nullptr);
cudaError_t launch_decode_fused(const Problem& p, const void* q, const void* k, const void* v,
                                const float* z, const float* beta, const float* a_log,
                                int gate_per_head, float* state, void* out,
                                const FusionArgs& fusion, cudaStream_t stream);

// Token-by-token prefill over a packed batch.
cudaError_t launch_recurrent(const Problem& p, const Args& a, cudaStream_t stream);
// The same with one warp per (sequence, head) for small states (dv = 32, dk <= 64).
bool recurrent_small_supported(const Problem& p);
cudaError_t launch_recurrent_small(const Problem& p, const Args& a, cudaStream_t stream);

// Chunked prefill on CUDA cores in fp32 (any supported size, fp32 or bf16 io).
cudaError_t launch_chunk_simt(const Problem& p, const Args& a, cudaStream_t stream);

// Chunked prefill on the tensor cores (bf16 io, dk = dv = 128, 16-byte
// aligned buffers).  cu_host (optional) orders the work longest-first and,
// with workspace (256-byte aligned), lets long sequences be split across SMs
// by the best plan whose segment summaries fit in ws_bytes.
bool chunk_tc_supported(const Problem& p, const Args& a);
size_t chunk_tc_workspace_bytes(const Problem& p, const int32_t* cu_host);
cudaError_t launch_chunk_tc(const Problem& p, const Args& a, const int32_t* cu_host, void* ws,
                            size_t ws_bytes, cudaStream_t stream);

// Affine summary of every sequence on the tensor cores (bf16, dk = dv = 128):
// m_out[n, h] = the transition M (state after the sequence = M S_in + S~) and
// a.final_state[n, h] = S~, the state reached from zeros.  With workspace
// (256-byte aligned) long sequences are cut into segments whose summaries
// are computed side by side and then composed.
size_t chunk_tc_summary_workspace_bytes(const Problem& p, const int32_t* cu_host);
cudaError_t launch_chunk_tc_summary(const Problem& p, const Args& a, const int32_t* cu_host,
                                    float* m_out, void* ws, size_t ws_bytes, cudaStream_t st);

// Chains of affine state maps S <- M_i S + b_i in fp32 (M_i [dk][dk]; S and b_i
// [dk][dv]), one chain per (entry, head), H heads.  Entry e starts from
// start + (start_idx * H + h) * dk * dv (start == nullptr: zeros); its step i
// reads M at m + ((m_idx + i * stride) * H + h) * dk * dk and b at
// b + ((b_idx + i * stride) * H + h) * dk * dv (b == nullptr: no offset); the
// result goes to out + (out_idx * H + h) * dk * dv.  out may alias start.
struct FoldEntry {
  int start_idx, m_idx, b_idx, out_idx, count;
};
cudaError_t launch_state_fold(int dk, int dv, int H, const float* start, const float* m,
                              const float* b, float* out, long long stride,
                              const FoldEntry* entries, int n_entries, cudaStream_t st);

// Reverse mode of the recurrence, token by token (fp32; dk = dv = 128).
struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* z;
  const float* beta;
  const float* initial_state;  // may be null (zeros)
  const int32_t* cu_seqlens;   // device
  const void* d_out;           // io dtype, like out
  const float* d_final;        // may be null (zeros)
  const float* a_log;          // may be null (A = 0)
  float* dq;
  float* dk;
  float* dv;
  float* dz;
  float* dbeta;
  float* d_initial;  // may be null
  int* err;
  int zhead = 0;     // 1: one gate per head (z, dz [T, H])
};
size_t recurrent_bwd_workspace_bytes(const Problem& p, const int32_t* cu_host);
cudaError_t launch_recurrent_bwd(const Problem& p, const BwdArgs& a, const int32_t* cu_host,
                                 void* ws, cudaStream_t stream);
// The same gradients from the chunked form (16-token chunks, tf32 tensor-core
// products); BwdArgs as above.
size_t chunk_bwd_workspace_bytes(const Problem& p, const int32_t* cu_host);
cudaError_t launch_chunk_bwd(const Problem& p, const BwdArgs& a, const int32_t* cu_host, void* ws,
                             cudaStream_t stream);
size_t chunk_bwd_inner_bytes(const Problem& p, const int32_t* cu_host);  // dk = dv = 128
cudaError_t launch_chunk_bwd_128(const Problem& p, const BwdArgs& a, const int32_t* cu_host,
                                 void* ws, cudaStream_t stream);

// The Q/K preprocessing convolution (depthwise, causal, width 1..4) + Swish.
struct ConvArgs {
  const void* x;           // [T, H, D] io dtype
  const float* weight;     // [H, D, W]
  const float* state_in;   // [N, H, D, W - 1] or null (zeros)
  const int32_t* cu_seqlens;
  void* y;                 // [T, H, D] io dtype
  float* state_out;        // [N, H, D, W - 1] or null; may equal state_in
  int width;
  int* err;
};
cudaError_t launch_short_conv(const Problem& p, const ConvArgs& a, cudaStream_t stream);
// Only its second step: each sequence's outgoing state (last W-1 inputs).
cudaError_t launch_short_conv_state(const Problem& p, const ConvArgs& a, cudaStream_t stream);

// The prefill over host buffers with copies overlapped (kda_host.cu).
struct HostArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* z;
  const float* beta;
  const float* initial_state;  // host, may be null
  const int32_t* cu_seqlens;   // host
  void* out;
  float* final_state;  // host, may be null
  const float* a_log;  // device, may be null
  int gate_per_head;
  int* err;
};
size_t chunk_fwd_host_workspace_bytes(const Problem& p, bool gate_per_head);
cudaError_t launch_chunk_fwd_host(const Problem& p, const HostArgs& h, int groups, void* ws,
                                  cudaStream_t stream);

}  // namespace kda

#include "../../include/kda.h"

namespace kda {
// The device error word of the current device (null if it cannot be found).
int* device_error();
// The descriptor checks shared by the prefill calls.
kda_status_t check_prefill_desc(const kda_desc_t* desc);
Problem problem_of(const kda_desc_t* desc);
// Host validation of a prefill call (the checks of kda_chunk_fwd); fills a and p.
kda_status_t validate_prefill(const kda_desc_t* desc, const void* q, const void* k,
                              const void* v, const float* z, const float* beta,
                              const float* initial_state, const int32_t* cu_seqlens, void* out,
                              float* final_state, Args& a, Problem& p);
}  // namespace kda
