// kda_api.cu -- the C ABI of libkda: argument validation, planning and
// dispatch to the kernels.  The declarations and their contract are in
// include/kda.h.
#include <cuda_runtime.h>

#include <stdint.h>
#include <string.h>

#include <initializer_list>

#include "../../include/kda.h"
#include "kda_launch.h"

namespace {

// The device error word: first device-detected problem since the last
// kda_get_device_error() on this device.
__device__ int g_kda_device_error = 0;

int* device_error_word() {
  // One address per device; cudaGetSymbolAddress resolves it for the
  // current device.
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_kda_device_error) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return static_cast<int*>(p);
}

bool supported_dim(int d) { return d == 32 || d == 64 || d == 128; }

kda_status_t check_desc(const kda_desc_t* d, bool decode) {
  if (!d) return KDA_ERR_INVALID_ARGUMENT;
  if (d->num_seqs < 0 || d->total_tokens < 0 || d->num_heads <= 0)
    return KDA_ERR_INVALID_ARGUMENT;
  if (!supported_dim(d->dk) || !supported_dim(d->dv)) return KDA_ERR_INVALID_ARGUMENT;
  if (d->io_dtype != KDA_F32 && d->io_dtype != KDA_BF16) return KDA_ERR_INVALID_ARGUMENT;
  if (decode) {
    if (d->total_tokens != d->num_seqs) return KDA_ERR_INVALID_ARGUMENT;
    return KDA_OK;
  }
  if (d->num_seqs == 0 && d->total_tokens != 0) return KDA_ERR_INVALID_ARGUMENT;
  if (d->cu_seqlens_host) {
    const int32_t* cu = d->cu_seqlens_host;
    if (cu[0] != 0) return KDA_ERR_INVALID_ARGUMENT;
    for (int i = 0; i < d->num_seqs; ++i)
      if (cu[i + 1] < cu[i]) return KDA_ERR_INVALID_ARGUMENT;
    if (cu[d->num_seqs] != d->total_tokens) return KDA_ERR_INVALID_ARGUMENT;
  }
  return KDA_OK;
}

kda::Problem to_problem(const kda_desc_t* d) {
  kda::Problem p;
  p.num_seqs = d->num_seqs;
  p.total_tokens = d->total_tokens;
  p.num_heads = d->num_heads;
  p.dk = d->dk;
  p.dv = d->dv;
  p.io_bf16 = d->io_dtype == KDA_BF16;
  return p;
}

kda_status_t prefill_common(const kda_desc_t* desc, const void* q, const void* k,
                            const void* v, const float* z, const float* beta,
                            const float* initial_state, const int32_t* cu_seqlens, void* out,
                            float* final_state, kda::Args& a) {
  kda_status_t s = check_desc(desc, false);
  if (s != KDA_OK) return s;
  if (!cu_seqlens) return KDA_ERR_INVALID_ARGUMENT;
  if (desc->total_tokens > 0 && (!q || !k || !v || !z || !beta || !out))
    return KDA_ERR_INVALID_ARGUMENT;
  if (out && (out == q || out == k || out == v || out == (const void*)z ||
              out == (const void*)beta))
    return KDA_ERR_INVALID_ARGUMENT;
  if (final_state && final_state != initial_state &&
      ((const void*)final_state == q || (const void*)final_state == k ||
       (const void*)final_state == v))
    return KDA_ERR_INVALID_ARGUMENT;
  a.q = q;
  a.k = k;
  a.v = v;
  a.z = z;
  a.beta = beta;
  a.initial_state = initial_state;
  a.cu_seqlens = cu_seqlens;
  a.out = out;
  a.final_state = final_state;
  a.a_log = desc->a_log;
  if (desc->checkpoint_every < 0 || desc->checkpoint_every % 64 != 0) return KDA_ERR_INVALID_ARGUMENT;
  if (desc->checkpoint_every > 0 && (!desc->checkpoints || !desc->checkpoint_offsets))
    return KDA_ERR_INVALID_ARGUMENT;
  a.ckpt_every = desc->checkpoint_every;
  a.ckpt = desc->checkpoint_every > 0 ? desc->checkpoints : nullptr;
  a.ckpt_off = desc->checkpoint_every > 0 ? desc->checkpoint_offsets : nullptr;
  if (desc->gate_per_head != 0 && desc->gate_per_head != 1) return KDA_ERR_INVALID_ARGUMENT;
  a.gate_per_head = desc->gate_per_head;
  a.err = device_error_word();
  if (!a.err) return KDA_ERR_CUDA;
  return KDA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

kda_status_t check_bwd(const kda_desc_t* desc, const void* q, const void* k, const void* v,
                       const float* z, const float* beta, const float* initial_state,
                       const int32_t* cu_seqlens, const void* d_out, const float* d_final,
                       const float* dq, const float* dk, const float* dv, const float* dz,
                       const float* dbeta, const float* d_initial) {
  kda_status_t s = check_desc(desc, false);
  if (s != KDA_OK) return s;
  if (!desc->cu_seqlens_host || !cu_seqlens) return KDA_ERR_INVALID_ARGUMENT;
  if (desc->gate_per_head != 0 && desc->gate_per_head != 1) return KDA_ERR_INVALID_ARGUMENT;

  if (desc->total_tokens > 0) {
    const void* need[] = {q, k, v, z, beta, d_out, dq, dk, dv, dz, dbeta};
    for (const void* x : need)
      if (!x) return KDA_ERR_INVALID_ARGUMENT;
    const void* outs[] = {dq, dk, dv, dz, dbeta};
    const void* ins[] = {q, k, v, z, beta, d_out};
    for (const void* o : outs)
      for (const void* i : ins)
        if (o == i) return KDA_ERR_INVALID_ARGUMENT;
  }
  const void* al[] = {q, k, v, z, d_out, dq, dk, dv, dz, initial_state, d_final, d_initial};
  for (const void* x : al)
    if (x && !aligned16(x)) return KDA_ERR_INVALID_ARGUMENT;
  return KDA_OK;
}

// Both reverse modes: validation, workspace check, launch.
kda_status_t run_bwd(bool chunked, const kda_desc_t* desc, const void* q, const void* k,
                     const void* v, const float* z, const float* beta,
                     const float* initial_state, const int32_t* cu_seqlens, const void* d_out,
                     const float* d_final_state, float* dq, float* dk, float* dv, float* dz,
                     float* dbeta, float* d_initial_state, kda_stream_t stream) {
  kda_status_t s = check_bwd(desc, q, k, v, z, beta, initial_state, cu_seqlens, d_out,
                             d_final_state, dq, dk, dv, dz, dbeta, d_initial_state);
  if (s != KDA_OK) return s;
  const kda::Problem p = to_problem(desc);
  const size_t need = chunked ? kda::chunk_bwd_workspace_bytes(p, desc->cu_seqlens_host)
                              : kda::recurrent_bwd_workspace_bytes(p, desc->cu_seqlens_host);
  if (need > 0 && (!desc->workspace || desc->workspace_bytes < need || !aligned16(desc->workspace)))
    return KDA_ERR_INVALID_ARGUMENT;
  kda::BwdArgs a;
  a.q = q; a.k = k; a.v = v; a.z = z; a.beta = beta;
  a.initial_state = initial_state;
  a.cu_seqlens = cu_seqlens;
  a.d_out = d_out;
  a.d_final = d_final_state;
  a.a_log = desc->a_log;
  a.dq = dq; a.dk = dk; a.dv = dv; a.dz = dz; a.dbeta = dbeta;
  a.d_initial = d_initial_state;
  a.zhead = desc->gate_per_head;
  a.err = device_error_word();
  if (!a.err) return KDA_ERR_CUDA;
  const cudaError_t e =
      chunked ? kda::launch_chunk_bwd(p, a, desc->cu_seqlens_host, desc->workspace,
                                      (cudaStream_t)stream)
              : kda::launch_recurrent_bwd(p, a, desc->cu_seqlens_host, desc->workspace,
                                          (cudaStream_t)stream);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
}  // namespace

namespace kda {
int* device_error() { return device_error_word(); }
kda_status_t check_prefill_desc(const kda_desc_t* desc) { return check_desc(desc, false); }
Problem problem_of(const kda_desc_t* desc) { return to_problem(desc); }

// Host-side validation shared with kda_chunk_fwd_noalloc (kda_noalloc.cu).
kda_status_t validate_prefill(const kda_desc_t* desc, const void* q, const void* k,
                              const void* v, const float* z, const float* beta,
                              const float* initial_state, const int32_t* cu_seqlens, void* out,
                              float* final_state, Args& a, Problem& p) {
  const kda_status_t s = prefill_common(desc, q, k, v, z, beta, initial_state, cu_seqlens, out,
                                        final_state, a);
  if (s == KDA_OK) p = to_problem(desc);
  return s;
}
}  // namespace kda

extern "C" {

kda_status_t kda_chunk_fwd(const kda_desc_t* desc, const void* q, const void* k,
                           const void* v, const float* z, const float* beta,
                           const float* initial_state, const int32_t* cu_seqlens, void* out,
                           float* final_state, kda_stream_t stream) {
  kda::Args a;
  kda_status_t s = prefill_common(desc, q, k, v, z, beta, initial_state, cu_seqlens, out,
                                  final_state, a);
  if (s != KDA_OK) return s;
  const kda::Problem p = to_problem(desc);
  cudaError_t e = kda::chunk_tc_supported(p, a)
                      ? kda::launch_chunk_tc(p, a, desc->cu_seqlens_host, desc->workspace,
                                             desc->workspace_bytes, (cudaStream_t)stream)
                      : kda::launch_chunk_simt(p, a, (cudaStream_t)stream);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_chunk_fwd_workspace_size(const kda_desc_t* desc, size_t* bytes) {
  if (!bytes) return KDA_ERR_INVALID_ARGUMENT;
  kda_status_t s = check_desc(desc, false);
  if (s != KDA_OK) return s;
  *bytes = kda::chunk_tc_workspace_bytes(to_problem(desc), desc->cu_seqlens_host);
  return KDA_OK;
}

kda_status_t kda_recurrent_fwd(const kda_desc_t* desc, const void* q, const void* k,
                               const void* v, const float* z, const float* beta,
                               const float* initial_state, const int32_t* cu_seqlens,
                               void* out, float* final_state, kda_stream_t stream) {
  // the token-by-token kernel moves states and checkpoints four floats at a time
  if (!desc || (initial_state && !aligned16(initial_state)) ||
      (final_state && !aligned16(final_state)) ||
      (desc->checkpoint_every > 0 && desc->checkpoints && !aligned16(desc->checkpoints)))
    return KDA_ERR_INVALID_ARGUMENT;
  kda::Args a;
  kda_status_t s = prefill_common(desc, q, k, v, z, beta, initial_state, cu_seqlens, out,
                                  final_state, a);
  if (s != KDA_OK) return s;
  cudaError_t e = kda::launch_recurrent(to_problem(desc), a, (cudaStream_t)stream);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_decode_step(const kda_desc_t* desc, const void* q, const void* k,
                             const void* v, const float* z, const float* beta, float* state,
                             void* out, kda_stream_t stream) {
  kda_status_t s = check_desc(desc, true);
  if (s != KDA_OK) return s;
  if (desc->num_seqs > 0 && (!q || !k || !v || !z || !beta || !state || !out))
    return KDA_ERR_INVALID_ARGUMENT;
  if (out && (out == q || out == k || out == v || out == (const void*)state))
    return KDA_ERR_INVALID_ARGUMENT;
  const kda::Problem p = to_problem(desc);
  if (desc->gate_per_head != 0 && desc->gate_per_head != 1) return KDA_ERR_INVALID_ARGUMENT;
  cudaError_t e = kda::launch_decode(p, q, k, v, z, beta, desc->a_log, desc->gate_per_head, state,
                                     out, nullptr, (cudaStream_t)stream);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

namespace {
kda_status_t check_window(const kda_desc_t* desc, int32_t window, const void* q, const void* k,
                          const void* v, const float* z, const float* beta, const void* state) {
  if (!desc) return KDA_ERR_INVALID_ARGUMENT;
  kda_desc_t d = *desc;
  d.cu_seqlens_host = nullptr;  // not used by the window calls
  if (d.gate_per_head != 0 && d.gate_per_head != 1) return KDA_ERR_INVALID_ARGUMENT;
  kda_status_t s = check_desc(&d, false);
  if (s != KDA_OK) return s;
  if (window < 1 || (int64_t)desc->num_seqs * window != desc->total_tokens)
    return KDA_ERR_INVALID_ARGUMENT;
  if (desc->num_seqs > 0 && (!q || !k || !v || !z || !beta || !state))
    return KDA_ERR_INVALID_ARGUMENT;
  if (state && !aligned16(state)) return KDA_ERR_INVALID_ARGUMENT;  // float4 / bulk copies
  return KDA_OK;
}
}  // namespace

kda_status_t kda_decode_window(const kda_desc_t* desc, int32_t window, const void* q,
                               const void* k, const void* v, const float* z, const float* beta,
                               const float* state, void* out, kda_stream_t stream) {
  kda_status_t s = check_window(desc, window, q, k, v, z, beta, state);
  if (s != KDA_OK) return s;
  if (desc->num_seqs > 0 && !out) return KDA_ERR_INVALID_ARGUMENT;
  if (out && (out == q || out == k || out == v || out == (const void*)state ||
              out == (const void*)z || out == (const void*)beta))
    return KDA_ERR_INVALID_ARGUMENT;
  int* err = device_error_word();
  if (!err) return KDA_ERR_CUDA;
  kda::WinInputs rp, wn;
  wn.q = q; wn.k = k; wn.v = v; wn.z = z; wn.beta = beta; wn.W = window;
  cudaError_t e = kda::launch_window(to_problem(desc), rp, wn, desc->a_log, desc->gate_per_head,
                                     const_cast<float*>(state), out, err, (cudaStream_t)stream);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_decode_replay(const kda_desc_t* desc, int32_t window, const void* q,
                               const void* k, const void* v, const float* z, const float* beta,
                               const int32_t* accept_len, float* state, kda_stream_t stream) {
  kda_status_t s = check_window(desc, window, q, k, v, z, beta, state);
  if (s != KDA_OK) return s;
  if (desc->num_seqs > 0 && !accept_len) return KDA_ERR_INVALID_ARGUMENT;
  int* err = device_error_word();
  if (!err) return KDA_ERR_CUDA;
  kda::WinInputs rp, wn;
  rp.q = q; rp.k = k; rp.v = v; rp.z = z; rp.beta = beta; rp.W = window; rp.accept = accept_len;
  cudaError_t e = kda::launch_window(to_problem(desc), rp, wn, desc->a_log, desc->gate_per_head,
                                     state, nullptr, err, (cudaStream_t)stream);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_decode_replay_window(const kda_desc_t* desc, int32_t prev_window,
                                      const void* prev_q, const void* prev_k, const void* prev_v,
                                      const float* prev_z, const float* prev_beta,
                                      const int32_t* accept_len, int32_t window, const void* q,
                                      const void* k, const void* v, const float* z,
                                      const float* beta, float* state, void* out,
                                      kda_stream_t stream) {
  kda_status_t s = check_window(desc, window, q, k, v, z, beta, state);
  if (s != KDA_OK) return s;
  if (prev_window < 1) return KDA_ERR_INVALID_ARGUMENT;
  if (desc->num_seqs > 0 &&
      (!prev_q || !prev_k || !prev_v || !prev_z || !prev_beta || !accept_len || !out))
    return KDA_ERR_INVALID_ARGUMENT;
  const void* ins[] = {q, k, v, z, beta, prev_q, prev_k, prev_v, prev_z, prev_beta, state};
  for (const void* x : ins)
    if (out && out == x) return KDA_ERR_INVALID_ARGUMENT;
  int* err = device_error_word();
  if (!err) return KDA_ERR_CUDA;
  kda::WinInputs rp, wn;
  rp.q = prev_q; rp.k = prev_k; rp.v = prev_v; rp.z = prev_z; rp.beta = prev_beta;
  rp.W = prev_window; rp.accept = accept_len;
  wn.q = q; wn.k = k; wn.v = v; wn.z = z; wn.beta = beta; wn.W = window;
  cudaError_t e = kda::launch_window(to_problem(desc), rp, wn, desc->a_log, desc->gate_per_head,
                                     state, out, err, (cudaStream_t)stream);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

namespace {
// Checks of a kda_fusion_t (NULL = nothing fused); fills fa.
kda_status_t check_fusion(const kda_fusion_t* f, kda::FusionArgs& fa) {
  fa = kda::FusionArgs{0, nullptr, nullptr, nullptr, nullptr, nullptr, 0.f};
  if (!f) return KDA_OK;
  if (f->conv_width < 0) return KDA_ERR_INVALID_ARGUMENT;
  if (f->conv_width > 4) return KDA_ERR_UNSUPPORTED;
  if (f->conv_width > 0) {
    if (!f->conv_weight_q || !f->conv_weight_k) return KDA_ERR_INVALID_ARGUMENT;
    if (f->conv_width > 1 && (!f->conv_state_q || !f->conv_state_k ||
                              f->conv_state_q == f->conv_state_k))
      return KDA_ERR_INVALID_ARGUMENT;
  }
  if (!(f->out_norm_eps >= 0.f)) return KDA_ERR_INVALID_ARGUMENT;  // also rejects NaN
  fa.width = f->conv_width;
  fa.wq = f->conv_weight_q;
  fa.wk = f->conv_weight_k;
  fa.sq = f->conv_width > 1 ? f->conv_state_q : nullptr;
  fa.sk = f->conv_width > 1 ? f->conv_state_k : nullptr;
  fa.onw = f->out_norm_weight;
  fa.eps = f->out_norm_eps;
  return KDA_OK;
}

bool any_equal(const void* x, std::initializer_list<const void*> ys) {
  if (!x) return false;
  for (const void* y : ys)
    if (x == y) return true;
  return false;
}
}  // namespace

kda_status_t kda_decode_step_fused(const kda_desc_t* desc, const kda_fusion_t* fusion,
                                   const void* q, const void* k, const void* v, const float* z,
                                   const float* beta, float* state, void* out,
                                   kda_stream_t stream) {
  kda_status_t s = check_desc(desc, true);
  if (s != KDA_OK) return s;
  if (desc->gate_per_head != 0 && desc->gate_per_head != 1) return KDA_ERR_INVALID_ARGUMENT;
  kda::FusionArgs fa;
  s = check_fusion(fusion, fa);
  if (s != KDA_OK) return s;
  if (desc->num_seqs > 0 && (!q || !k || !v || !z || !beta || !state || !out))
    return KDA_ERR_INVALID_ARGUMENT;
  if (any_equal(out, {q, k, v, state, z, beta, fa.sq, fa.sk}) ||
      any_equal(fa.sq, {q, k, v, state, z, beta}) || any_equal(fa.sk, {q, k, v, state, z, beta}))
    return KDA_ERR_INVALID_ARGUMENT;
  if (state && !aligned16(state)) return KDA_ERR_INVALID_ARGUMENT;
  cudaError_t e = kda::launch_decode_fused(to_problem(desc), q, k, v, z, beta, desc->a_log,
                                           desc->gate_per_head, state, out, fa,
                                           (cudaStream_t)stream);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_decode_replay_window_fused(
    const kda_desc_t* desc, const kda_fusion_t* fusion, int32_t prev_window, const void* prev_q,
    const void* prev_k, const void* prev_v, const float* prev_z, const float* prev_beta,
    const int32_t* accept_len, int32_t window, const void* q, const void* k, const void* v,
    const float* z, const float* beta, float* state, void* out, kda_stream_t stream) {
  if (!desc) return KDA_ERR_INVALID_ARGUMENT;
  kda_desc_t d = *desc;
  d.cu_seqlens_host = nullptr;  // not used by the window calls
  if (d.gate_per_head != 0 && d.gate_per_head != 1) return KDA_ERR_INVALID_ARGUMENT;
  kda_status_t s = check_desc(&d, false);
  if (s != KDA_OK) return s;
  if (prev_window < 0 || window < 0 || (prev_window == 0 && window == 0))
    return KDA_ERR_INVALID_ARGUMENT;
  if ((int64_t)desc->num_seqs * window != desc->total_tokens) return KDA_ERR_INVALID_ARGUMENT;
  kda::FusionArgs fa;
  s = check_fusion(fusion, fa);
  if (s != KDA_OK) return s;
  if (fa.onw && !aligned16(fa.onw)) return KDA_ERR_INVALID_ARGUMENT;  // read as float4
  const int B = desc->num_seqs;
  if (B > 0) {
    if (!state) return KDA_ERR_INVALID_ARGUMENT;
    if (prev_window > 0 &&
        (!prev_q || !prev_k || !prev_v || !prev_z || !prev_beta || !accept_len))
      return KDA_ERR_INVALID_ARGUMENT;
    if (window > 0 && (!q || !k || !v || !z || !beta || !out)) return KDA_ERR_INVALID_ARGUMENT;
  }
  if (state && !aligned16(state)) return KDA_ERR_INVALID_ARGUMENT;
  const std::initializer_list<const void*> ins = {q, k, v, z, beta, prev_q, prev_k,
                                                  prev_v, prev_z, prev_beta, state};
  if ((window > 0 && any_equal(out, ins)) || any_equal(fa.sq, ins) || any_equal(fa.sk, ins) ||
      (window > 0 && out && (out == fa.sq || out == fa.sk)))
    return KDA_ERR_INVALID_ARGUMENT;
  int* err = device_error_word();
  if (!err) return KDA_ERR_CUDA;
  kda::WinInputs rp, wn;
  if (prev_window > 0) {
    rp.q = prev_q; rp.k = prev_k; rp.v = prev_v; rp.z = prev_z; rp.beta = prev_beta;
    rp.W = prev_window; rp.accept = accept_len;
  }
  if (window > 0) {
    wn.q = q; wn.k = k; wn.v = v; wn.z = z; wn.beta = beta; wn.W = window;
  }
  cudaError_t e = kda::launch_window(to_problem(desc), rp, wn, desc->a_log, desc->gate_per_head,
                                     state, window > 0 ? out : nullptr, err,
                                     (cudaStream_t)stream, &fa);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_chunk_fwd_fused(const kda_desc_t* desc, const kda_fusion_t* fusion,
                                 const void* q, const void* k, const void* v, const float* z,
                                 const float* beta, const float* initial_state,
                                 const int32_t* cu_seqlens, void* out, float* final_state,
                                 kda_stream_t stream) {
  kda::Args a;
  kda_status_t s = prefill_common(desc, q, k, v, z, beta, initial_state, cu_seqlens, out,
                                  final_state, a);
  if (s != KDA_OK) return s;
  kda::FusionArgs fa;
  s = check_fusion(fusion, fa);
  if (s != KDA_OK) return s;
  if (fa.onw) return KDA_ERR_UNSUPPORTED;  // the output norm belongs to the decode side
  const kda::Problem p = to_problem(desc);
  const bool tc = kda::chunk_tc_supported(p, a);
  if (fa.width > 0) {
    if (!tc) return KDA_ERR_UNSUPPORTED;
    const std::initializer_list<const void*> bufs = {q, k, v, z, beta, out, initial_state,
                                                     final_state, cu_seqlens};
    if (any_equal(fa.sq, bufs) || any_equal(fa.sk, bufs)) return KDA_ERR_INVALID_ARGUMENT;
    a.conv_w = fa.width;
    a.conv_wq = fa.wq;
    a.conv_wk = fa.wk;
    a.conv_sq = fa.sq;
    a.conv_sk = fa.sk;
  }
  cudaError_t e = tc ? kda::launch_chunk_tc(p, a, desc->cu_seqlens_host, desc->workspace,
                                            desc->workspace_bytes, (cudaStream_t)stream)
                     : kda::launch_chunk_simt(p, a, (cudaStream_t)stream);
  if (e == cudaSuccess && fa.width > 1) {
    // each sequence's last W-1 raw inputs, once every reader of the incoming
    // states is done (so the states may be updated in place)
    kda::ConvArgs c{};
    c.cu_seqlens = cu_seqlens;
    c.width = fa.width;
    c.err = a.err;
    c.x = q;
    c.state_in = fa.sq;
    c.state_out = fa.sq;
    e = kda::launch_short_conv_state(p, c, (cudaStream_t)stream);
    if (e == cudaSuccess) {
      c.x = k;
      c.state_in = fa.sk;
      c.state_out = fa.sk;
      e = kda::launch_short_conv_state(p, c, (cudaStream_t)stream);
    }
  }
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_chunk_fwd_host_workspace_size(const kda_desc_t* desc, size_t* bytes) {
  if (!bytes || !desc) return KDA_ERR_INVALID_ARGUMENT;
  kda_status_t s = check_desc(desc, false);
  if (s != KDA_OK) return s;
  if (desc->gate_per_head != 0 && desc->gate_per_head != 1) return KDA_ERR_INVALID_ARGUMENT;
  *bytes = kda::chunk_fwd_host_workspace_bytes(to_problem(desc), desc->gate_per_head == 1);
  return KDA_OK;
}

kda_status_t kda_chunk_fwd_host(const kda_desc_t* desc, int32_t groups, const void* q,
                                const void* k, const void* v, const float* z, const float* beta,
                                const float* initial_state, const int32_t* cu_seqlens, void* out,
                                float* final_state, kda_stream_t stream) {
  if (!desc || !cu_seqlens) return KDA_ERR_INVALID_ARGUMENT;
  if (desc->cu_seqlens_host && desc->cu_seqlens_host != cu_seqlens) return KDA_ERR_INVALID_ARGUMENT;
  kda_desc_t d = *desc;
  d.cu_seqlens_host = cu_seqlens;  // validated as the host copy
  kda_status_t s = check_desc(&d, false);
  if (s != KDA_OK) return s;
  if (groups < 1) return KDA_ERR_INVALID_ARGUMENT;
  if (d.gate_per_head != 0 && d.gate_per_head != 1) return KDA_ERR_INVALID_ARGUMENT;
  if (d.checkpoint_every != 0) return KDA_ERR_UNSUPPORTED;
  if (d.total_tokens > 0 && (!q || !k || !v || !z || !beta || !out)) return KDA_ERR_INVALID_ARGUMENT;
  const kda::Problem p = to_problem(&d);
  const size_t need = kda::chunk_fwd_host_workspace_bytes(p, d.gate_per_head == 1);
  if (!d.workspace || d.workspace_bytes < need ||
      (reinterpret_cast<uintptr_t>(d.workspace) & 255) != 0)
    return KDA_ERR_INVALID_ARGUMENT;
  if (d.num_seqs == 0) return KDA_OK;
  kda::HostArgs h;
  h.q = q; h.k = k; h.v = v; h.z = z; h.beta = beta;
  h.initial_state = initial_state;
  h.cu_seqlens = cu_seqlens;
  h.out = out;
  h.final_state = final_state;
  h.a_log = d.a_log;
  h.gate_per_head = d.gate_per_head;
  h.err = device_error_word();
  if (!h.err) return KDA_ERR_CUDA;
  cudaError_t e = kda::launch_chunk_fwd_host(p, h, groups, d.workspace, (cudaStream_t)stream);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_short_conv(const kda_desc_t* desc, int32_t width, const void* x,
                            const float* weight, const float* conv_state_in,
                            const int32_t* cu_seqlens, void* y, float* conv_state_out,
                            kda_stream_t stream) {
  kda_status_t s = check_desc(desc, false);
  if (s != KDA_OK) return s;
  if (width < 1) return KDA_ERR_INVALID_ARGUMENT;
  if (width > 4) return KDA_ERR_UNSUPPORTED;
  if (!cu_seqlens || !weight) return KDA_ERR_INVALID_ARGUMENT;
  if (desc->total_tokens > 0 && (!x || !y)) return KDA_ERR_INVALID_ARGUMENT;
  if (y && (y == x || y == (const void*)weight || y == (const void*)conv_state_in))
    return KDA_ERR_INVALID_ARGUMENT;
  if (conv_state_out && conv_state_out != conv_state_in &&
      ((const void*)conv_state_out == x || (const void*)conv_state_out == y))
    return KDA_ERR_INVALID_ARGUMENT;
  const void* al[] = {x, y};
  for (const void* p : al)
    if (p && !aligned16(p)) return KDA_ERR_INVALID_ARGUMENT;
  kda::ConvArgs a;
  a.x = x;
  a.weight = weight;
  a.state_in = conv_state_in;
  a.cu_seqlens = cu_seqlens;
  a.y = y;
  a.state_out = conv_state_out;
  a.width = width;
  a.err = device_error_word();
  if (!a.err) return KDA_ERR_CUDA;
  cudaError_t e = kda::launch_short_conv(to_problem(desc), a, (cudaStream_t)stream);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_recurrent_bwd_workspace_size(const kda_desc_t* desc, size_t* bytes) {
  if (!bytes || !desc) return KDA_ERR_INVALID_ARGUMENT;
  kda_status_t s = check_desc(desc, false);
  if (s != KDA_OK) return s;
  if (!desc->cu_seqlens_host) return KDA_ERR_INVALID_ARGUMENT;
  *bytes = kda::recurrent_bwd_workspace_bytes(to_problem(desc), desc->cu_seqlens_host);
  return KDA_OK;
}

kda_status_t kda_chunk_bwd_workspace_size(const kda_desc_t* desc, size_t* bytes) {
  if (!bytes || !desc) return KDA_ERR_INVALID_ARGUMENT;
  kda_status_t s = check_desc(desc, false);
  if (s != KDA_OK) return s;
  if (!desc->cu_seqlens_host) return KDA_ERR_INVALID_ARGUMENT;
  *bytes = kda::chunk_bwd_workspace_bytes(to_problem(desc), desc->cu_seqlens_host);
  return KDA_OK;
}

kda_status_t kda_recurrent_bwd(const kda_desc_t* desc, const void* q, const void* k,
                               const void* v, const float* z, const float* beta,
                               const float* initial_state, const int32_t* cu_seqlens,
                               const void* d_out, const float* d_final_state, float* dq,
                               float* dk, float* dv, float* dz, float* dbeta,
                               float* d_initial_state, kda_stream_t stream) {
  return run_bwd(false, desc, q, k, v, z, beta, initial_state, cu_seqlens, d_out, d_final_state,
                 dq, dk, dv, dz, dbeta, d_initial_state, stream);
}

kda_status_t kda_chunk_bwd(const kda_desc_t* desc, const void* q, const void* k, const void* v,
                           const float* z, const float* beta, const float* initial_state,
                           const int32_t* cu_seqlens, const void* d_out,
                           const float* d_final_state, float* dq, float* dk, float* dv,
                           float* dz, float* dbeta, float* d_initial_state, kda_stream_t stream) {
  return run_bwd(true, desc, q, k, v, z, beta, initial_state, cu_seqlens, d_out, d_final_state,
                 dq, dk, dv, dz, dbeta, d_initial_state, stream);
}

const char* kda_status_string(kda_status_t status) {
  switch (status) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARGUMENT: return "KDA_ERR_INVALID_ARGUMENT";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
    case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
    case KDA_ERR_DEVICE_CHECK: return "KDA_ERR_DEVICE_CHECK";
  }
  return "KDA_ERR_UNKNOWN";
}

kda_status_t kda_get_device_error(kda_stream_t stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return KDA_ERR_CUDA;
  int h = 0;
  if (cudaMemcpyFromSymbol(&h, g_kda_device_error, sizeof(int)) != cudaSuccess)
    return KDA_ERR_CUDA;
  if (h != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_kda_device_error, &zero, sizeof(int)) != cudaSuccess)
      return KDA_ERR_CUDA;
  }
  switch (h) {
    case 0: return KDA_OK;
    case KDA_ERR_TIMEOUT: return KDA_ERR_TIMEOUT;
    default: return KDA_ERR_DEVICE_CHECK;
  }
}

}  // extern "C"
