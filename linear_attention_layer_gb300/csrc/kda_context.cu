// kda_context.cu -- context parallelism: the affine summary of a segment of
// a sequence and the prefix scan that turns the summaries of consecutive
// segments into each segment's entering state.
//
// The state update is affine in the state (mhpq.cn/news/56770, section
// "KDA 到底在算什么"), so a segment maps its entering state S_in to
// S_out = M S_in + S~, M [dk][dk] being the product of the segment's
// per-token transitions and S~ the state it reaches from zeros.  The pages'
// context-parallel KDA (blog.higcp.com "猜想：K3 可能是最适合 TPU 的 MoE 架构",
// section "第二层") has every device summarise its own segment this way,
// exchange the summaries in one all-gather and rebuild its entering state by
// a prefix scan before running its segment.  kda_chunk_fwd_summary computes
// the summaries (on the tensor cores, long segments split across SMs and
// composed); kda_state_scan applies a list of them to a state.
#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "../../include/kda.h"
#include "kda_launch.h"

namespace kda {
namespace fold {

constexpr int kThreads = 256;
constexpr int kMaxEntries = 512;  // chains per launch (the host loops beyond)

struct Params {
  const float* start;
  const float* m;
  const float* b;
  float* out;
  long long stride;
  int H;
  FoldEntry e[kMaxEntries];
};

// One CTA per (entry, head).  Thread (ty, tx) of a 16 x 16 grid owns rows
// RT ty .. RT ty + RT - 1 and columns CT tx .. CT tx + CT - 1 of the state,
// kept in registers across the steps; each step stages M_i (transposed) and
// the state in shared memory and accumulates b_i + M_i S.
template <int DK, int DV>
__global__ void __launch_bounds__(kThreads) fold_kernel(const __grid_constant__ Params P) {
  constexpr int RT = DK / 16, CT = DV / 16;
  constexpr int LDM = DK + 4, LDS = DV + 4;
  extern __shared__ __align__(16) float fold_smem[];
  float* Mt = fold_smem;             // Mt[k][r] = M[r][k]
  float* Ss = fold_smem + DK * LDM;  // Ss[k][c] = S[k][c]
  const FoldEntry en = P.e[blockIdx.x / P.H];
  const int h = blockIdx.x % P.H, tid = threadIdx.x;
  const int r0 = (tid >> 4) * RT, c0 = (tid & 15) * CT;
  const size_t ms = (size_t)DK * DK, ss = (size_t)DK * DV;
  float s[RT][CT];
  {
    const float* src = P.start ? P.start + ((size_t)en.start_idx * P.H + h) * ss : nullptr;
#pragma unroll
    for (int i = 0; i < RT; ++i)
#pragma unroll
      for (int j = 0; j < CT; ++j) s[i][j] = src ? src[(size_t)(r0 + i) * DV + c0 + j] : 0.f;
  }
  for (int step = 0; step < en.count; ++step) {
    const float* M = P.m + ((size_t)(en.m_idx + step * P.stride) * P.H + h) * ms;
    const float* B = P.b ? P.b + ((size_t)(en.b_idx + step * P.stride) * P.H + h) * ss : nullptr;
    __syncthreads();  // the previous step's reads of Mt and Ss are done
    for (int idx = tid; idx < DK * DK; idx += kThreads) {
      const int r = idx / DK, k = idx % DK;
      Mt[k * LDM + r] = M[idx];
    }
#pragma unroll
    for (int i = 0; i < RT; ++i)
#pragma unroll
      for (int j = 0; j < CT; ++j) Ss[(r0 + i) * LDS + c0 + j] = s[i][j];
    __syncthreads();
    float acc[RT][CT];
#pragma unroll
    for (int i = 0; i < RT; ++i)
#pragma unroll
      for (int j = 0; j < CT; ++j) acc[i][j] = B ? B[(size_t)(r0 + i) * DV + c0 + j] : 0.f;
#pragma unroll 4
    for (int k = 0; k < DK; ++k) {
      float mv[RT], sv[CT];
#pragma unroll
      for (int i = 0; i < RT; ++i) mv[i] = Mt[k * LDM + r0 + i];
#pragma unroll
      for (int j = 0; j < CT; ++j) sv[j] = Ss[k * LDS + c0 + j];
#pragma unroll
      for (int i = 0; i < RT; ++i)
#pragma unroll
        for (int j = 0; j < CT; ++j) acc[i][j] = fmaf(mv[i], sv[j], acc[i][j]);
    }
#pragma unroll
    for (int i = 0; i < RT; ++i)
#pragma unroll
      for (int j = 0; j < CT; ++j) s[i][j] = acc[i][j];
  }
  float* dst = P.out + ((size_t)en.out_idx * P.H + h) * ss;
#pragma unroll
  for (int i = 0; i < RT; ++i)
#pragma unroll
    for (int j = 0; j < CT; ++j) dst[(size_t)(r0 + i) * DV + c0 + j] = s[i][j];
}

template <int DK, int DV>
cudaError_t launch_t(const Params& prm, int n, cudaStream_t st) {
  constexpr size_t smem = sizeof(float) * (DK * (DK + 4) + DK * (DV + 4));
  static PerDeviceInit attrs;
  const cudaError_t e = attrs.run([] {
    return cudaFuncSetAttribute(fold_kernel<DK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem);
  });
  if (e != cudaSuccess) return e;
  fold_kernel<DK, DV><<<n * prm.H, kThreads, smem, st>>>(prm);
  return cudaGetLastError();
}

}  // namespace fold

cudaError_t launch_state_fold(int dk, int dv, int H, const float* start, const float* m,
                              const float* b, float* out, long long stride,
                              const FoldEntry* entries, int n_entries, cudaStream_t st) {
  static thread_local fold::Params prm;  // large: keep off the stack
  prm.start = start;
  prm.m = m;
  prm.b = b;
  prm.out = out;
  prm.stride = stride;
  prm.H = H;
  for (int e0 = 0; e0 < n_entries; e0 += fold::kMaxEntries) {
    const int n = std::min(fold::kMaxEntries, n_entries - e0);
    std::copy(entries + e0, entries + e0 + n, prm.e);
    cudaError_t err = cudaErrorInvalidValue;
#define KDA_FOLD_CASE(A, B) \
  if (dk == A && dv == B) err = fold::launch_t<A, B>(prm, n, st);
    KDA_FOLD_CASE(32, 32) KDA_FOLD_CASE(32, 64) KDA_FOLD_CASE(32, 128)
    KDA_FOLD_CASE(64, 32) KDA_FOLD_CASE(64, 64) KDA_FOLD_CASE(64, 128)
    KDA_FOLD_CASE(128, 32) KDA_FOLD_CASE(128, 64) KDA_FOLD_CASE(128, 128)
#undef KDA_FOLD_CASE
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace kda

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

kda_status_t check_summary(const kda_desc_t* desc, const void* q, const void* k, const void* v,
                           const float* z, const float* beta, const int32_t* cu_seqlens,
                           const float* transition, const float* offset_state) {
  const kda_status_t s = kda::check_prefill_desc(desc);
  if (s != KDA_OK) return s;
  if (!desc->cu_seqlens_host || !cu_seqlens) return KDA_ERR_INVALID_ARGUMENT;
  if (desc->gate_per_head != 0 && desc->gate_per_head != 1) return KDA_ERR_INVALID_ARGUMENT;
  if (desc->num_seqs > 0 && (!transition || !offset_state)) return KDA_ERR_INVALID_ARGUMENT;
  if (desc->total_tokens > 0 && (!q || !k || !v || !z || !beta)) return KDA_ERR_INVALID_ARGUMENT;
  if (desc->io_dtype != KDA_BF16 || desc->dk != 128 || desc->dv != 128) return KDA_ERR_UNSUPPORTED;
  const void* al[] = {q, k, v, z, transition, offset_state};
  for (const void* x : al)
    if (x && !aligned16(x)) return KDA_ERR_INVALID_ARGUMENT;
  const void* outs[] = {transition, offset_state};
  const void* ins[] = {q, k, v, z, beta};
  for (const void* o : outs)
    for (const void* i : ins)
      if (o && o == i) return KDA_ERR_INVALID_ARGUMENT;
  if (transition && transition == offset_state) return KDA_ERR_INVALID_ARGUMENT;
  return KDA_OK;
}

}  // namespace

extern "C" kda_status_t kda_chunk_fwd_summary(const kda_desc_t* desc, const void* q,
                                              const void* k, const void* v, const float* z,
                                              const float* beta, const int32_t* cu_seqlens,
                                              float* transition, float* offset_state,
                                              kda_stream_t stream) {
  const kda_status_t s =
      check_summary(desc, q, k, v, z, beta, cu_seqlens, transition, offset_state);
  if (s != KDA_OK) return s;
  kda::Args a = {};
  a.q = q;
  a.k = k;
  a.v = v;
  a.z = z;
  a.beta = beta;
  a.initial_state = nullptr;
  a.cu_seqlens = cu_seqlens;
  a.out = nullptr;
  a.final_state = offset_state;
  a.err = kda::device_error();
  if (!a.err) return KDA_ERR_CUDA;
  a.a_log = desc->a_log;
  a.ckpt = nullptr;
  a.ckpt_off = nullptr;
  a.ckpt_every = 0;
  a.gate_per_head = desc->gate_per_head;
  const cudaError_t e = kda::launch_chunk_tc_summary(
      kda::problem_of(desc), a, desc->cu_seqlens_host, transition, desc->workspace,
      desc->workspace_bytes, (cudaStream_t)stream);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

extern "C" kda_status_t kda_chunk_fwd_summary_workspace_size(const kda_desc_t* desc,
                                                             size_t* bytes) {
  if (!bytes) return KDA_ERR_INVALID_ARGUMENT;
  const kda_status_t s = kda::check_prefill_desc(desc);
  if (s != KDA_OK) return s;
  *bytes = kda::chunk_tc_summary_workspace_bytes(kda::problem_of(desc), desc->cu_seqlens_host);
  return KDA_OK;
}

extern "C" kda_status_t kda_state_scan(const kda_desc_t* desc, int32_t count,
                                       const float* transitions, const float* offsets,
                                       const float* initial_state, float* entry_state,
                                       kda_stream_t stream) {
  if (!desc || count < 0) return KDA_ERR_INVALID_ARGUMENT;
  const int N = desc->num_seqs, H = desc->num_heads, dk = desc->dk, dv = desc->dv;
  auto dim_ok = [](int d) { return d == 32 || d == 64 || d == 128; };
  if (N < 0 || H <= 0 || !dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_INVALID_ARGUMENT;
  if (N == 0) return KDA_OK;
  if (!entry_state || (count > 0 && (!transitions || !offsets))) return KDA_ERR_INVALID_ARGUMENT;
  if (count > 0 && ((const void*)entry_state == transitions || entry_state == offsets))
    return KDA_ERR_INVALID_ARGUMENT;
  std::vector<kda::FoldEntry> en(N);
  for (int n = 0; n < N; ++n) en[n] = kda::FoldEntry{n, n, n, n, count};
  const cudaError_t e = kda::launch_state_fold(dk, dv, H, initial_state, transitions, offsets,
                                               entry_state, N, en.data(), N,
                                               (cudaStream_t)stream);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
