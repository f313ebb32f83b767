// kda_host.cu -- kda_chunk_fwd_host: the prefill over inputs and outputs in
// host memory, with the copies overlapped with the kernels.
//
// The packed batch is cut into groups of whole sequences of about equal token
// count; every per-token array of a group is one contiguous row range, and
// every state array one contiguous range of (sequence, head) blocks.  Three
// streams: host-to-device copies of group g+1 run while the kernel of group g
// computes and the device-to-host copies of group g-1 drain (the two copy
// directions use separate engines).  A group's kernel also reads the up to 63
// rows past its last sequence (the 64-row tiles of a chunk), so it starts
// only once the NEXT group's inputs have landed as well: every row it reads
// holds this call's data.  Each group is one launch of the usual chunked
// kernel over absolute token offsets (its cu_seqlens are a slice of the whole
// batch's), so nothing is re-based.
#include <algorithm>
#include <mutex>
#include <vector>

#include "kda_launch.h"

namespace kda {
namespace {

struct HostLayout {
  size_t q, k, v, z, beta, out, s0, sfin, cu, total;
};

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Device staging area: every input and output of the batch (both state arrays
// always reserved, so the size depends on the shapes only).
HostLayout host_layout(const Problem& p, bool gate_per_head) {
  const size_t es = p.io_bf16 ? 2 : 4, T = (size_t)p.total_tokens, H = (size_t)p.num_heads;
  const size_t state = (size_t)p.num_seqs * H * p.dk * p.dv * 4;
  HostLayout L;
  size_t o = 0;
  L.q = o; o += up256(T * H * p.dk * es);
  L.k = o; o += up256(T * H * p.dk * es);
  L.v = o; o += up256(T * H * p.dv * es);
  L.z = o; o += up256(T * H * (gate_per_head ? 1 : p.dk) * 4);
  L.beta = o; o += up256(T * H * 4);
  L.out = o; o += up256(T * H * p.dv * es);
  L.s0 = o; o += up256(state);
  L.sfin = o; o += up256(state);
  L.cu = o; o += up256(((size_t)p.num_seqs + 1) * 4);
  L.total = o;
  return L;
}

// Side streams and events, created once per device and kept.
struct Pipes {
  cudaStream_t h2d = nullptr, d2h = nullptr;
  std::vector<cudaEvent_t> ev;  // grows on demand
};
std::mutex g_pipes_mu;
Pipes g_pipes[64];

cudaError_t get_pipes(Pipes** out, size_t nev) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  Pipes& P = g_pipes[dev];
  if (!P.h2d) {
    if ((e = cudaStreamCreateWithFlags(&P.h2d, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&P.d2h, cudaStreamNonBlocking)) != cudaSuccess) return e;
  }
  while (P.ev.size() < nev) {
    cudaEvent_t x;
    if ((e = cudaEventCreateWithFlags(&x, cudaEventDisableTiming)) != cudaSuccess) return e;
    P.ev.push_back(x);
  }
  *out = &P;
  return cudaSuccess;
}

}  // namespace

size_t chunk_fwd_host_workspace_bytes(const Problem& p, bool gate_per_head) {
  return host_layout(p, gate_per_head).total;
}

cudaError_t launch_chunk_fwd_host(const Problem& p, const HostArgs& h, int groups, void* ws,
                                  cudaStream_t st) {
  const bool with_s0 = h.initial_state != nullptr, with_fin = h.final_state != nullptr;
  const HostLayout L = host_layout(p, h.gate_per_head != 0);
  unsigned char* W = static_cast<unsigned char*>(ws);
  const int N = p.num_seqs, H = p.num_heads;
  const int32_t* cu = h.cu_seqlens;
  const size_t es = p.io_bf16 ? 2 : 4;
  const size_t zrow = (size_t)H * (h.gate_per_head ? 1 : p.dk) * 4;
  const size_t state = (size_t)H * p.dk * p.dv * 4;  // per sequence

  // groups of whole sequences, about total / groups tokens each
  groups = std::max(1, std::min(groups, N));
  std::vector<int> first{0};
  for (int g = 1; g < groups; ++g) {
    const long long target = (long long)p.total_tokens * g / groups;
    int n = first.back();
    while (n < N && cu[n] < target) ++n;
    if (n > first.back() && n < N) first.push_back(n);
  }
  first.push_back(N);
  const int G = (int)first.size() - 1;

  std::lock_guard<std::mutex> lock(g_pipes_mu);  // the side streams are shared per device
  Pipes* P = nullptr;
  cudaError_t e = get_pipes(&P, 2 * (size_t)G + 2);
  if (e != cudaSuccess) return e;
  cudaEvent_t ev_start = P->ev[0], ev_done = P->ev[1];
  cudaEvent_t* ev_in = P->ev.data() + 2;       // G events: inputs of group g landed
  cudaEvent_t* ev_comp = P->ev.data() + 2 + G;  // G events: kernel of group g done
  // the side streams start after earlier work on the caller's stream
  if ((e = cudaEventRecord(ev_start, st)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(P->h2d, ev_start, 0)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(P->d2h, ev_start, 0)) != cudaSuccess) return e;

  auto h2d = [&](size_t off, const void* src, size_t bytes) {
    return bytes ? cudaMemcpyAsync(W + off, src, bytes, cudaMemcpyHostToDevice, P->h2d)
                 : cudaSuccess;
  };
  auto d2h = [&](void* dst, size_t off, size_t bytes) {
    return bytes ? cudaMemcpyAsync(dst, W + off, bytes, cudaMemcpyDeviceToHost, P->d2h)
                 : cudaSuccess;
  };
  if ((e = h2d(L.cu, cu, ((size_t)N + 1) * 4)) != cudaSuccess) return e;
  for (int g = 0; g < G; ++g) {
    const size_t t0 = (size_t)cu[first[g]], t1 = (size_t)cu[first[g + 1]];
    const size_t n0 = (size_t)first[g], n1 = (size_t)first[g + 1];
    const size_t rq = (size_t)H * p.dk * es, rv = (size_t)H * p.dv * es;
    const unsigned char* q = static_cast<const unsigned char*>(h.q);
    const unsigned char* k = static_cast<const unsigned char*>(h.k);
    const unsigned char* v = static_cast<const unsigned char*>(h.v);
    const unsigned char* z = reinterpret_cast<const unsigned char*>(h.z);
    const unsigned char* b = reinterpret_cast<const unsigned char*>(h.beta);
    if ((e = h2d(L.q + t0 * rq, q + t0 * rq, (t1 - t0) * rq)) != cudaSuccess) return e;
    if ((e = h2d(L.k + t0 * rq, k + t0 * rq, (t1 - t0) * rq)) != cudaSuccess) return e;
    if ((e = h2d(L.v + t0 * rv, v + t0 * rv, (t1 - t0) * rv)) != cudaSuccess) return e;
    if ((e = h2d(L.z + t0 * zrow, z + t0 * zrow, (t1 - t0) * zrow)) != cudaSuccess) return e;
    if ((e = h2d(L.beta + t0 * H * 4, b + t0 * H * 4, (t1 - t0) * H * 4)) != cudaSuccess)
      return e;
    if (with_s0 &&
        (e = h2d(L.s0 + n0 * state, reinterpret_cast<const unsigned char*>(h.initial_state) +
                                        n0 * state,
                 (n1 - n0) * state)) != cudaSuccess)
      return e;
    if ((e = cudaEventRecord(ev_in[g], P->h2d)) != cudaSuccess) return e;
  }
  for (int g = 0; g < G; ++g) {
    // the kernel of group g reads into group g + 1's first rows
    if ((e = cudaStreamWaitEvent(st, ev_in[std::min(g + 1, G - 1)], 0)) != cudaSuccess) return e;
    const int n0 = first[g], ng = first[g + 1] - first[g];
    Problem pg = p;
    pg.num_seqs = ng;
    Args a{};
    a.q = W + L.q;
    a.k = W + L.k;
    a.v = W + L.v;
    a.z = reinterpret_cast<const float*>(W + L.z);
    a.beta = reinterpret_cast<const float*>(W + L.beta);
    a.initial_state = with_s0 ? reinterpret_cast<const float*>(W + L.s0 + (size_t)n0 * state)
                              : nullptr;
    a.cu_seqlens = reinterpret_cast<const int32_t*>(W + L.cu) + n0;
    a.out = W + L.out;
    a.final_state = with_fin ? reinterpret_cast<float*>(W + L.sfin + (size_t)n0 * state) : nullptr;
    a.err = h.err;
    a.a_log = h.a_log;
    a.ckpt = nullptr;
    a.ckpt_off = nullptr;
    a.ckpt_every = 0;
    a.gate_per_head = h.gate_per_head;
    e = chunk_tc_supported(pg, a) ? launch_chunk_tc(pg, a, cu + n0, nullptr, 0, st)
                                  : launch_chunk_simt(pg, a, st);
    if (e != cudaSuccess) return e;
    if ((e = cudaEventRecord(ev_comp[g], st)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(P->d2h, ev_comp[g], 0)) != cudaSuccess) return e;
    const size_t t0 = (size_t)cu[n0], t1 = (size_t)cu[n0 + ng];
    const size_t rv = (size_t)H * p.dv * es;
    if ((e = d2h(static_cast<unsigned char*>(h.out) + t0 * rv, L.out + t0 * rv, (t1 - t0) * rv)) !=
        cudaSuccess)
      return e;
    if (with_fin && (e = d2h(reinterpret_cast<unsigned char*>(h.final_state) + (size_t)n0 * state,
                             L.sfin + (size_t)n0 * state, (size_t)ng * state)) != cudaSuccess)
      return e;
  }
  // later work on the caller's stream sees the outputs in host memory
  if ((e = cudaEventRecord(ev_done, P->d2h)) != cudaSuccess) return e;
  return cudaStreamWaitEvent(st, ev_done, 0);
}

}  // namespace kda
