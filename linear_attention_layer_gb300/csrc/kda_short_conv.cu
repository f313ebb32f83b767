// kda_short_conv.cu -- the Q/K preprocessing convolution.
//
// mhpq.cn/news/56770, section "KDA 到底在算什么" (the Q/K preprocessing
// paragraph): query and key first pass a short causal convolution over the
// most recent few positions, then a Swish activation, then the L2
// normalisation (which the KDA kernels apply themselves).  Depthwise (one
// filter per head and channel), width W, no bias:
//     y[t, h, d] = swish( sum_j w[h, d, j] x[t - (W - 1) + j, h, d] ),  swish(u) = u sigmoid(u),
// positions before a sequence's first token reading its convolution state
// (the W - 1 inputs before it, oldest first; zeros without one).
//
// HBM-bound: each input is read once and each output written once.  A thread
// takes 4 channels of one head over a 64-token segment of the packed batch,
// keeping the last W - 1 inputs in registers and four loads in flight; a warp
// covers 32 x 4 consecutive channels of a token, so every access is coalesced.  A
// second, tiny launch writes each sequence's outgoing state (its last W - 1
// inputs) after the first has read the incoming one, so the two may share
// memory.
#include "kda_common.cuh"
#include "kda_launch.h"

namespace kda {
namespace conv {

constexpr int kSeg = 64;  // tokens per thread
constexpr int kVec = 4;   // channels per thread
constexpr int kNT = 256;

template <typename T>
struct Vec4;
template <>
struct Vec4<float> {
  static __device__ __forceinline__ void ld(const float* p, float (&x)[4]) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  }
  static __device__ __forceinline__ void st(float* p, const float (&x)[4]) {
    st_stream(reinterpret_cast<float4*>(p), make_float4(x[0], x[1], x[2], x[3]));
  }
};
template <>
struct Vec4<__nv_bfloat16> {
  static __device__ __forceinline__ void ld(const __nv_bfloat16* p, float (&x)[4]) {
    const uint2 a = __ldg(reinterpret_cast<const uint2*>(p));
    x[0] = __uint_as_float(a.x << 16);
    x[1] = __uint_as_float(a.x & 0xffff0000u);
    x[2] = __uint_as_float(a.y << 16);
    x[3] = __uint_as_float(a.y & 0xffff0000u);
  }
  static __device__ __forceinline__ void st(__nv_bfloat16* p, const float (&x)[4]) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]);
    const __nv_bfloat162 b = __floats2bfloat162_rn(x[2], x[3]);
    __stcs(reinterpret_cast<uint2*>(p), make_uint2(*reinterpret_cast<const uint32_t*>(&a),
                                                   *reinterpret_cast<const uint32_t*>(&b)));
  }
};

// The sequence holding token t: the largest n with cu[n] <= t, which skips
// empty sequences; the caller checks cu[n] <= t < cu[n + 1].
__device__ __forceinline__ int find_seq(const int32_t* cu, int N, int t) {
  int lo = 0, hi = N - 1;
  while (lo < hi) {  // largest n with cu[n] <= t
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Load the W - 1 inputs before token t of sequence [bos, ...) into win
// (oldest first), from x where they are inside the sequence, else from the
// sequence's state (zeros without one).
template <typename T, int W>
__device__ __forceinline__ void fill_window(float (&win)[W > 1 ? W - 1 : 1][kVec], const T* x,
                                            const float* st, int H, int D, int n, int h, int d0,
                                            int bos, int t) {
#pragma unroll
  for (int j = 0; j < W - 1; ++j) {
    const int pos = t - (W - 1) + j;
    if (pos >= bos) {
      Vec4<T>::ld(x + ((size_t)pos * H + h) * D + d0, win[j]);
    } else if (st) {
      const float* s = st + (((size_t)n * H + h) * D + d0) * (W - 1) + (pos - bos + W - 1);
#pragma unroll
      for (int c = 0; c < kVec; ++c) win[j][c] = __ldg(s + c * (W - 1));
    } else {
#pragma unroll
      for (int c = 0; c < kVec; ++c) win[j][c] = 0.f;
    }
  }
}

template <typename T, int W>
__global__ void __launch_bounds__(kNT, 3) conv_kernel(const T* __restrict__ x,
                                                      const float* __restrict__ w,
                                                      const float* st_in, const int32_t* cu,
                                                      int N, int total, int H, int D,
                                                      T* __restrict__ y, int* err) {
  const int groups = D / kVec;
  const long long g = (long long)blockIdx.x * kNT + threadIdx.x;
  const long long nseg = (total + kSeg - 1) / kSeg;
  if (g >= nseg * H * groups) return;
  const int cg = (int)(g % groups), h = (int)((g / groups) % H);
  const int s = (int)(g / ((long long)groups * H));
  const int d0 = cg * kVec;
  const int t0 = s * kSeg, t1 = min(t0 + kSeg, total);
  if (__ldg(cu) != 0 || __ldg(cu + N) != total) {
    report_error(err, kErrDeviceCheck);
    return;
  }
  float wr[W][kVec];
#pragma unroll
  for (int c = 0; c < kVec; ++c)
#pragma unroll
    for (int j = 0; j < W; ++j) wr[j][c] = __ldg(w + ((size_t)h * D + d0 + c) * W + j);

  int n = find_seq(cu, N, t0);
  int bos = __ldg(cu + n), eos = __ldg(cu + n + 1);
  if (bos > t0 || eos <= t0) {  // cu not monotone
    report_error(err, kErrDeviceCheck);
    return;
  }
  float win[W > 1 ? W - 1 : 1][kVec];
  fill_window<T, W>(win, x, st_in, H, D, n, h, d0, bos, t0);
  // One token: y_t from the window and x_t, then x_t enters the window.
  auto token = [&](int t, const float (&xt)[kVec]) {
    float out[kVec];
#pragma unroll
    for (int c = 0; c < kVec; ++c) {
      float acc = wr[W - 1][c] * xt[c];
#pragma unroll
      for (int j = 0; j < W - 1; ++j) acc = fmaf(wr[j][c], win[j][c], acc);
      out[c] = acc / (1.f + __expf(-acc));  // swish
    }
    Vec4<T>::st(y + ((size_t)t * H + h) * D + d0, out);
#pragma unroll
    for (int j = 0; j + 1 < W - 1; ++j)
#pragma unroll
      for (int c = 0; c < kVec; ++c) win[j][c] = win[j + 1][c];
    if (W > 1)
#pragma unroll
      for (int c = 0; c < kVec; ++c) win[W > 1 ? W - 2 : 0][c] = xt[c];
  };
  int t = t0;
  for (;;) {
    // tokens [t, te) all belong to sequence n: four loads in flight at a time
    const int te = min(t1, eos);
    for (; t + 4 <= te; t += 4) {
      float xs[4][kVec];
#pragma unroll
      for (int u = 0; u < 4; ++u) Vec4<T>::ld(x + ((size_t)(t + u) * H + h) * D + d0, xs[u]);
#pragma unroll
      for (int u = 0; u < 4; ++u) token(t + u, xs[u]);
    }
    for (; t < te; ++t) {
      float xt[kVec];
      Vec4<T>::ld(x + ((size_t)t * H + h) * D + d0, xt);
      token(t, xt);
    }
    if (t >= t1) break;
    while (eos <= t) {  // the next non-empty sequence starts at t
      ++n;
      bos = __ldg(cu + n);
      eos = __ldg(cu + n + 1);
      if (eos < bos || bos > t) {
        report_error(err, kErrDeviceCheck);
        return;
      }
    }
    fill_window<T, W>(win, x, st_in, H, D, n, h, d0, bos, t);
  }
}

// Outgoing state of sequence n: its last W - 1 inputs (oldest first), from x
// inside the sequence, else from its incoming state.  One thread per (n, h, d);
// it reads all it needs before writing, so st_out may be st_in.
template <typename T, int W>
__global__ void __launch_bounds__(kNT) state_kernel(const T* x, const float* st_in,
                                                    const int32_t* cu, int N, int total, int H,
                                                    int D, float* st_out, int* err) {
  const long long g = (long long)blockIdx.x * kNT + threadIdx.x;
  if (g >= (long long)N * H * D) return;
  const int d = (int)(g % D), h = (int)((g / D) % H), n = (int)(g / ((long long)D * H));
  int bos, eos;
  if (!seq_range(cu, n, total, err, bos, eos)) return;
  float v[W > 1 ? W - 1 : 1];
#pragma unroll
  for (int j = 0; j < W - 1; ++j) {
    const int pos = eos - (W - 1) + j;
    if (pos >= bos) v[j] = IO<T>::ld(x + ((size_t)pos * H + h) * D + d);
    else v[j] = st_in ? st_in[(((size_t)n * H + h) * D + d) * (W - 1) + (pos - bos + W - 1)] : 0.f;
  }
#pragma unroll
  for (int j = 0; j < W - 1; ++j) st_out[(((size_t)n * H + h) * D + d) * (W - 1) + j] = v[j];
}

template <typename T, int W>
cudaError_t launch_w(const Problem& p, const ConvArgs& a, cudaStream_t st) {
  const int D = p.dk, H = p.num_heads;
  if (p.total_tokens > 0) {
    const long long nseg = (p.total_tokens + kSeg - 1) / kSeg;
    const long long threads = nseg * H * (D / kVec);
    conv_kernel<T, W><<<(unsigned)((threads + kNT - 1) / kNT), kNT, 0, st>>>(
        static_cast<const T*>(a.x), a.weight, a.state_in, a.cu_seqlens, p.num_seqs,
        p.total_tokens, H, D, static_cast<T*>(a.y), a.err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (a.state_out && W > 1 && p.num_seqs > 0) {
    const long long threads = (long long)p.num_seqs * H * D;
    state_kernel<T, W><<<(unsigned)((threads + kNT - 1) / kNT), kNT, 0, st>>>(
        static_cast<const T*>(a.x), a.state_in, a.cu_seqlens, p.num_seqs, p.total_tokens, H, D,
        a.state_out, a.err);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

template <typename T>
cudaError_t launch_t(const Problem& p, const ConvArgs& a, cudaStream_t st) {
  switch (a.width) {
    case 1: return launch_w<T, 1>(p, a, st);
    case 2: return launch_w<T, 2>(p, a, st);
    case 3: return launch_w<T, 3>(p, a, st);
    case 4: return launch_w<T, 4>(p, a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace conv

cudaError_t launch_short_conv_state(const Problem& p, const ConvArgs& a, cudaStream_t st) {
  if (!a.state_out || a.width < 2 || p.num_seqs == 0) return cudaSuccess;
  const long long threads = (long long)p.num_seqs * p.num_heads * p.dk;
  const unsigned blocks = (unsigned)((threads + conv::kNT - 1) / conv::kNT);
  auto go = [&](auto tag) {
    using T = decltype(tag);
    switch (a.width) {
      case 2: conv::state_kernel<T, 2><<<blocks, conv::kNT, 0, st>>>(
          static_cast<const T*>(a.x), a.state_in, a.cu_seqlens, p.num_seqs, p.total_tokens,
          p.num_heads, p.dk, a.state_out, a.err); break;
      case 3: conv::state_kernel<T, 3><<<blocks, conv::kNT, 0, st>>>(
          static_cast<const T*>(a.x), a.state_in, a.cu_seqlens, p.num_seqs, p.total_tokens,
          p.num_heads, p.dk, a.state_out, a.err); break;
      default: conv::state_kernel<T, 4><<<blocks, conv::kNT, 0, st>>>(
          static_cast<const T*>(a.x), a.state_in, a.cu_seqlens, p.num_seqs, p.total_tokens,
          p.num_heads, p.dk, a.state_out, a.err); break;
    }
    return cudaGetLastError();
  };
  if (a.width > 4) return cudaErrorInvalidValue;
  return p.io_bf16 ? go(__nv_bfloat16{}) : go(float{});
}

cudaError_t launch_short_conv(const Problem& p, const ConvArgs& a, cudaStream_t st) {
  return p.io_bf16 ? conv::launch_t<__nv_bfloat16>(p, a, st) : conv::launch_t<float>(p, a, st);
}

}  // namespace kda
