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
// HBM-bound: each input is read once and each output written once.  The
// packed batch is a [T, C] matrix (C = H * D channels, each filtered on its
// own), cut into tiles of 64 tokens (up to 240 for narrow rows) by a slab of
// SB bytes of each row.  A persistent CTA (two per SM) streams its tiles
// through a three-stage ring in shared memory -- each tile with the three rows
// before it is one tensor-map copy (cp.async.bulk.tensor, 2-D) completing on
// the stage's mbarrier -- so the bytes in flight are set by the ring, not by
// registers; a thread then filters four channels over a run of 16 (fp32: 8)
// of the tile's tokens and stores them with one 8- or 16-byte store per
// token.  The Swish divides with the fast reciprocal (the correctly rounded
// division cost more than all the rest of the arithmetic).  Shapes whose rows
// are not a multiple of 128 bytes take a register-only kernel (a thread: 4
// channels of one head over a 64-token segment, four loads in flight).  A
// second, tiny launch writes each sequence's outgoing state (its last W - 1
// inputs) after the first has read the incoming one, so the two may share
// memory.
#include <cuda.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "kda_common.cuh"
#include "kda_launch.h"
#include "tc_ptx.cuh"

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
      out[c] = __fdividef(acc, 1.f + __expf(-acc));  // swish
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

// ---- the tiled kernel ----
constexpr int kStages = 3;
constexpr int kHalo = 3;  // rows before a tile (W - 1 <= 3)

template <typename T, int SB>
struct TileShape {
  static constexpr int Q = SB / (4 * (int)sizeof(T));      // channel quads per slab row
  static constexpr int G = kNT / Q;                        // token runs per tile
  static constexpr int TPT0 = sizeof(T) == 2 ? 16 : 8;
  static constexpr int TPT =                               // tokens per run (a box has
      TPT0 * G + kHalo <= 256 ? TPT0 : (256 - kHalo) / G;  // at most 256 rows)
  static constexpr int TILE = TPT * G;                     // tokens per tile
  static constexpr int ROWS = TILE + kHalo;
  static constexpr int STAGE = ROWS * SB;                  // bytes per ring stage
  static_assert(kNT % Q == 0 && SB % 128 == 0 && ROWS <= 256 && TPT >= 1, "tile shape");
};

template <typename T, int SB>
constexpr int tile_smem() {
  return kStages * TileShape<T, SB>::STAGE;
}

// One tile (box) of the [T, C] tensor map at column x, row y (y may be
// negative or run past the end: those rows read as zeros) into dst.
__device__ __forceinline__ void tma_tile(void* dst, const CUtensorMap* map, int x, int y,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(tc::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(tc::smem_u32(bar))
      : "memory");
}

// Four channels from shared memory (an io-dtype row)
__device__ __forceinline__ void ld4_smem(const float* p, float (&x)[kVec]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
}
__device__ __forceinline__ void ld4_smem(const __nv_bfloat16* p, float (&x)[kVec]) {
  const uint2 a = *reinterpret_cast<const uint2*>(p);
  x[0] = __uint_as_float(a.x << 16);
  x[1] = __uint_as_float(a.x & 0xffff0000u);
  x[2] = __uint_as_float(a.y << 16);
  x[3] = __uint_as_float(a.y & 0xffff0000u);
}

// Tile item i: tokens [TILE * (i / slabs), +TILE) of slab i % slabs.  CTA b
// takes items b, b + gridDim.x, ...; item k of a CTA lives in stage k % kStages.
template <typename T, int W, int SB>
__global__ void __launch_bounds__(kNT, 2) conv_tile_kernel(const __grid_constant__ CUtensorMap xmap,
                                                           const float* __restrict__ w,
                                                           const float* st_in, const int32_t* cu,
                                                           int N, int total, int C,
                                                           T* __restrict__ y, int* err) {
  using TS = TileShape<T, SB>;
  constexpr int CS = SB / (int)sizeof(T);  // channels per slab
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ __align__(8) uint64_t full[kStages];
  const int slabs = C / CS;
  const long long ntiles = (total + TS::TILE - 1) / TS::TILE;
  const long long items = ntiles * slabs;
  if (blockIdx.x >= items) return;
  if (__ldg(cu) != 0 || __ldg(cu + N) != total) {
    if (threadIdx.x == 0) report_error(err, kErrDeviceCheck);
    return;
  }
  const int tid = threadIdx.x, q = tid % TS::Q, gi = tid / TS::Q;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) tc::mbar_init(&full[s], 1);
    tc::mbar_fence_init();
  }
  __syncthreads();
  // item `it` into stage st (thread 0): the tile's rows and the three before
  // it, one tensor-map copy (rows outside [0, T) arrive as zeros, never read)
  auto issue = [&](long long it, int st) {
    const long long r = it / slabs;
    const int sl = (int)(it % slabs);
    tc::fence_proxy_async_smem();  // the stage's earlier generic reads come first
    tc::mbar_arrive_expect_tx(&full[st], (uint32_t)TS::STAGE);
    tma_tile(ring + st * TS::STAGE, &xmap, sl * CS, (int)(r * TS::TILE) - kHalo, &full[st]);
  };
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      const long long it = blockIdx.x + (long long)s * gridDim.x;
      if (it < items) issue(it, s);
    }
  }
  int wslab = -1;
  float wr[W][kVec];
  int n = 0;  // the sequence of this thread's last run (its runs only move forward)
  for (long long k = 0;; ++k) {
    const long long it = blockIdx.x + k * gridDim.x;
    if (it >= items) break;
    const int st = (int)(k % kStages);
    const uint32_t par = (uint32_t)((k / kStages) & 1);
    const long long r = it / slabs;
    const int sl = (int)(it % slabs);
    if (sl != wslab) {  // this thread's taps
      wslab = sl;
#pragma unroll
      for (int c = 0; c < kVec; ++c)
#pragma unroll
        for (int j = 0; j < W; ++j) wr[j][c] = __ldg(w + ((size_t)sl * CS + 4 * q + c) * W + j);
    }
    {  // bounded wait (about 2 s) for the stage's copies; the CTA decides as one
      const long long c0 = clock64();
      int ok = 1;
      while (!tc::mbar_try_wait(&full[st], par))
        if (clock64() - c0 > 4000000000LL) {
          ok = 0;
          break;
        }
      if (!__syncthreads_and(ok)) {
        if (threadIdx.x == 0) report_error(err, kErrTimeout);
        return;
      }
    }
    const T* const rows = reinterpret_cast<const T*>(ring + st * TS::STAGE);
    const int t0 = (int)(r * TS::TILE);  // row kHalo of the stage
    const int ta = t0 + gi * TS::TPT, tb = min(ta + TS::TPT, total);
    const int cch = sl * CS + 4 * q;      // first channel
    if (ta < tb) {
      while (n + 1 < N && __ldg(cu + n + 1) <= ta) ++n;  // largest n with cu[n] <= ta
      int bos = __ldg(cu + n), eos = __ldg(cu + n + 1);
      float win[W > 1 ? W - 1 : 1][kVec];
      // the W - 1 inputs before token t: rows of the stage inside the
      // sequence, else its incoming state (zeros without one)
      auto fill = [&](int t) {
#pragma unroll
        for (int j = 0; j < W - 1; ++j) {
          const int pos = t - (W - 1) + j;
          if (pos >= bos) {
            ld4_smem(rows + (size_t)(pos - t0 + kHalo) * CS + 4 * q, win[j]);
          } else if (st_in) {
            const float* sp = st_in + ((size_t)n * C + cch) * (W - 1) + (pos - bos + W - 1);
#pragma unroll
            for (int c = 0; c < kVec; ++c) win[j][c] = __ldg(sp + c * (W - 1));
          } else {
#pragma unroll
            for (int c = 0; c < kVec; ++c) win[j][c] = 0.f;
          }
        }
      };
      if (bos > ta || eos <= ta) {  // cu not monotone
        report_error(err, kErrDeviceCheck);
      } else {
        fill(ta);
        // one token: y_t from the window and x_t, then x_t enters the window
        auto token = [&](int t, const float (&xt)[kVec]) {
          float out[kVec];
#pragma unroll
          for (int c = 0; c < kVec; ++c) {
            float acc = wr[W - 1][c] * xt[c];
#pragma unroll
            for (int j = 0; j < W - 1; ++j) acc = fmaf(wr[j][c], win[j][c], acc);
            out[c] = __fdividef(acc, 1.f + __expf(-acc));  // swish
          }
          Vec4<T>::st(y + (size_t)t * C + cch, out);
#pragma unroll
          for (int j = 0; j + 1 < W - 1; ++j)
#pragma unroll
            for (int c = 0; c < kVec; ++c) win[j][c] = win[j + 1][c];
          if (W > 1)
#pragma unroll
            for (int c = 0; c < kVec; ++c) win[W > 1 ? W - 2 : 0][c] = xt[c];
        };
        if (tb - ta == TS::TPT && eos >= tb) {  // a whole run inside one sequence: unrolled
          const T* const rr = rows + (size_t)(ta - t0 + kHalo) * CS + 4 * q;
#pragma unroll
          for (int u = 0; u < TS::TPT; ++u) {
            float xt[kVec];
            ld4_smem(rr + u * CS, xt);
            token(ta + u, xt);
          }
        } else {
          for (int t = ta; t < tb; ++t) {
            if (t >= eos) {  // the next non-empty sequence starts at t
              bool bad = false;
              while (eos <= t) {
                ++n;
                bos = __ldg(cu + n);
                eos = __ldg(cu + n + 1);
                if (eos < bos || bos > t) {
                  bad = true;
                  break;
                }
              }
              if (bad) {
                report_error(err, kErrDeviceCheck);
                break;
              }
              fill(t);
            }
            float xt[kVec];
            ld4_smem(rows + (size_t)(t - t0 + kHalo) * CS + 4 * q, xt);
            token(t, xt);
          }
        }
      }
    }
    __syncthreads();  // the stage is read by every thread
    const long long nx = it + (long long)kStages * gridDim.x;
    if (threadIdx.x == 0 && nx < items) issue(nx, st);
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

// The [T, C] input as a 2-D tensor map with boxes of `rows` x `cols`.
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
#pragma GCC diagnostic push
#pragma GCC diagnostic ignored "-Wdeprecated-declarations"
bool encode_rows(CUtensorMap* m, const void* x, CUtensorMapDataType dt, int esize, int C, int T,
                 int cols, int rows) {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)T};
  const cuuint64_t strides[1] = {(cuuint64_t)C * esize};
  const cuuint32_t box[2] = {(cuuint32_t)cols, (cuuint32_t)rows};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(m, dt, 2, const_cast<void*>(x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
#pragma GCC diagnostic pop

template <typename T, int W>
cudaError_t launch_w(const Problem& p, const ConvArgs& a, cudaStream_t st) {
  const int D = p.dk, H = p.num_heads;
  const int C = H * D, rowb = C * (int)sizeof(T);
  if (p.total_tokens > 0 && rowb % 128 == 0) {  // the tiled kernel, slabs of 512, 256 or 128 B
    auto tiled = [&](auto sb) -> cudaError_t {
      constexpr int SB = decltype(sb)::value;
      constexpr int kDyn = tile_smem<T, SB>();
      static PerDeviceInit attrs;
      cudaError_t e = attrs.run([] {
        return cudaFuncSetAttribute(conv_tile_kernel<T, W, SB>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kDyn);
      });
      if (e != cudaSuccess) return e;
      int dev = 0, sms = 0;
      if (cudaGetDevice(&dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidDevice;
      using TS = TileShape<T, SB>;
      const long long items =
          (long long)((p.total_tokens + TS::TILE - 1) / TS::TILE) * (C / (SB / (int)sizeof(T)));
      const int slabs = C / (SB / (int)sizeof(T));
      // two CTAs per SM, a multiple of the slab count (each CTA keeps one slab's taps)
      long long nb = 2LL * sms;
      if (nb >= slabs) nb -= nb % slabs;
      const unsigned blocks = (unsigned)std::min<long long>(items, nb);
      CUtensorMap map;
      if (!encode_rows(&map, a.x, sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                       (int)sizeof(T), C, p.total_tokens, SB / (int)sizeof(T), TS::ROWS))
        return cudaErrorInvalidValue;
      conv_tile_kernel<T, W, SB><<<blocks, kNT, kDyn, st>>>(
          map, a.weight, a.state_in, a.cu_seqlens, p.num_seqs, p.total_tokens, C,
          static_cast<T*>(a.y), a.err);
      return cudaGetLastError();
    };
    cudaError_t e = rowb % 512 == 0 ? tiled(std::integral_constant<int, 512>{})
                    : rowb % 256 == 0 ? tiled(std::integral_constant<int, 256>{})
                                      : tiled(std::integral_constant<int, 128>{});
    if (e != cudaSuccess) return e;
  } else if (p.total_tokens > 0) {
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
