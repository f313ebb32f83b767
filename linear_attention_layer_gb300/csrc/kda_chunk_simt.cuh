// kda_chunk_simt.cuh -- chunked KDA prefill on CUDA cores, fp32 throughout.
//
// The chunked form of the recurrence (mhpq.cn/news/56770, section
// "KDA 到底在算什么"), evaluated 16 tokens at a time.  Within a chunk, with
// G_t the inclusive cumulative sum of the log-decay g over the chunk (per key
// channel) and S_0 the entry state:
//
//   U = (I + A)^{-1} diag(beta) (V - K+ S_0),  A[t,j] = beta_t sum_c k_tc k_jc e^{G_tc - G_jc}  (j < t)
//   O = Q+ S_0 + P U,                          P[t,j] = sum_c q_tc k_jc e^{G_tc - G_jc}           (j <= t)
//   S_C = Diag(e^{G_C}) S_0 + Khat^T U,        Khat_t = k_t * e^{G_C - G_t}
//
// with Q+ = q * e^{G}, K+ = k * e^{G}.  The pairwise factor e^{G_t - G_j} is
// evaluated as (x e^{G_t}) . (y e^{-G_j}): the reciprocal decay e^{-G_j}
// stays below e^80 because a 16-token chunk cannot decay by more than
// 16 * 5 (blog.higcp.com "猜想：K3 可能是最适合 TPU 的 MoE 架构", section
// "下界衰减": the lower-bounded gate keeps a 16-token tile's cumulative
// log-decay in (-80, 0)), well inside fp32.
//
// (I + A) is unit lower triangular, so U comes from forward substitution,
// one value column at a time.  Each value column of S evolves on its own,
// which gives the thread layout: 2*dv threads, thread (n, half) owns column
// n of S for half of the dk rows, in registers.  This path serves fp32 io
// (where it must match the fp64 recurrence to 1e-4) and every size the
// tensor-core path does not cover.
#pragma once
#include "kda_common.cuh"
#include "kda_launch.h"

namespace kda {
namespace simt {

constexpr int kC = 16;  // chunk length (one decay tile)

template <int DK, int DV>
struct SimtSmem {
  float qp[kC][DK + 1];  // q^ e^{G}
  float kp[kC][DK + 1];  // k^ e^{G}
  float km[kC][DK + 1];  // k^ e^{-G}
  float kh[kC][DK + 1];  // k^ e^{G_C - G}
  float vs[kC][DV];
  float akk[kC][kC + 1];
  float aqk[kC][kC + 1];
  float decay_last[DK];  // e^{G_C}
  float beta[kC];
  float rq[kC], rk[kC];
};

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(2 * DV)
chunk_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                  const float* __restrict__ z, const float* __restrict__ beta,
                  const float* initial_state, const int32_t* __restrict__ cu, T* __restrict__ out,
                  float* final_state, int H, int total, int* err,
                  const float* __restrict__ a_log, float* ckpt,
                  const int32_t* __restrict__ ckpt_off, int ckpt_every, int zhead) {
  constexpr int NT = 2 * DV;
  constexpr int NW = NT / 32;
  constexpr int RH = DK / 2;  // rows per thread
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtSmem<DK, DV>& sm = *reinterpret_cast<SimtSmem<DK, DV>*>(smem_raw);

  const int n = blockIdx.x / H, h = blockIdx.x % H;
  int bos, eos;
  if (!seq_range(cu, n, total, err, bos, eos)) return;
  const float zscale = gate_scale(a_log, h);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int col = tid >> 1, half = tid & 1, row0 = half * RH;

  const size_t sbase = (size_t)blockIdx.x * DK * DV;
  float s[RH];
#pragma unroll
  for (int i = 0; i < RH; ++i)
    s[i] = initial_state ? initial_state[sbase + (size_t)(row0 + i) * DV + col] : 0.f;

  for (int c0 = bos; c0 < eos; c0 += kC) {
    const int len = min(kC, eos - c0);
    __syncthreads();  // previous chunk done with shared memory
    // ---- load: raw q, k into qp / kp, log-decay into km, v, beta ----
    for (int idx = tid; idx < kC * DK; idx += NT) {
      const int t = idx / DK, c = idx % DK;
      float a = 0.f, b = 0.f, g = 0.f;
      if (t < len) {
        const size_t o = ((size_t)(c0 + t) * H + h) * DK + c;
        a = IO<T>::ld(q + o);
        b = IO<T>::ld(k + o);
        g = log_decay(zscale * __ldg(zhead ? z + (size_t)(c0 + t) * H + h : z + o));
      }
      sm.qp[t][c] = a;
      sm.kp[t][c] = b;
      sm.km[t][c] = g;
    }
    for (int idx = tid; idx < kC * DV; idx += NT) {
      const int t = idx / DV, j = idx % DV;
      sm.vs[t][j] = t < len ? IO<T>::ld(v + ((size_t)(c0 + t) * H + h) * DV + j) : 0.f;
    }
    if (tid < kC) sm.beta[tid] = tid < len ? __ldg(beta + (size_t)(c0 + tid) * H + h) : 0.f;
    __syncthreads();
    // ---- L2 norms of q_t, k_t ----
    for (int t = warp; t < kC; t += NW) {
      float qq = 0.f, kk = 0.f;
      for (int c = lane; c < DK; c += 32) {
        qq += sm.qp[t][c] * sm.qp[t][c];
        kk += sm.kp[t][c] * sm.kp[t][c];
      }
      qq = warp_sum(qq);
      kk = warp_sum(kk);
      if (lane == 0) {
        sm.rq[t] = rsqrtf(qq + kNormEps);
        sm.rk[t] = rsqrtf(kk + kNormEps);
      }
    }
    __syncthreads();
    // ---- cumulative decay and decayed operands, one key channel per thread ----
    for (int c = tid; c < DK; c += NT) {
      float G = 0.f;
#pragma unroll
      for (int t = 0; t < kC; ++t) {
        G += sm.km[t][c];
        const float eg = __expf(G), emg = __expf(-G);
        const float qn = sm.qp[t][c] * sm.rq[t], kn = sm.kp[t][c] * sm.rk[t];
        sm.qp[t][c] = qn * eg;
        sm.kp[t][c] = kn * eg;
        sm.km[t][c] = kn * emg;
      }
      const float eG = __expf(G);
      sm.decay_last[c] = eG;
#pragma unroll
      for (int t = 0; t < kC; ++t) sm.kh[t][c] = sm.km[t][c] * eG;
    }
    __syncthreads();
    // ---- A (strictly lower, scaled by beta_t) and P (lower incl. diagonal) ----
    for (int e = tid; e < kC * kC; e += NT) {
      const int t = e / kC, j = e % kC;
      float a = 0.f, p = 0.f;
      if (j <= t) {
        for (int c = 0; c < DK; ++c) {
          const float kmj = sm.km[j][c];
          a += sm.kp[t][c] * kmj;
          p += sm.qp[t][c] * kmj;
        }
      }
      sm.akk[t][j] = j < t ? sm.beta[t] * a : 0.f;
      sm.aqk[t][j] = p;
    }
    __syncthreads();
    // ---- per value column: K+ S_0, Q+ S_0, forward substitution, output ----
    float ks[kC], qs[kC];
#pragma unroll
    for (int t = 0; t < kC; ++t) {
      float a = 0.f, b = 0.f;
#pragma unroll
      for (int i = 0; i < RH; ++i) {
        a += sm.kp[t][row0 + i] * s[i];
        b += sm.qp[t][row0 + i] * s[i];
      }
      ks[t] = a + __shfl_xor_sync(0xffffffffu, a, 1);
      qs[t] = b + __shfl_xor_sync(0xffffffffu, b, 1);
    }
    float u[kC];
#pragma unroll
    for (int t = 0; t < kC; ++t) {
      float x = sm.beta[t] * (sm.vs[t][col] - ks[t]);
#pragma unroll
      for (int j = 0; j < t; ++j) x -= sm.akk[t][j] * u[j];
      u[t] = x;
    }
#pragma unroll
    for (int t = 0; t < kC; ++t) {
      float o = qs[t];
#pragma unroll
      for (int j = 0; j <= t; ++j) o += sm.aqk[t][j] * u[j];
      if (half == 0 && t < len) IO<T>::st(out + ((size_t)(c0 + t) * H + h) * DV + col, o);
    }
    // ---- state: S <- Diag(e^{G_C}) S + Khat^T U ----
#pragma unroll
    for (int i = 0; i < RH; ++i) {
      float x = sm.decay_last[row0 + i] * s[i];
#pragma unroll
      for (int t = 0; t < kC; ++t) x += sm.kh[t][row0 + i] * u[t];
      s[i] = x;
    }
    if (ckpt && (c0 + len - bos) % ckpt_every == 0) {  // state after a multiple of ckpt_every tokens
      const size_t j = (size_t)__ldg(ckpt_off + n) + (c0 + len - bos) / ckpt_every - 1;
      float* dst = ckpt + (j * H + h) * DK * DV;
#pragma unroll
      for (int i = 0; i < RH; ++i) dst[(size_t)(row0 + i) * DV + col] = s[i];
    }
  }
  if (final_state) {
#pragma unroll
    for (int i = 0; i < RH; ++i) final_state[sbase + (size_t)(row0 + i) * DV + col] = s[i];
  }
}

template <int DK, int DV, typename T>
cudaError_t dispatch(const Problem& p, const Args& a, cudaStream_t st) {
  const size_t smem = sizeof(SimtSmem<DK, DV>);
  auto kern = chunk_simt_kernel<DK, DV, T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const unsigned blocks = (unsigned)p.num_seqs * (unsigned)p.num_heads;
  kern<<<blocks, 2 * DV, smem, st>>>((const T*)a.q, (const T*)a.k, (const T*)a.v, a.z, a.beta,
                                     a.initial_state, a.cu_seqlens, (T*)a.out, a.final_state,
                                     p.num_heads, p.total_tokens, a.err, a.a_log, a.ckpt,
                                     a.ckpt_off, a.ckpt_every, a.gate_per_head);
  return cudaGetLastError();
}


template <int DK>
cudaError_t launch_dk(const Problem& p, const Args& a, cudaStream_t st) {
  switch (p.dv) {
    case 32: return p.io_bf16 ? dispatch<DK, 32, __nv_bfloat16>(p, a, st) : dispatch<DK, 32, float>(p, a, st);
    case 64: return p.io_bf16 ? dispatch<DK, 64, __nv_bfloat16>(p, a, st) : dispatch<DK, 64, float>(p, a, st);
    case 128: return p.io_bf16 ? dispatch<DK, 128, __nv_bfloat16>(p, a, st) : dispatch<DK, 128, float>(p, a, st);
    default: return cudaErrorInvalidValue;
  }
}

// One translation unit per key width instantiates launch_dk<DK>.
cudaError_t launch_dk32(const Problem& p, const Args& a, cudaStream_t st);
cudaError_t launch_dk64(const Problem& p, const Args& a, cudaStream_t st);
cudaError_t launch_dk128(const Problem& p, const Args& a, cudaStream_t st);

}  // namespace simt
}  // namespace kda
