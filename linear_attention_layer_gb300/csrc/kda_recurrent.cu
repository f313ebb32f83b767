// kda_recurrent.cu -- token-by-token KDA kernels: the decode step and the
// recurrent prefill.
//
// Both evaluate, for one (sequence, head), the state update and read-out of
// mhpq.cn/news/56770, section "KDA 到底在算什么", one token at a time:
//     Sbar = Diag(alpha_t) S_{t-1}
//     e    = v_t - Sbar^T k_t            (erase: what the key currently reads)
//     S_t  = Sbar + beta_t k_t e^T       (= (I - b k k^T) Sbar + b k v^T)
//     o_t  = S_t^T q_t = Sbar^T q_t + beta_t (k_t . q_t) e
// so one pass over S gives both reductions (Sbar^T k and Sbar^T q) and the
// write-back.  The decode step is the regime where that pass dominates: the
// fp32 state streams HBM -> registers -> HBM once per token with 128-bit
// coalesced accesses (blog.higcp.com "猜想：K3 可能是最适合 TPU 的 MoE 架构",
// section "三条容易被忽略的代价" (3), decode as its own regime).
//
// Thread layout: one CTA of 256 threads per (sequence, head).  A state row
// (dv floats) is covered by dv/4 threads holding one float4 each; the 1024/dv
// row groups of a CTA stride over the dk rows, so every thread holds
// R = dk*dv/1024 float4 of S (16 at dk = dv = 128) in registers.
#include "kda_common.cuh"
#include "kda_launch.h"

namespace kda {
namespace {

constexpr int kNT = 256;

template <int DK, int DV>
struct RecShape {
  static constexpr int TPR = DV / 4;    // threads per row
  static constexpr int RG = kNT / TPR;  // row groups
  static constexpr int R = DK / RG;     // rows (float4) per thread
  static_assert(DK % RG == 0 && R >= 1, "unsupported shape");
};

template <int DK, int DV>
struct RecSmem {
  float qs[DK], ks[DK], as[DK];
  float vs[DV], es[DV];
  float red[2][RecShape<DK, DV>::RG][DV];
  float part[3][kNT / 32];
  float onorm[kNT / 32];  // per-warp sums of o^2 (output norm)
};

// Optional pre- and post-processing fused into the decode-side kernels
// (kda_fusion_t): the short causal convolution + Swish of q and k before their
// L2 norm, and a per-head RMS norm of the outputs.
struct Fusion {
  int W;                 // convolution width, 0 = none
  const float* wq;       // [H, DK, W] taps (tap j multiplies x[t - (W-1) + j])
  const float* wk;
  float* sq;             // [B, H, DK, W-1] last W-1 raw inputs, oldest first
  float* sk;
  const float* onw;      // [H, DV] output-norm weight, or null
  float eps;
};

// The convolution of one channel (thread tid < DK) of q and of k: its taps
// and its last three raw inputs, right-aligned so that any width 1..4 is the
// same four-tap sum (unused taps are zero):
//   u = t[0] h[0] + t[1] h[1] + t[2] h[2] + t[3] x,   y = u sigmoid(u).
struct ConvRegs {
  float hq[3], hk[3], tq[4], tk[4];
};

__device__ __forceinline__ float swish(float u) { return __fdividef(u, 1.f + __expf(-u)); }

// One token of a channel's convolution: taps t[0..3] (registers or shared
// memory), history h advanced by the raw input x; returns the Swish output.
__device__ __forceinline__ float conv_step(float (&h)[3], const float* t, float x) {
  const float u = fmaf(t[0], h[0], fmaf(t[1], h[1], fmaf(t[2], h[2], t[3] * x)));
  h[0] = h[1];
  h[1] = h[2];
  h[2] = x;
  return swish(u);
}

// Load channel c's taps and history of (unit = b * H + h).
template <int DK>
__device__ __forceinline__ void conv_load(ConvRegs& cr, const Fusion& f, size_t unit, int h,
                                          int c) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int tj = j - (4 - f.W);  // tap index, < 0 for unused slots
    cr.tq[j] = tj >= 0 ? __ldg(f.wq + ((size_t)h * DK + c) * f.W + tj) : 0.f;
    cr.tk[j] = tj >= 0 ? __ldg(f.wk + ((size_t)h * DK + c) * f.W + tj) : 0.f;
  }
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const int sj = j - (4 - f.W);  // history index (W-1 kept), < 0 for unused slots
    cr.hq[j] = sj >= 0 ? f.sq[(unit * DK + c) * (f.W - 1) + sj] : 0.f;
    cr.hk[j] = sj >= 0 ? f.sk[(unit * DK + c) * (f.W - 1) + sj] : 0.f;
  }
}

template <int DK>
__device__ __forceinline__ void conv_store(const ConvRegs& cr, const Fusion& f, size_t unit, int c) {
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const int sj = j - (4 - f.W);
    if (sj >= 0) {
      f.sq[(unit * DK + c) * (f.W - 1) + sj] = cr.hq[j];
      f.sk[(unit * DK + c) * (f.W - 1) + sj] = cr.hk[j];
    }
  }
}

// Stage one token's q, k, alpha = exp(g), v into shared memory and the
// partial sums |q|^2, |k|^2, q.k per warp.
template <int DK, int DV, typename T, bool CONV = false>
__device__ __forceinline__ void stage_token(RecSmem<DK, DV>& sm, const T* qp, const T* kp,
                                            const T* vp, const float* zp, float zscale,
                                            bool zhead, ConvRegs* cr = nullptr,
                                            bool conv_on = false) {
  const int tid = threadIdx.x;
  float qq = 0.f, kk = 0.f, kq = 0.f;
  if (tid < DK) {
    float a = IO<T>::ld(qp + tid);
    float b = IO<T>::ld(kp + tid);
    if (CONV && conv_on) {  // raw inputs through this channel's convolution + Swish
      a = conv_step(cr->hq, cr->tq, a);
      b = conv_step(cr->hk, cr->tk, b);
    }
    sm.qs[tid] = a;
    sm.ks[tid] = b;
    sm.as[tid] = __expf(log_decay(zscale * __ldg(zp + (zhead ? 0 : tid))));
    qq = a * a;
    kk = b * b;
    kq = a * b;
  }
  if (tid < DV) sm.vs[tid] = IO<T>::ld(vp + tid);
  if (tid < ((DK + 31) & ~31)) {
    qq = warp_sum(qq);
    kk = warp_sum(kk);
    kq = warp_sum(kq);
    if ((tid & 31) == 0) {
      sm.part[0][tid >> 5] = qq;
      sm.part[1][tid >> 5] = kk;
      sm.part[2][tid >> 5] = kq;
    }
  }
}

// Apply one token to the register-resident state s.  Requires stage_token
// followed by __syncthreads().  Writes o_t (when op != nullptr).
template <int DK, int DV, typename T, bool ONORM = false>
__device__ __forceinline__ void apply_token(RecSmem<DK, DV>& sm, float4 (&s)[RecShape<DK, DV>::R],
                                            float b, T* op, const float* onw = nullptr,
                                            float eps = 0.f) {
  using SH = RecShape<DK, DV>;
  const int tid = threadIdx.x;
  const int c4 = tid % SH::TPR, rg = tid / SH::TPR;
  constexpr int NW = (DK + 31) / 32;
  float qq = 0.f, kk = 0.f, kq = 0.f;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    qq += sm.part[0][w];
    kk += sm.part[1][w];
    kq += sm.part[2][w];
  }
  const float rq = rsqrtf(qq + kNormEps), rk = rsqrtf(kk + kNormEps);
  float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
  for (int i = 0; i < SH::R; ++i) {
    const int r = rg + i * SH::RG;
    const float a = sm.as[r], kr = sm.ks[r] * rk, qr = sm.qs[r] * rq;
    s[i].x *= a; s[i].y *= a; s[i].z *= a; s[i].w *= a;
    pk.x += kr * s[i].x; pk.y += kr * s[i].y; pk.z += kr * s[i].z; pk.w += kr * s[i].w;
    pq.x += qr * s[i].x; pq.y += qr * s[i].y; pq.z += qr * s[i].z; pq.w += qr * s[i].w;
  }
  reinterpret_cast<float4*>(sm.red[0][rg])[c4] = pk;
  reinterpret_cast<float4*>(sm.red[1][rg])[c4] = pq;
  __syncthreads();
  float o = 0.f;
  if (tid < DV) {
    float sk = 0.f, sq = 0.f;
#pragma unroll
    for (int g = 0; g < SH::RG; ++g) {
      sk += sm.red[0][g][tid];
      sq += sm.red[1][g][tid];
    }
    const float e = sm.vs[tid] - sk;
    o = sq + b * (kq * rk * rq) * e;
    if (op && !ONORM) IO<T>::st(op + tid, o);
    sm.es[tid] = b * e;
  }
  if (ONORM && op && tid < DV) {  // per-warp sums of o^2 over the value channels
    const float o2 = warp_sum(o * o);
    if ((tid & 31) == 0) sm.onorm[tid >> 5] = o2;
  }
  __syncthreads();
  if (ONORM && op && tid < DV) {  // o / sqrt(mean(o^2) + eps) * weight
    float ss = 0.f;
#pragma unroll
    for (int w = 0; w < DV / 32; ++w) ss += sm.onorm[w];
    IO<T>::st(op + tid, o * rsqrtf(ss * (1.f / DV) + eps) * __ldg(onw + tid));
  }
  const float4 e4 = reinterpret_cast<const float4*>(sm.es)[c4];
#pragma unroll
  for (int i = 0; i < SH::R; ++i) {
    const float kr = sm.ks[rg + i * SH::RG] * rk;
    s[i].x += kr * e4.x; s[i].y += kr * e4.y; s[i].z += kr * e4.z; s[i].w += kr * e4.w;
  }
}

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kNT, 2)
decode_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
              const float* __restrict__ z, const float* __restrict__ beta,
              const float* __restrict__ a_log, int H, int zhead, float* __restrict__ state,
              T* __restrict__ out) {
  using SH = RecShape<DK, DV>;
  __shared__ __align__(16) RecSmem<DK, DV> sm;
  const size_t unit = blockIdx.x;  // n * H + h
  const int c4 = threadIdx.x % SH::TPR, rg = threadIdx.x / SH::TPR;
  float4* S = reinterpret_cast<float4*>(state + unit * DK * DV);
  float4 s[SH::R];
#pragma unroll
  for (int i = 0; i < SH::R; ++i) s[i] = ld_stream(S + (size_t)(rg + i * SH::RG) * SH::TPR + c4);
  stage_token<DK, DV, T>(sm, q + unit * DK, k + unit * DK, v + unit * DV,
                         z + unit * (zhead ? 1 : DK), gate_scale(a_log, (int)(unit % H)), zhead);
  __syncthreads();
  apply_token<DK, DV, T>(sm, s, __ldg(beta + unit), out + unit * DV);
#pragma unroll
  for (int i = 0; i < SH::R; ++i) st_stream(S + (size_t)(rg + i * SH::RG) * SH::TPR + c4, s[i]);
}

// decode_kernel with the fused pre- and post-processing of kda_fusion_t:
// q and k through the short convolution (whose state advances by this
// token), the outputs through the per-head RMS norm.
template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kNT, 2)
decode_fused_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                    const float* __restrict__ z, const float* __restrict__ beta,
                    const float* __restrict__ a_log, int H, int zhead, float* __restrict__ state,
                    T* __restrict__ out, const Fusion f) {
  using SH = RecShape<DK, DV>;
  __shared__ __align__(16) RecSmem<DK, DV> sm;
  const size_t unit = blockIdx.x;  // n * H + h
  const int h = (int)(unit % H);
  const int c4 = threadIdx.x % SH::TPR, rg = threadIdx.x / SH::TPR;
  float4* S = reinterpret_cast<float4*>(state + unit * DK * DV);
  float4 s[SH::R];
#pragma unroll
  for (int i = 0; i < SH::R; ++i) s[i] = ld_stream(S + (size_t)(rg + i * SH::RG) * SH::TPR + c4);
  const bool conv = f.W > 0;
  ConvRegs cr;
  if (conv && threadIdx.x < DK) conv_load<DK>(cr, f, unit, h, threadIdx.x);
  stage_token<DK, DV, T, true>(sm, q + unit * DK, k + unit * DK, v + unit * DV,
                               z + unit * (zhead ? 1 : DK), gate_scale(a_log, h), zhead, &cr,
                               conv);
  __syncthreads();
  if (f.onw)
    apply_token<DK, DV, T, true>(sm, s, __ldg(beta + unit), out + unit * DV,
                                 f.onw + (size_t)h * DV, f.eps);
  else
    apply_token<DK, DV, T>(sm, s, __ldg(beta + unit), out + unit * DV);
#pragma unroll
  for (int i = 0; i < SH::R; ++i) st_stream(S + (size_t)(rg + i * SH::RG) * SH::TPR + c4, s[i]);
  if (conv && threadIdx.x < DK) conv_store<DK>(cr, f, unit, threadIdx.x);
}

// Speculative decoding.  One CTA per (request, head).  A window's draft
// tokens of request b are rows [b*W, b*W + W) of its [B*W, H, .] inputs.
// With a replay part (rp.accept != null): the first accept[b] tokens of the
// previous window rp (0 <= accept[b] <= rp.W) are applied again and the
// state is written once, without outputs.  With a window part (wn.W > 0):
// the outputs of its W tokens, from the (replayed) state, which the window
// part does not write back.  Both parts in one launch read the state from
// HBM once and write it once.
template <typename T>
struct WinPart {
  const T* q;
  const T* k;
  const T* v;
  const float* z;
  const float* beta;
  int W;
  const int32_t* accept;  // replay part only
  bool vec;               // q, k, v (and per-channel z) 16-byte aligned: bulk copies
};

// The window kernel's thread layout: a thread holds four adjacent value
// columns (a column quad) of R consecutive key rows, and the RG threads of a
// quad are lanes of one warp (lane = g * QPW + quad within the warp), so the
// two sums over the key rows (Sbar^T k, Sbar^T q) are warp shuffles and each
// thread gets e for its own columns: a token needs one block barrier, with
// the next token staged into the other half of a double buffer meanwhile.
//
// The registers hold S~ = Gamma^{-1} S, Gamma = Diag of the decays' running
// product since the last renormalisation, so the decay costs no pass over
// the state: with K_G = Gamma_t k, Q_G = Gamma_t q (row scalings of the
// staged vectors), Sbar_t^T k = S~^T K_G, Sbar_t^T q = S~^T Q_G and the update
// is S~ += (Gamma_t^{-1} k) (beta e)^T.  S = Gamma S~ is formed every
// kWinRenorm tokens of a part (the decay of one token is at least e^{-5}, so
// Gamma stays above e^{-40}) and where the replayed state is stored; a part
// starts from Gamma = I, so the replay and the window give the same results
// in one call as in two.
template <int DK, int DV>
struct WinShape {
  static constexpr int QPW = DV / 32;  // column quads per warp
  static constexpr int RG = 32 / QPW;  // threads per quad
  static constexpr int R = DK / RG;    // key rows per thread
  static_assert(DV % 32 == 0 && kNT / 32 * QPW * 4 == DV && DK % RG == 0 && R >= 1,
                "unsupported shape");
};

template <int DK, int DV>
struct WinSmem {
  float kg[2][DK], qg[2][DK], ki[2][DK], gm[2][DK];  // Gamma k, Gamma q, Gamma^{-1} k, Gamma
  float vs[2][DV];
  float part[2][3][kNT / 32];  // per staging warp: |q|^2, |k|^2, q.k
  float onorm[2][kNT / 32];    // per warp: the sum of o^2 over its columns
  float os[2][DV];             // raw outputs awaiting the output norm
  float beta[2];
};

// A token's inputs as they are in global memory, copied into shared memory
// by cp.async three tokens ahead (no registers held meanwhile).
template <int DK, int DV, typename T>
struct WinRaw {
  T q[DK], k[DK], v[DV];
  float z[DK];
  float beta, zh;
  float pad[2];
};
constexpr int kWinSlots = 4;
constexpr int kWinRenorm = 8;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ float ld_raw(const float* p) { return *p; }
__device__ __forceinline__ float ld_raw(const __nv_bfloat16* p) { return __bfloat162float(*p); }

__device__ __forceinline__ void cp_async_b16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_b4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_pending() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// The copies of token row th of part p into slot x: one 16-byte piece (or a
// 4-byte scalar) per thread.
template <int DK, int DV, typename T>
__device__ __forceinline__ void win_copy(WinRaw<DK, DV, T>& x, const WinPart<T>& p, size_t th,
                                         bool zhead) {
  constexpr int QB = DK * (int)sizeof(T) / 16, VB = DV * (int)sizeof(T) / 16, ZB = DK / 4;
  constexpr int QE = 16 / (int)sizeof(T);  // elements per piece
  int t = threadIdx.x;
  if (!p.vec) {  // element by element
    if (t < DK) {
      x.q[t] = p.q[th * DK + t];
      x.k[t] = p.k[th * DK + t];
      if (!zhead) x.z[t] = __ldg(p.z + th * DK + t);
    }
    if (t < DV) x.v[t] = p.v[th * DV + t];
    if (t == 0) {
      x.beta = __ldg(p.beta + th);
      if (zhead) x.zh = __ldg(p.z + th);
    }
    return;
  }
  if (t < QB) {
    cp_async_b16(x.q + QE * t, p.q + th * DK + QE * t);
  } else if ((t -= QB) < QB) {
    cp_async_b16(x.k + QE * t, p.k + th * DK + QE * t);
  } else if ((t -= QB) < VB) {
    cp_async_b16(x.v + QE * t, p.v + th * DV + QE * t);
  } else if ((t -= VB) < ZB) {
    if (!zhead) cp_async_b16(x.z + 4 * t, p.z + th * DK + 4 * t);
  } else if ((t -= ZB) == 0) {
    cp_async_b4(&x.beta, p.beta + th);
  } else if (t == 1 && zhead) {
    cp_async_b4(&x.zh, p.z + th);
  }
}

// The fused convolution of one channel, in a shared-memory row of its own
// thread: taps of q then k (right-aligned as in ConvRegs), then the last
// three raw inputs of q then of k (an odd row length keeps the rows of a
// warp's threads in different banks).
constexpr int kConvRow = 15;
constexpr int kConvHq = 8, kConvHk = 11;

// Token j of the unit (whose part starts afresh when `fresh`): q, k (through
// the fused convolution), the decay's running product gam (this channel's,
// kept by its thread), v and beta from the raw slot into buffer `bf`, with
// the per-warp partial sums |q|^2, |k|^2, q.k of the convolved q, k.
template <int DK, int DV, typename T, bool CONV>
__device__ __forceinline__ void win_stage(WinSmem<DK, DV>& sm, int bf, const WinRaw<DK, DV, T>& x,
                                          float zscale, bool zhead, bool fresh, float& gam,
                                          float (*conv_rows)[kConvRow], bool conv_on) {
  const int tid = threadIdx.x;
  if (tid < DK) {
    float a = ld_raw(x.q + tid), b = ld_raw(x.k + tid);
    if (CONV && conv_on) {
      float* const r = conv_rows[tid];
      float hq[3] = {r[kConvHq], r[kConvHq + 1], r[kConvHq + 2]};
      float hk[3] = {r[kConvHk], r[kConvHk + 1], r[kConvHk + 2]};
      a = conv_step(hq, r, a);
      b = conv_step(hk, r + 4, b);
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        r[kConvHq + j] = hq[j];
        r[kConvHk + j] = hk[j];
      }
    }
    const float al = __expf(log_decay(zscale * (zhead ? x.zh : x.z[tid])));
    gam = fresh ? al : gam * al;
    sm.kg[bf][tid] = b * gam;
    sm.qg[bf][tid] = a * gam;
    sm.ki[bf][tid] = __fdividef(b, gam);
    sm.gm[bf][tid] = gam;
    const float qq = warp_sum(a * a), kk = warp_sum(b * b), kq = warp_sum(a * b);
    if ((tid & 31) == 0) {
      sm.part[bf][0][tid >> 5] = qq;
      sm.part[bf][1][tid >> 5] = kk;
      sm.part[bf][2][tid >> 5] = kq;
    }
  }
  if (tid < DV) sm.vs[bf][tid] = ld_raw(x.v + tid);
  if (tid == 0) sm.beta[bf] = x.beta;
}

// V consecutive floats of shared memory (V = 4, 2 or 1, aligned to V floats)
template <int V>
__device__ __forceinline__ void lds_v(float (&d)[V], const float* p) {
  if constexpr (V == 4) {
    const float4 t = *reinterpret_cast<const float4*>(p);
    d[0] = t.x; d[1] = t.y; d[2] = t.z; d[3] = t.w;
  } else if constexpr (V == 2) {
    const float2 t = *reinterpret_cast<const float2*>(p);
    d[0] = t.x; d[1] = t.y;
  } else {
    d[0] = *p;
  }
}

template <typename T>
__device__ __forceinline__ void st4_io(T* p, float4 o) {
  IO<T>::st(p, o.x);
  IO<T>::st(p + 1, o.y);
  IO<T>::st(p + 2, o.z);
  IO<T>::st(p + 3, o.w);
}

template <int DK, int DV, typename T, bool FUSED = false>
__global__ void __launch_bounds__(kNT, 2)
window_kernel(WinPart<T> rp, WinPart<T> wn, const float* __restrict__ a_log, int H, int zhead,
              float* __restrict__ state, T* __restrict__ out, int* err, const Fusion f) {
  using SH = WinShape<DK, DV>;
  static_assert(!FUSED || (DK <= kNT - 32 && DV <= 128), "the last warp stages no q or k");
  __shared__ __align__(16) WinSmem<DK, DV> sm;
  __shared__ __align__(16) WinRaw<DK, DV, T> raw[kWinSlots];
  __shared__ float conv_rows[FUSED ? DK : 1][kConvRow];
  const size_t unit = blockIdx.x;  // b * H + h
  const int b = (int)(unit / H), h = (int)(unit % H);
  int nrep = 0;
  if (rp.accept) {
    nrep = __ldg(rp.accept + b);
    if (nrep < 0 || nrep > rp.W) {  // bad acceptance length: leave this request alone
      if (threadIdx.x == 0) report_error(err, kErrDeviceCheck);
      return;
    }
  }
  const int ntok = nrep + wn.W;
  if (ntok == 0) return;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane / SH::QPW;                        // row group: rows [g R, g R + R)
  const int c = 4 * (w * SH::QPW + lane % SH::QPW);    // first of this thread's columns
  // token i (the replayed tokens first, then the window's) into its raw slot;
  // one commit group per token, empty past the last
  auto fetch = [&](int i) {
    if (i < nrep)
      win_copy<DK, DV, T>(raw[i % kWinSlots], rp, ((size_t)b * rp.W + i) * H + h, zhead);
    else if (i < ntok)
      win_copy<DK, DV, T>(raw[i % kWinSlots], wn, ((size_t)b * wn.W + (i - nrep)) * H + h, zhead);
    cp_async_commit();
  };
  fetch(0);
  fetch(1);
  fetch(2);
  float4* S = reinterpret_cast<float4*>(state + unit * DK * DV);
  float4 s[SH::R];
#pragma unroll
  for (int i = 0; i < SH::R; ++i) s[i] = ld_stream(S + ((size_t)(g * SH::R + i) * DV + c) / 4);
  const float zscale = gate_scale(a_log, h);
  // (fused) the convolution history of this thread's channel; the replayed
  // tokens advance it and it is stored with the state, the window's drafts
  // advance only this copy
  const bool conv = FUSED && f.W > 0;
  if (conv && threadIdx.x < DK) {
    ConvRegs cr;
    conv_load<DK>(cr, f, unit, h, threadIdx.x);
    float* const r = conv_rows[threadIdx.x];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      r[j] = cr.tq[j];
      r[4 + j] = cr.tk[j];
    }
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      r[kConvHq + j] = cr.hq[j];
      r[kConvHk + j] = cr.hk[j];
    }
  }
  auto conv_save = [&]() {  // the history after the replayed tokens
    if (conv && threadIdx.x < DK) {
      ConvRegs cr;
      const float* const r = conv_rows[threadIdx.x];
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        cr.hq[j] = r[kConvHq + j];
        cr.hk[j] = r[kConvHk + j];
      }
      conv_store<DK>(cr, f, unit, threadIdx.x);
    }
  };
  // a part (replay, window) starts afresh, and renormalises every kWinRenorm tokens
  auto fresh = [&](int j) { return j == nrep || (j < nrep ? j : j - nrep) % kWinRenorm == 0; };
  float gam = 1.f;  // (staging threads) this channel's running decay product
  const bool onorm = FUSED && f.onw != nullptr;
  // (output norm) token i's raw outputs wait in sm.os[i & 1] for the next
  // barrier; the last warp, which stages no q or k, scales and stores them
  auto finish = [&](int i) {
    if (w != kNT / 32 - 1 || 4 * lane >= DV) return;
    const int cc = 4 * lane;
    float ss = 0.f;
#pragma unroll
    for (int ww = 0; ww < kNT / 32; ++ww) ss += sm.onorm[i & 1][ww];
    const float r = rsqrtf(ss * (1.f / DV) + f.eps);
    const float4 o = *reinterpret_cast<const float4*>(&sm.os[i & 1][cc]);
    const float4 gm = __ldg(reinterpret_cast<const float4*>(f.onw + (size_t)h * DV + cc));
    st4_io(out + (((size_t)b * wn.W + (i - nrep)) * H + h) * DV + cc,
           make_float4(o.x * r * gm.x, o.y * r * gm.y, o.z * r * gm.z, o.w * r * gm.w));
  };

  cp_async_wait_pending<2>();  // token 0's copies (this thread's)
  __syncthreads();             // ... and every thread's
  win_stage<DK, DV, T, FUSED>(sm, 0, raw[0], zscale, zhead, true, gam, conv_rows, conv);
  if (nrep == 1) conv_save();
  cp_async_wait_pending<1>();  // token 1's
  for (int i = 0; i < ntok; ++i) {
    const int bf = i & 1;
    __syncthreads();  // token i staged; token i - 1's buffer read by every thread
    if (onorm && i > nrep) finish(i - 1);  // the previous token's outputs, normalised
    if (i + 1 < ntok) {  // token i + 1 into the other buffer
      win_stage<DK, DV, T, FUSED>(sm, bf ^ 1, raw[(i + 1) % kWinSlots], zscale, zhead,
                                  fresh(i + 1), gam, conv_rows, conv);
      if (i + 2 == nrep) conv_save();
    }
    fetch(i + 3);  // into the slot of token i - 1, staged before the barrier above
    // token i
    float qq = 0.f, kk = 0.f, kq = 0.f;
#pragma unroll
    for (int ww = 0; ww < (DK + 31) / 32; ++ww) {
      qq += sm.part[bf][0][ww];
      kk += sm.part[bf][1][ww];
      kq += sm.part[bf][2][ww];
    }
    const float rq = rsqrtf(qq + kNormEps), rk = rsqrtf(kk + kNormEps);
    const float bt = sm.beta[bf];
    constexpr int V = SH::R % 4 == 0 ? 4 : (SH::R % 2 == 0 ? 2 : 1);
    float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
    for (int j0 = 0; j0 < SH::R; j0 += V) {
      float kv[V], qv[V];
      lds_v<V>(kv, &sm.kg[bf][g * SH::R + j0]);
      lds_v<V>(qv, &sm.qg[bf][g * SH::R + j0]);
#pragma unroll
      for (int u = 0; u < V; ++u) {
        const float4 x = s[j0 + u];
        pk.x += kv[u] * x.x; pk.y += kv[u] * x.y; pk.z += kv[u] * x.z; pk.w += kv[u] * x.w;
        pq.x += qv[u] * x.x; pq.y += qv[u] * x.y; pq.z += qv[u] * x.z; pq.w += qv[u] * x.w;
      }
    }
#pragma unroll
    for (int o = SH::QPW; o < 32; o <<= 1) {  // over the row groups of this quad
      pk.x += __shfl_xor_sync(0xffffffffu, pk.x, o);
      pk.y += __shfl_xor_sync(0xffffffffu, pk.y, o);
      pk.z += __shfl_xor_sync(0xffffffffu, pk.z, o);
      pk.w += __shfl_xor_sync(0xffffffffu, pk.w, o);
      pq.x += __shfl_xor_sync(0xffffffffu, pq.x, o);
      pq.y += __shfl_xor_sync(0xffffffffu, pq.y, o);
      pq.z += __shfl_xor_sync(0xffffffffu, pq.z, o);
      pq.w += __shfl_xor_sync(0xffffffffu, pq.w, o);
    }
    const float4 v4 = *reinterpret_cast<const float4*>(&sm.vs[bf][c]);
    // e = v - Sbar^T k^ ; o = Sbar^T q^ + beta (k^ . q^) e ; S~ += Gamma^{-1} k^ beta e^T
    const float4 e = make_float4(v4.x - pk.x * rk, v4.y - pk.y * rk, v4.z - pk.z * rk,
                                 v4.w - pk.w * rk);
    if (i >= nrep) {
      const float m = bt * (kq * rk * rq);
      const float4 o = make_float4(pq.x * rq + m * e.x, pq.y * rq + m * e.y,
                                   pq.z * rq + m * e.z, pq.w * rq + m * e.w);
      if (onorm) {  // normalised after the next barrier, when every warp's sum is in
        float ss = g == 0 ? o.x * o.x + o.y * o.y + o.z * o.z + o.w * o.w : 0.f;
#pragma unroll
        for (int q = 1; q < SH::QPW; q <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, q);
        if (lane == 0) sm.onorm[bf][w] = ss;
        if (g == 0) *reinterpret_cast<float4*>(&sm.os[bf][c]) = o;
      } else if (g == 0) {
        st4_io(out + (((size_t)b * wn.W + (i - nrep)) * H + h) * DV + c, o);
      }
    }
    const float bk = bt * rk;
    const float4 be = make_float4(bk * e.x, bk * e.y, bk * e.z, bk * e.w);
#pragma unroll
    for (int j0 = 0; j0 < SH::R; j0 += V) {
      float kv[V];
      lds_v<V>(kv, &sm.ki[bf][g * SH::R + j0]);
#pragma unroll
      for (int u = 0; u < V; ++u) {
        float4& x = s[j0 + u];
        x.x += kv[u] * be.x; x.y += kv[u] * be.y; x.z += kv[u] * be.z; x.w += kv[u] * be.w;
      }
    }
    if (i + 1 < ntok ? fresh(i + 1) : i + 1 == nrep) {  // S = Gamma S~
#pragma unroll
      for (int j0 = 0; j0 < SH::R; j0 += V) {
        float gv[V];
        lds_v<V>(gv, &sm.gm[bf][g * SH::R + j0]);
#pragma unroll
        for (int u = 0; u < V; ++u) {
          float4& x = s[j0 + u];
          x.x *= gv[u]; x.y *= gv[u]; x.z *= gv[u]; x.w *= gv[u];
        }
      }
    }
    if (i + 1 == nrep) {  // the replayed state, written once
#pragma unroll
      for (int j = 0; j < SH::R; ++j) st_stream(S + ((size_t)(g * SH::R + j) * DV + c) / 4, s[j]);
    }
    cp_async_wait_pending<1>();  // token i + 2's copies, staged after the next barrier
  }
  if (onorm && ntok > nrep) {  // the last token's outputs
    __syncthreads();
    finish(ntok - 1);
  }
}

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kNT, 2)
recurrent_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                 const float* __restrict__ z, const float* __restrict__ beta,
                 const float* initial_state, const int32_t* __restrict__ cu, T* __restrict__ out,
                 float* final_state, int H, int total, int* err, const float* __restrict__ a_log,
                 float* ckpt, const int32_t* __restrict__ ckpt_off, int ckpt_every, int zhead) {
  using SH = RecShape<DK, DV>;
  __shared__ __align__(16) RecSmem<DK, DV> sm;
  const int n = blockIdx.x / H, h = blockIdx.x % H;
  int bos, eos;
  if (!seq_range(cu, n, total, err, bos, eos)) return;
  const int c4 = threadIdx.x % SH::TPR, rg = threadIdx.x / SH::TPR;
  const size_t sbase = (size_t)blockIdx.x * DK * DV;
  float4 s[SH::R];
#pragma unroll
  for (int i = 0; i < SH::R; ++i) {
    s[i] = initial_state
               ? __ldg(reinterpret_cast<const float4*>(initial_state + sbase) +
                       (size_t)(rg + i * SH::RG) * SH::TPR + c4)
               : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const float zscale = gate_scale(a_log, h);
  for (int t = bos; t < eos; ++t) {
    const size_t th = (size_t)t * H + h;
    __syncthreads();  // previous token finished reading shared memory
    stage_token<DK, DV, T>(sm, q + th * DK, k + th * DK, v + th * DV, z + th * (zhead ? 1 : DK),
                           zscale, zhead);
    __syncthreads();
    apply_token<DK, DV, T>(sm, s, __ldg(beta + th), out + th * DV);
    if (ckpt && (t + 1 - bos) % ckpt_every == 0) {  // state after a multiple of ckpt_every tokens
      const size_t j = (size_t)__ldg(ckpt_off + n) + (t + 1 - bos) / ckpt_every - 1;
      float4* dst = reinterpret_cast<float4*>(ckpt + (j * H + h) * DK * DV);
#pragma unroll
      for (int i = 0; i < SH::R; ++i) dst[(size_t)(rg + i * SH::RG) * SH::TPR + c4] = s[i];
    }
  }
  if (final_state) {
#pragma unroll
    for (int i = 0; i < SH::R; ++i)
      reinterpret_cast<float4*>(final_state + sbase)[(size_t)(rg + i * SH::RG) * SH::TPR + c4] = s[i];
  }
}

// Small states (dv = 32, dk <= 64): one warp per (sequence, head), lane j
// holding value column j of S (dk floats in registers), four warps per CTA.
// A token costs no block barrier: its q, k and retentions go through the
// warp's own shared-memory rows, both reductions over the key channels
// (S^T k and S^T q) are per-lane sums, and the rank-one write is per lane.
// Used for short latency-bound calls where a block per unit would spend its
// time in barriers.
constexpr int kSmallWarps = 4;

template <int DK, typename T>
__global__ void __launch_bounds__(32 * kSmallWarps)
recurrent_small_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                       const float* __restrict__ z, const float* __restrict__ beta,
                       const float* initial_state, const int32_t* __restrict__ cu,
                       T* __restrict__ out, float* final_state, int H, int total, int units,
                       int* err, const float* __restrict__ a_log, float* ckpt,
                       const int32_t* __restrict__ ckpt_off, int ckpt_every, int zhead) {
  constexpr int DV = 32, CPL = DK / 32;  // channels staged per lane
  __shared__ __align__(16) float sh[kSmallWarps][3][DK];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x * kSmallWarps + w;
  if (unit >= units) return;
  const int n = unit / H, h = unit % H;
  int bos, eos;
  if (!seq_range(cu, n, total, lane == 0 ? err : nullptr, bos, eos)) return;
  const size_t sbase = (size_t)unit * DK * DV;
  float s[DK];
#pragma unroll
  for (int c = 0; c < DK; ++c)
    s[c] = initial_state ? __ldg(initial_state + sbase + (size_t)c * DV + lane) : 0.f;
  const float zscale = gate_scale(a_log, h);
  float* qs = sh[w][0];
  float* ks = sh[w][1];
  float* as = sh[w][2];
  // this lane's inputs of the next two tokens, loaded ahead so that a token's
  // global-memory latency hides behind the work of the tokens before it
  struct In {
    float q[CPL], k[CPL], z[CPL], v, b;
  };
  In n1{}, n2{};
  auto fetch = [&](In& x, int t) {
    if (t >= eos) return;
    const size_t th = (size_t)t * H + h;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int c = lane + 32 * i;
      x.q[i] = IO<T>::ld(q + th * DK + c);
      x.k[i] = IO<T>::ld(k + th * DK + c);
      x.z[i] = __ldg(z + th * (zhead ? 1 : DK) + (zhead ? 0 : c));
    }
    x.v = IO<T>::ld(v + th * DV + lane);
    x.b = __ldg(beta + th);
  };
  fetch(n1, bos);
  fetch(n2, bos + 1);
  for (int t = bos; t < eos; ++t) {
    const size_t th = (size_t)t * H + h;
    const In cur = n1;
    n1 = n2;
    fetch(n2, t + 2);
    float qq = 0.f, kk = 0.f, kq = 0.f;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int c = lane + 32 * i;
      const float a = cur.q[i], b = cur.k[i];
      qs[c] = a;
      ks[c] = b;
      as[c] = __expf(log_decay(zscale * cur.z[i]));
      qq += a * a;
      kk += b * b;
      kq += a * b;
    }
    const float vj = cur.v;
    const float bt = cur.b;
    qq = warp_sum(qq);
    kk = warp_sum(kk);
    kq = warp_sum(kq);
    __syncwarp();
    const float rq = rsqrtf(qq + kNormEps), rk = rsqrtf(kk + kNormEps);
    float ek[4] = {0.f, 0.f, 0.f, 0.f}, eq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < DK; c += 4) {
      const float4 a4 = *reinterpret_cast<const float4*>(as + c);
      const float4 k4 = *reinterpret_cast<const float4*>(ks + c);
      const float4 q4 = *reinterpret_cast<const float4*>(qs + c);
      s[c] *= a4.x; s[c + 1] *= a4.y; s[c + 2] *= a4.z; s[c + 3] *= a4.w;
      ek[0] = fmaf(s[c], k4.x, ek[0]); ek[1] = fmaf(s[c + 1], k4.y, ek[1]);
      ek[2] = fmaf(s[c + 2], k4.z, ek[2]); ek[3] = fmaf(s[c + 3], k4.w, ek[3]);
      eq[0] = fmaf(s[c], q4.x, eq[0]); eq[1] = fmaf(s[c + 1], q4.y, eq[1]);
      eq[2] = fmaf(s[c + 2], q4.z, eq[2]); eq[3] = fmaf(s[c + 3], q4.w, eq[3]);
    }
    const float e = vj - (ek[0] + ek[1] + ek[2] + ek[3]) * rk;
    const float o = (eq[0] + eq[1] + eq[2] + eq[3]) * rq + bt * (kq * rk * rq) * e;
    IO<T>::st(out + th * DV + lane, o);
    const float be = bt * e * rk;
#pragma unroll
    for (int c = 0; c < DK; c += 4) {
      const float4 k4 = *reinterpret_cast<const float4*>(ks + c);
      s[c] = fmaf(k4.x, be, s[c]); s[c + 1] = fmaf(k4.y, be, s[c + 1]);
      s[c + 2] = fmaf(k4.z, be, s[c + 2]); s[c + 3] = fmaf(k4.w, be, s[c + 3]);
    }
    if (ckpt && (t + 1 - bos) % ckpt_every == 0) {
      const size_t j = (size_t)__ldg(ckpt_off + n) + (t + 1 - bos) / ckpt_every - 1;
      float* dst = ckpt + (j * H + h) * DK * DV;
#pragma unroll
      for (int c = 0; c < DK; ++c) dst[(size_t)c * DV + lane] = s[c];
    }
    __syncwarp();  // this token's rows are read before the next overwrites them
  }
  if (final_state) {
#pragma unroll
    for (int c = 0; c < DK; ++c) final_state[sbase + (size_t)c * DV + lane] = s[c];
  }
}

// Small states (dv = 32, dk <= 64) with few (sequence, head) units: one
// 256-thread CTA per unit, the sequence in blocks of BLK tokens.  First all
// threads stage the block -- q and k normalised, the decays, beta, (q^.k^), v
// and the products below, none of which depends on the state -- in shared
// memory; then each warp runs the token loop for its own four value columns,
// lane (rg, col) holding key rows [rg R, rg R + R) of its column, the sums
// over the key rows by warp shuffles: no block barrier inside the token loop,
// and only the state chain left on it.
constexpr int kCtaNT = 256;
constexpr long long kCtaUnitsMax = 1024;  // (sequence, head) units for a CTA each

template <int DK>
struct CtaShape {
  static constexpr int BLK = DK == 64 ? 32 : 64;  // tokens per block
  static constexpr int TPK = kCtaNT / BLK;        // staging threads per token
  static constexpr int CH = DK / TPK;             // channels each stages
  static constexpr int R = DK / 8;                // key rows per thread
};

// The token loop takes four tokens at a time.  For a group j = 0..3 entered
// with state S, A_j the decays' running product over the group's tokens
// 0..j (per key row) and x_i = beta_i e_i:
//     Sbar_j^T k_j = K_j + sum_{i<j} c_ji x_i,   K_j = S^T (A_j k_j),
//     Sbar_j^T q_j = Q_j + sum_{i<j} d_ji x_i,   Q_j = S^T (A_j q_j),
//     c_ji = k_j . (A_j / A_i) k_i,  d_ji = q_j . (A_j / A_i) k_i,
//     e_j = v_j - Sbar_j^T k_j,  o_j = Sbar_j^T q_j + (q_j . k_j) x_j,
//     S' = A_3 S + sum_i (A_3 / A_i) k_i x_i^T,
// so one pass over the state gives the eight sums of a group (reduced by one
// round of shuffles), the e_j follow from a 4 x 4 triangular solve on
// scalars, and one more pass applies the group: the state chain is a quarter
// as long.  (k, q normalised; every ratio A_j / A_i is a product of decays,
// so nothing leaves the fp32 range.)  The c, d and the scaled key and query
// rows are staged with the block.  Checkpoints fall on group ends (the call
// takes checkpoint intervals in multiples of 64 tokens).
template <int DK, typename T>
__global__ void __launch_bounds__(kCtaNT, 1)
recurrent_cta_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                      const float* __restrict__ z, const float* __restrict__ beta,
                      const float* initial_state, const int32_t* __restrict__ cu,
                      T* __restrict__ out, float* final_state, int H, int total, int* err,
                      const float* __restrict__ a_log, float* ckpt,
                      const int32_t* __restrict__ ckpt_off, int ckpt_every, int zhead,
                      int vec) {
  using CS = CtaShape<DK>;
  constexpr int DV = 32, BLK = CS::BLK, R = CS::R, NG = BLK / 4;
  constexpr int TPG = kCtaNT / NG;  // group-staging threads per group
  constexpr int CPT = DK / TPG;  // channels per group-staging thread
  static_assert(CPT == 2, "two channels per group-staging thread");
  // per token: q^ then A_j q^, k^ then A_j k^, alpha then (A_3 / A_j) k^
  __shared__ __align__(16) float qs[BLK][DK], ks[BLK][DK], as[BLK][DK];
  __shared__ __align__(16) float a3s[NG][DK];
  __shared__ __align__(16) float vs[BLK][DV];
  __shared__ float bs[BLK], kqs[BLK];
  __shared__ float cds[NG][12];  // c10 c20 c21 c30 c31 c32, then d in the same order
  __shared__ float zh[BLK];      // (one gate per head) the block's logits
  // (16-byte aligned inputs) the block's raw q, k, v rows, copied in by cp.async
  // (fp32: straight into qs, ks, vs; bf16: here, then widened)
  constexpr bool kNarrow = sizeof(T) == 2;
  __shared__ __align__(16) T rawbuf[kNarrow ? BLK * (2 * DK + DV) : 8];
  T* const rq = kNarrow ? rawbuf : reinterpret_cast<T*>(&qs[0][0]);
  T* const rkk = kNarrow ? rawbuf + BLK * DK : reinterpret_cast<T*>(&ks[0][0]);
  T* const rv = kNarrow ? rawbuf + 2 * BLK * DK : reinterpret_cast<T*>(&vs[0][0]);
  const int n = blockIdx.x / H, h = blockIdx.x % H;
  int bos, eos;
  if (!seq_range(cu, n, total, threadIdx.x == 0 ? err : nullptr, bos, eos)) return;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col = 4 * w + (lane & 3), rg = lane >> 2;
  const size_t sbase = (size_t)blockIdx.x * DK * DV;
  float s[R];
#pragma unroll
  for (int i = 0; i < R; ++i)
    s[i] = initial_state ? __ldg(initial_state + sbase + (size_t)(rg * R + i) * DV + col) : 0.f;
  const float zscale = gate_scale(a_log, h);
  for (int b0 = bos; b0 < eos; b0 += BLK) {
    const int nb = min(BLK, eos - b0);
    __syncthreads();  // the previous block's rows are read
    if (vec) {  // the block's rows in one round trip: 16-byte pieces, every thread
      constexpr int QP = DK * (int)sizeof(T) / 16, VP = DV * (int)sizeof(T) / 16, ZP = DK / 4;
      constexpr int QE = 16 / (int)sizeof(T);  // elements per piece
      for (int i = threadIdx.x; i < nb * QP; i += kCtaNT) {
        const int t = i / QP, j = i % QP;
        const size_t th = (size_t)(b0 + t) * H + h;
        cp_async_b16(rq + t * DK + QE * j, q + th * DK + QE * j);
        cp_async_b16(rkk + t * DK + QE * j, k + th * DK + QE * j);
      }
      for (int i = threadIdx.x; i < nb * VP; i += kCtaNT) {
        const int t = i / VP, j = i % VP;
        cp_async_b16(rv + t * DV + QE * j, v + ((size_t)(b0 + t) * H + h) * DV + QE * j);
      }
      if (!zhead) {
        for (int i = threadIdx.x; i < nb * ZP; i += kCtaNT) {
          const int t = i / ZP, j = i % ZP;
          cp_async_b16(&as[t][4 * j], z + ((size_t)(b0 + t) * H + h) * DK + 4 * j);
        }
      }
      for (int t = threadIdx.x; t < nb; t += kCtaNT) {
        const size_t th = (size_t)(b0 + t) * H + h;
        cp_async_b4(&bs[t], beta + th);
        if (zhead) cp_async_b4(&zh[t], z + th);
      }
      cp_async_commit();
      cp_async_wait_pending<0>();
      __syncthreads();
    }
    {  // stage the tokens (rows past the sequence: k = q = v = 0, alpha = 1, beta = 0)
      const int t = threadIdx.x / CS::TPK, part = threadIdx.x % CS::TPK, c0 = part * CS::CH;
      float qq = 0.f, kk = 0.f, kq = 0.f;
      const bool live = t < nb;
      const size_t th = (size_t)(b0 + t) * H + h;
#pragma unroll
      for (int c = 0; c < CS::CH; ++c) {
        float a = 0.f, b = 0.f, zz = 0.f;
        if (live) {
          if (vec) {
            a = ld_raw(rq + t * DK + c0 + c);
            b = ld_raw(rkk + t * DK + c0 + c);
            zz = zhead ? zh[t] : as[t][c0 + c];
          } else {
            a = IO<T>::ld(q + th * DK + c0 + c);
            b = IO<T>::ld(k + th * DK + c0 + c);
            zz = __ldg(z + (zhead ? th : th * DK + c0 + c));
          }
        }
        qs[t][c0 + c] = a;
        ks[t][c0 + c] = b;
        as[t][c0 + c] = live ? __expf(log_decay(zscale * zz)) : 1.f;
        qq += a * a;
        kk += b * b;
        kq += a * b;
      }
#pragma unroll
      for (int c = part; c < DV; c += CS::TPK)
        vs[t][c] = live ? (vec ? ld_raw(rv + t * DV + c) : IO<T>::ld(v + th * DV + c)) : 0.f;
#pragma unroll
      for (int o = 1; o < CS::TPK; o <<= 1) {
        qq += __shfl_xor_sync(0xffffffffu, qq, o);
        kk += __shfl_xor_sync(0xffffffffu, kk, o);
        kq += __shfl_xor_sync(0xffffffffu, kq, o);
      }
      const float rq = rsqrtf(qq + kNormEps), rk = rsqrtf(kk + kNormEps);
#pragma unroll
      for (int c = 0; c < CS::CH; ++c) {
        qs[t][c0 + c] *= rq;
        ks[t][c0 + c] *= rk;
      }
      if (part == 0) {
        bs[t] = live ? (vec ? bs[t] : __ldg(beta + th)) : 0.f;
        kqs[t] = kq * rq * rk;
      }
    }
    __syncthreads();
    {  // per group: A_j, the scaled rows (in place) and c, d (TPG threads, CPT channels each)
      const int gi = threadIdx.x / TPG, p = threadIdx.x % TPG, c0 = CPT * p, t0 = 4 * gi;
      float kh[4][CPT], qh[4][CPT], al[4][CPT];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 k2 = *reinterpret_cast<const float2*>(&ks[t0 + j][c0]);
        const float2 q2 = *reinterpret_cast<const float2*>(&qs[t0 + j][c0]);
        const float2 a2 = *reinterpret_cast<const float2*>(&as[t0 + j][c0]);
        kh[j][0] = k2.x; kh[j][1] = k2.y;
        qh[j][0] = q2.x; qh[j][1] = q2.y;
        al[j][0] = a2.x; al[j][1] = a2.y;
      }
      float cd[12];
#pragma unroll
      for (int m = 0; m < 12; ++m) cd[m] = 0.f;
#pragma unroll
      for (int u = 0; u < CPT; ++u) {  // channel c0 + u
        float A[4];
        A[0] = al[0][u];
#pragma unroll
        for (int j = 1; j < 4; ++j) A[j] = A[j - 1] * al[j][u];
        // rho(j, i) = A_j / A_i as products of the decays in between
        const float r10 = al[1][u], r21 = al[2][u], r32 = al[3][u];
        const float r20 = r21 * r10, r31 = r32 * r21, r30 = r31 * r10;
        cd[0] += kh[1][u] * r10 * kh[0][u];
        cd[1] += kh[2][u] * r20 * kh[0][u];
        cd[2] += kh[2][u] * r21 * kh[1][u];
        cd[3] += kh[3][u] * r30 * kh[0][u];
        cd[4] += kh[3][u] * r31 * kh[1][u];
        cd[5] += kh[3][u] * r32 * kh[2][u];
        cd[6] += qh[1][u] * r10 * kh[0][u];
        cd[7] += qh[2][u] * r20 * kh[0][u];
        cd[8] += qh[2][u] * r21 * kh[1][u];
        cd[9] += qh[3][u] * r30 * kh[0][u];
        cd[10] += qh[3][u] * r31 * kh[1][u];
        cd[11] += qh[3][u] * r32 * kh[2][u];
        const float e3[4] = {r30, r31, r32, 1.f};  // A_3 / A_j
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          ks[t0 + j][c0 + u] = A[j] * kh[j][u];
          qs[t0 + j][c0 + u] = A[j] * qh[j][u];
          as[t0 + j][c0 + u] = e3[j] * kh[j][u];
        }
        a3s[gi][c0 + u] = A[3];
      }
#pragma unroll
      for (int o = 1; o < TPG; o <<= 1)
#pragma unroll
        for (int m = 0; m < 12; ++m) cd[m] += __shfl_xor_sync(0xffffffffu, cd[m], o);
      if (p == 0)
#pragma unroll
        for (int m = 0; m < 12; ++m) cds[gi][m] = cd[m];
    }
    __syncthreads();
    const int ngr = (nb + 3) / 4;
    for (int gi = 0; gi < ngr; ++gi) {
      const int t0 = 4 * gi;
      float K[4] = {0.f, 0.f, 0.f, 0.f}, Q[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i0 = 0; i0 < R; i0 += 4) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 k4 = *reinterpret_cast<const float4*>(&ks[t0 + j][rg * R + i0]);
          const float4 q4 = *reinterpret_cast<const float4*>(&qs[t0 + j][rg * R + i0]);
          K[j] = fmaf(k4.x, s[i0], K[j]); K[j] = fmaf(k4.y, s[i0 + 1], K[j]);
          K[j] = fmaf(k4.z, s[i0 + 2], K[j]); K[j] = fmaf(k4.w, s[i0 + 3], K[j]);
          Q[j] = fmaf(q4.x, s[i0], Q[j]); Q[j] = fmaf(q4.y, s[i0 + 1], Q[j]);
          Q[j] = fmaf(q4.z, s[i0 + 2], Q[j]); Q[j] = fmaf(q4.w, s[i0 + 3], Q[j]);
        }
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1)  // over the row groups of this column
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          K[j] += __shfl_xor_sync(0xffffffffu, K[j], o);
          Q[j] += __shfl_xor_sync(0xffffffffu, Q[j], o);
        }
      const float* const cd = cds[gi];
      float x[4];
      x[0] = bs[t0] * (vs[t0][col] - K[0]);
      x[1] = bs[t0 + 1] * (vs[t0 + 1][col] - K[1] - cd[0] * x[0]);
      x[2] = bs[t0 + 2] * (vs[t0 + 2][col] - K[2] - cd[1] * x[0] - cd[2] * x[1]);
      x[3] = bs[t0 + 3] * (vs[t0 + 3][col] - K[3] - cd[3] * x[0] - cd[4] * x[1] - cd[5] * x[2]);
      if (rg == 0) {
        const float o[4] = {Q[0] + kqs[t0] * x[0],
                            Q[1] + cd[6] * x[0] + kqs[t0 + 1] * x[1],
                            Q[2] + cd[7] * x[0] + cd[8] * x[1] + kqs[t0 + 2] * x[2],
                            Q[3] + cd[9] * x[0] + cd[10] * x[1] + cd[11] * x[2] +
                                kqs[t0 + 3] * x[3]};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (t0 + j < nb) IO<T>::st(out + ((size_t)(b0 + t0 + j) * H + h) * DV + col, o[j]);
      }
#pragma unroll
      for (int i0 = 0; i0 < R; i0 += 4) {
        const float4 a4 = *reinterpret_cast<const float4*>(&a3s[gi][rg * R + i0]);
        float4 e[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) e[j] = *reinterpret_cast<const float4*>(&as[t0 + j][rg * R + i0]);
        s[i0] = fmaf(e[3].x, x[3], fmaf(e[2].x, x[2], fmaf(e[1].x, x[1], fmaf(e[0].x, x[0], a4.x * s[i0]))));
        s[i0 + 1] = fmaf(e[3].y, x[3], fmaf(e[2].y, x[2], fmaf(e[1].y, x[1], fmaf(e[0].y, x[0], a4.y * s[i0 + 1]))));
        s[i0 + 2] = fmaf(e[3].z, x[3], fmaf(e[2].z, x[2], fmaf(e[1].z, x[1], fmaf(e[0].z, x[0], a4.z * s[i0 + 2]))));
        s[i0 + 3] = fmaf(e[3].w, x[3], fmaf(e[2].w, x[2], fmaf(e[1].w, x[1], fmaf(e[0].w, x[0], a4.w * s[i0 + 3]))));
      }
      const int done = min(t0 + 4, nb);  // tokens of the block applied
      if (ckpt && (b0 + done - bos) % ckpt_every == 0) {  // a checkpoint ends this group
        const size_t j = (size_t)__ldg(ckpt_off + n) + (b0 + done - bos) / ckpt_every - 1;
        float* dst = ckpt + (j * H + h) * DK * DV;
#pragma unroll
        for (int i = 0; i < R; ++i) dst[(size_t)(rg * R + i) * DV + col] = s[i];
      }
    }
  }
  if (final_state) {
#pragma unroll
    for (int i = 0; i < R; ++i) final_state[sbase + (size_t)(rg * R + i) * DV + col] = s[i];
  }
}

template <int DK, typename T>
cudaError_t cta_dispatch(const Problem& p, const Args& a, cudaStream_t st) {
  const unsigned blocks = (unsigned)p.num_seqs * (unsigned)p.num_heads;
  if (a.ckpt && a.ckpt_every % 4 != 0) return cudaErrorInvalidValue;  // the API takes 64s
  auto a16 = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
  const int vec = a16(a.q) && a16(a.k) && a16(a.v) && (a.gate_per_head || a16(a.z));
  recurrent_cta_kernel<DK, T><<<blocks, kCtaNT, 0, st>>>(
      (const T*)a.q, (const T*)a.k, (const T*)a.v, a.z, a.beta, a.initial_state, a.cu_seqlens,
      (T*)a.out, a.final_state, p.num_heads, p.total_tokens, a.err, a.a_log, a.ckpt, a.ckpt_off,
      a.ckpt_every, a.gate_per_head, vec);
  return cudaGetLastError();
}

template <int DK, typename T>
cudaError_t small_dispatch(const Problem& p, const Args& a, cudaStream_t st) {
  const int units = p.num_seqs * p.num_heads;
  const unsigned blocks = (unsigned)((units + kSmallWarps - 1) / kSmallWarps);
  recurrent_small_kernel<DK, T><<<blocks, 32 * kSmallWarps, 0, st>>>(
      (const T*)a.q, (const T*)a.k, (const T*)a.v, a.z, a.beta, a.initial_state, a.cu_seqlens,
      (T*)a.out, a.final_state, p.num_heads, p.total_tokens, units, a.err, a.a_log, a.ckpt,
      a.ckpt_off, a.ckpt_every, a.gate_per_head);
  return cudaGetLastError();
}

template <int DK, int DV, typename T>
cudaError_t decode_dispatch(const Problem& p, const void* q, const void* k, const void* v,
                            const float* z, const float* beta, const float* a_log, int zhead,
                            float* state, void* out, cudaStream_t st) {
  const unsigned blocks = (unsigned)p.num_seqs * (unsigned)p.num_heads;
  decode_kernel<DK, DV, T><<<blocks, kNT, 0, st>>>(
      (const T*)q, (const T*)k, (const T*)v, z, beta, a_log, p.num_heads, zhead, state, (T*)out);
  return cudaGetLastError();
}

template <int DK, int DV, typename T>
cudaError_t decode_fused_dispatch(const Problem& p, const void* q, const void* k, const void* v,
                                  const float* z, const float* beta, const float* a_log,
                                  int zhead, float* state, void* out, const Fusion& f,
                                  cudaStream_t st) {
  const unsigned blocks = (unsigned)p.num_seqs * (unsigned)p.num_heads;
  decode_fused_kernel<DK, DV, T><<<blocks, kNT, 0, st>>>(
      (const T*)q, (const T*)k, (const T*)v, z, beta, a_log, p.num_heads, zhead, state, (T*)out,
      f);
  return cudaGetLastError();
}

template <int DK, int DV, typename T>
cudaError_t window_dispatch(const Problem& p, const WinInputs& rp, const WinInputs& wn,
                            const float* a_log, int zhead, float* state, void* out, int* err,
                            const Fusion* f, cudaStream_t st) {
  auto part = [zhead](const WinInputs& x) {
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    const bool vec = a16(x.q) && a16(x.k) && a16(x.v) && (zhead || a16(x.z));
    return WinPart<T>{(const T*)x.q, (const T*)x.k, (const T*)x.v, x.z, x.beta, x.W, x.accept,
                      vec};
  };
  const unsigned blocks = (unsigned)p.num_seqs * (unsigned)p.num_heads;
  if (f)
    window_kernel<DK, DV, T, true><<<blocks, kNT, 0, st>>>(part(rp), part(wn), a_log,
                                                           p.num_heads, zhead, state, (T*)out,
                                                           err, *f);
  else
    window_kernel<DK, DV, T><<<blocks, kNT, 0, st>>>(part(rp), part(wn), a_log, p.num_heads,
                                                     zhead, state, (T*)out, err, Fusion{});
  return cudaGetLastError();
}

template <int DK, int DV, typename T>
cudaError_t recurrent_dispatch(const Problem& p, const Args& a, cudaStream_t st) {
  const unsigned blocks = (unsigned)p.num_seqs * (unsigned)p.num_heads;
  recurrent_kernel<DK, DV, T><<<blocks, kNT, 0, st>>>(
      (const T*)a.q, (const T*)a.k, (const T*)a.v, a.z, a.beta, a.initial_state, a.cu_seqlens,
      (T*)a.out, a.final_state, p.num_heads, p.total_tokens, a.err, a.a_log, a.ckpt, a.ckpt_off,
      a.ckpt_every, a.gate_per_head);
  return cudaGetLastError();
}

#define KDA_SIZE_SWITCH(DKV, DVV, ...)                                         \
  [&]() -> cudaError_t {                                                       \
    switch ((DKV) * 1000 + (DVV)) {                                            \
      case 32032: { constexpr int DK = 32, DV = 32; return __VA_ARGS__(); }    \
      case 32064: { constexpr int DK = 32, DV = 64; return __VA_ARGS__(); }    \
      case 32128: { constexpr int DK = 32, DV = 128; return __VA_ARGS__(); }   \
      case 64032: { constexpr int DK = 64, DV = 32; return __VA_ARGS__(); }    \
      case 64064: { constexpr int DK = 64, DV = 64; return __VA_ARGS__(); }    \
      case 64128: { constexpr int DK = 64, DV = 128; return __VA_ARGS__(); }   \
      case 128032: { constexpr int DK = 128, DV = 32; return __VA_ARGS__(); }  \
      case 128064: { constexpr int DK = 128, DV = 64; return __VA_ARGS__(); }  \
      case 128128: { constexpr int DK = 128, DV = 128; return __VA_ARGS__(); } \
      default: return cudaErrorInvalidValue;                                   \
    }                                                                          \
  }()

}  // namespace

cudaError_t launch_decode(const Problem& p, const void* q, const void* k, const void* v,
                          const float* z, const float* beta, const float* a_log, int zhead,
                          float* state, void* out, int* /*err*/, cudaStream_t st) {
  if (p.num_seqs == 0) return cudaSuccess;
  return KDA_SIZE_SWITCH(p.dk, p.dv, [&] {
    return p.io_bf16 ? decode_dispatch<DK, DV, __nv_bfloat16>(p, q, k, v, z, beta, a_log, zhead,
                                                              state, out, st)
                     : decode_dispatch<DK, DV, float>(p, q, k, v, z, beta, a_log, zhead, state,
                                                      out, st);
  });
}

cudaError_t launch_window(const Problem& p, const WinInputs& rp, const WinInputs& wn,
                          const float* a_log, int zhead, float* state, void* out, int* err,
                          cudaStream_t st, const FusionArgs* fa) {
  if (p.num_seqs == 0 || (!rp.accept && wn.W == 0)) return cudaSuccess;
  Fusion f{};
  if (fa) f = Fusion{fa->width, fa->wq, fa->wk, fa->sq, fa->sk, fa->onw, fa->eps};
  const Fusion* fp = fa ? &f : nullptr;
  return KDA_SIZE_SWITCH(p.dk, p.dv, [&] {
    return p.io_bf16 ? window_dispatch<DK, DV, __nv_bfloat16>(p, rp, wn, a_log, zhead, state, out,
                                                              err, fp, st)
                     : window_dispatch<DK, DV, float>(p, rp, wn, a_log, zhead, state, out, err,
                                                      fp, st);
  });
}

cudaError_t launch_decode_fused(const Problem& p, const void* q, const void* k, const void* v,
                                const float* z, const float* beta, const float* a_log, int zhead,
                                float* state, void* out, const FusionArgs& fa, cudaStream_t st) {
  if (p.num_seqs == 0) return cudaSuccess;
  const Fusion f{fa.width, fa.wq, fa.wk, fa.sq, fa.sk, fa.onw, fa.eps};
  return KDA_SIZE_SWITCH(p.dk, p.dv, [&] {
    return p.io_bf16 ? decode_fused_dispatch<DK, DV, __nv_bfloat16>(p, q, k, v, z, beta, a_log,
                                                                    zhead, state, out, f, st)
                     : decode_fused_dispatch<DK, DV, float>(p, q, k, v, z, beta, a_log, zhead,
                                                            state, out, f, st);
  });
}

bool recurrent_small_supported(const Problem& p) { return p.dv == 32 && p.dk <= 64; }

cudaError_t launch_recurrent_small(const Problem& p, const Args& a, cudaStream_t st) {
  if (p.num_seqs == 0) return cudaSuccess;
  if (p.dv != 32) return cudaErrorInvalidValue;
  // few units: a CTA each (the token chain shortened by staging each block
  // first); many: a warp each, four to a CTA
  if ((long long)p.num_seqs * p.num_heads <= kCtaUnitsMax) {
    if (p.dk == 32)
      return p.io_bf16 ? cta_dispatch<32, __nv_bfloat16>(p, a, st) : cta_dispatch<32, float>(p, a, st);
    if (p.dk == 64)
      return p.io_bf16 ? cta_dispatch<64, __nv_bfloat16>(p, a, st) : cta_dispatch<64, float>(p, a, st);
    return cudaErrorInvalidValue;
  }
  if (p.dk == 32)
    return p.io_bf16 ? small_dispatch<32, __nv_bfloat16>(p, a, st) : small_dispatch<32, float>(p, a, st);
  if (p.dk == 64)
    return p.io_bf16 ? small_dispatch<64, __nv_bfloat16>(p, a, st) : small_dispatch<64, float>(p, a, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_recurrent(const Problem& p, const Args& a, cudaStream_t st) {
  if (p.num_seqs == 0) return cudaSuccess;
  return KDA_SIZE_SWITCH(p.dk, p.dv, [&] {
    return p.io_bf16 ? recurrent_dispatch<DK, DV, __nv_bfloat16>(p, a, st)
                     : recurrent_dispatch<DK, DV, float>(p, a, st);
  });
}

}  // namespace kda
