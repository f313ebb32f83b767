// kda_bwd.cu -- reverse mode of the KDA recurrence, token by token, fp32.
//
// Forward (mhpq.cn/news/56770, section "KDA 到底在算什么"; the gate of
// blog.higcp.com "猜想：K3 可能是最适合 TPU 的 MoE 架构", section "下界衰减"),
// per (sequence, head) and token t:
//     q^ = q r_q, k^ = k r_k,  r_x = (sum x^2 + eps)^{-1/2}
//     g = -5 sigmoid(s z) (s = e^{A_h}),  alpha = e^g
//     Sbar = Diag(alpha) S_{t-1},  e = v - Sbar^T k^,  S_t = Sbar + beta k^ e^T,
//     o_t = S_t^T q^.
// The pages print no gradient; this is the chain rule through those lines,
// in reverse token order, with dS the gradient of the loss w.r.t. S_t:
//     dS += q^ do^T;                 dq^ = S_t do
//     y = dS^T k^;  de = beta y;     dbeta = y . e;   dv = de
//     dk^ = beta dS e - Sbar de
//     dSbar = dS - k^ de^T;          dalpha = rowsum(dSbar o S_{t-1})
//     dS <- Diag(alpha) dSbar        (the gradient w.r.t. S_{t-1})
//     dz = dalpha alpha g (1 + g/5) s          (d/du of -5 sigmoid(u) = g (1 + g/5))
//     dq = r_q (dq^ - q^ (q^ . dq^)), the same for dk.
// S_{t-1} and S_t are rebuilt forward from states kept every kSub tokens:
// a first forward pass over the sequence stores them to the workspace, then
// the reverse sweep recomputes each kSub-token sub-block into a ring of
// states (workspace, L2-resident) and walks it backwards.
//
// Thread layout: one CTA of 512 threads per (sequence, head), persistent over
// work items.  Thread (w, l) holds S[c][n] for the 8 key channels
// c = 8 cgp + i (cgp = 4 (w >> 2) + (l >> 3)) and the 4 value channels
// n = 4 ng + j (ng = 8 (w & 3) + (l & 7)).  Sums over c finish across lanes
// l ^ 8, l ^ 16 and the four warps w >> 2; sums over n across lanes l ^ 1,
// l ^ 2, l ^ 4 and the four warps w & 3.  Every state a thread stores to the
// workspace is read back only by that thread.
#include <algorithm>
#include <mutex>
#include <numeric>
#include <vector>

#include "kda_common.cuh"
#include "kda_launch.h"
#include "kda_schedule.h"

namespace kda {
namespace bwd {

constexpr int kD = 128;
constexpr int kNT = 512;
constexpr int kBlk = 64;  // tokens whose inputs are staged in shared memory at once
constexpr int kSub = 8;   // tokens between stored states
constexpr int kMaxOrder = 4096;
constexpr size_t kState = (size_t)kD * kD;  // floats per state

struct Params {
  const void* q;
  const void* k;
  const void* v;
  const float* z;
  const float* beta;
  const float* initial_state;
  const int32_t* cu;
  const void* d_out;
  const float* d_final;
  const float* a_log;
  float* dq;
  float* dk;
  float* dv;
  float* dz;
  float* dbeta;
  float* d_initial;
  float* ws;             // per CTA: ws_states states
  long long ws_states;   // max_len / kSub rounded up, + kSub (the ring)
  int* err;
  int H;
  int total;
  int num_seqs;
  int num_units;
  int use_order;
  int zhead;  // 1: one gate logit per (token, head), z and dz [T, H]
  int order[kMaxOrder];
};

struct Smem {
  float qh[kBlk][kD];   // q^
  float kh[kBlk][kD];   // k^
  float al[kBlk][kD];   // alpha
  float v[kBlk][kD];    // v ; after token t is done: dk^
  float dO[kBlk][kD];   // d out
  float dqh[kBlk][kD];  // dq^
  float e[kSub][kD];    // e of the sub-block being reversed
  float redy[2][4][kD];       // sums over c, per warp row (w >> 2)
  float red3[2][3][4][kD];    // sums over n (dq^ of the token before, dk^, dalpha), per warp column (w & 3)
  float redq[4][kD];          // sums over n: dq^ of a sub-block's last token
  float beta[kBlk], rq[kBlk], rk[kBlk], db[kBlk];
  float dzh[kBlk];  // one gate per head: dz of the block's tokens, summed over channels
};

template <typename T>
struct Vec16;  // 16 consecutive channels of one token
template <>
struct Vec16<float> {
  static __device__ __forceinline__ void ld(const float* p, float (&x)[16]) {
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(p + i));
      x[i] = a.x; x[i + 1] = a.y; x[i + 2] = a.z; x[i + 3] = a.w;
    }
  }
};
template <>
struct Vec16<__nv_bfloat16> {
  static __device__ __forceinline__ void ld(const __nv_bfloat16* p, float (&x)[16]) {
#pragma unroll
    for (int i = 0; i < 16; i += 8) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(p + i));
      const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[i + 2 * j] = __uint_as_float(w[j] << 16);
        x[i + 2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
      }
    }
  }
};

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 x) { *reinterpret_cast<float4*>(p) = x; }

// Stage the inputs of tokens [t0, t0 + len) of head h: eight threads per
// token, 16 channels each.  Rows at or past len are zero.
template <typename T, bool kZHead>
__device__ void stage_block(Smem& sm, const Params& P, int h, int t0, int len, float zc,
                            bool with_q) {
  const int t = threadIdx.x >> 3, part = threadIdx.x & 7, c0 = 16 * part;
  const bool live = t < len;
  const size_t row = ((size_t)(t0 + t) * P.H + h) * kD + c0;
  float x[16], y[16];
  // k^ (and q^)
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    if (pass == 0 && !with_q) continue;
    const T* src = static_cast<const T*>(pass == 0 ? P.q : P.k);
    if (live) Vec16<T>::ld(src + row, x);
    else
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = 0.f;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) ss += x[i] * x[i];
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    ss += __shfl_xor_sync(0xffffffffu, ss, 4);
    const float r = live ? rsqrtf(ss + kNormEps) : 0.f;
    float* dst = pass == 0 ? sm.qh[t] : sm.kh[t];
#pragma unroll
    for (int i = 0; i < 16; i += 4)
      st4(dst + c0 + i, make_float4(x[i] * r, x[i + 1] * r, x[i + 2] * r, x[i + 3] * r));
    if (part == 0) (pass == 0 ? sm.rq : sm.rk)[t] = r;
  }
  // alpha = e^g, g = -5 sigmoid(s z)
  if (live && kZHead) {
    const float zz = __ldg(P.z + (size_t)(t0 + t) * P.H + h);
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i] = zz;
  } else if (live) {
    Vec16<float>::ld(P.z + row, y);
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) y[i] = live ? ex2_approx(log_decay_c(y[i], zc) * 1.4426950408889634f) : 1.f;
#pragma unroll
  for (int i = 0; i < 16; i += 4) st4(sm.al[t] + c0 + i, make_float4(y[i], y[i + 1], y[i + 2], y[i + 3]));
  // v
  if (live) Vec16<T>::ld(static_cast<const T*>(P.v) + row, x);
  else
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = 0.f;
#pragma unroll
  for (int i = 0; i < 16; i += 4) st4(sm.v[t] + c0 + i, make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]));
  if (with_q) {
    if (live) Vec16<T>::ld(static_cast<const T*>(P.d_out) + row, x);
    else
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = 0.f;
#pragma unroll
    for (int i = 0; i < 16; i += 4)
      st4(sm.dO[t] + c0 + i, make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]));
  }
  if (part == 0) {
    sm.beta[t] = live ? __ldg(P.beta + (size_t)(t0 + t) * P.H + h) : 0.f;
    sm.db[t] = 0.f;
  }
}

// This thread's part of a state, S[8 cgp + i][4 ng + j], to / from global.
__device__ __forceinline__ void st_state(float* g, const float (&s)[8][4], int cgp, int ng) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
    st4(g + (size_t)(8 * cgp + i) * kD + 4 * ng, make_float4(s[i][0], s[i][1], s[i][2], s[i][3]));
}
__device__ __forceinline__ void ld_state(const float* g, float (&s)[8][4], int cgp, int ng) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 a = ld4(g + (size_t)(8 * cgp + i) * kD + 4 * ng);
    s[i][0] = a.x; s[i][1] = a.y; s[i][2] = a.z; s[i][3] = a.w;
  }
}

// On x[0 .. M): keep one of two halves by a lane bit and add the partner's
// other half (lane ^ o); the kept sums land in x[0 .. M/2).
template <int M, int N>
__device__ __forceinline__ void fold(float (&x)[N], bool up, int o) {
  static_assert(M <= N && M % 2 == 0, "fold width");
#pragma unroll
  for (int j = 0; j < M / 2; ++j) {
    const float send = up ? x[j] : x[j + M / 2];
    const float keep = up ? x[j + M / 2] : x[j];
    x[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
  }
}

// One forward token: S <- Diag(alpha) S; e = v - S^T k^; S += beta k^ e^T.
// Returns this thread's four e values (n = 4 ng + j).
__device__ __forceinline__ float4 fwd_token(Smem& sm, float (&s)[8][4], int t, int par, int w,
                                            int l, int cgp, int ng) {
  float kc[8], ac[8];
  {
    const float4 k0 = ld4(sm.kh[t] + 8 * cgp), k1 = ld4(sm.kh[t] + 8 * cgp + 4);
    const float4 a0 = ld4(sm.al[t] + 8 * cgp), a1 = ld4(sm.al[t] + 8 * cgp + 4);
    kc[0] = k0.x; kc[1] = k0.y; kc[2] = k0.z; kc[3] = k0.w;
    kc[4] = k1.x; kc[5] = k1.y; kc[6] = k1.z; kc[7] = k1.w;
    ac[0] = a0.x; ac[1] = a0.y; ac[2] = a0.z; ac[3] = a0.w;
    ac[4] = a1.x; ac[5] = a1.y; ac[6] = a1.z; ac[7] = a1.w;
  }
  float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      s[i][j] *= ac[i];
      p[j] = fmaf(s[i][j], kc[i], p[j]);
    }
  fold<4>(p, l & 16, 16);
  fold<2>(p, l & 8, 8);
  sm.redy[par][w >> 2][4 * ng + ((l >> 3) & 3)] = p[0];
  __syncthreads();
  const float4 vv = ld4(sm.v[t] + 4 * ng);
  float4 e = vv;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const float4 x = ld4(sm.redy[par][r] + 4 * ng);
    e.x -= x.x; e.y -= x.y; e.z -= x.z; e.w -= x.w;
  }
  const float b = sm.beta[t];
  const float ev[4] = {b * e.x, b * e.y, b * e.z, b * e.w};
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) s[i][j] = fmaf(kc[i], ev[j], s[i][j]);
  return e;
}

// kZHead: one gate logit per (token, head) (z and dz [T, H]).
template <typename T, bool kZHead>
__global__ void __launch_bounds__(kNT, 1) bwd_kernel(const __grid_constant__ Params P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
  const int cgp = 4 * (w >> 2) + (l >> 3), ng = 8 * (w & 3) + (l & 7);
  float* const ring = P.ws + (size_t)blockIdx.x * P.ws_states * kState;  // kSub states
  float* const subck = ring + kSub * kState;                             // every kSub tokens

  for (int unit = blockIdx.x; unit < P.num_units; unit += gridDim.x) {
    int si = unit / P.H, h = unit % P.H;
    if (P.use_order == 2) {  // the host's schedule: order[unit] = seq * H + head, or -1
      const int pk = P.order[unit];
      if (pk < 0) continue;
      si = pk / P.H;
      h = pk % P.H;
    }
    const int seq = P.use_order == 1 ? P.order[si] : si;
    int bos, eos;
    if (!seq_range(P.cu, seq, P.total, P.err, bos, eos)) continue;
    const int len = eos - bos;
    if ((len + kSub - 1) / kSub + kSub > P.ws_states) {  // workspace planned for shorter sequences
      report_error(P.err, kErrDeviceCheck);
      continue;
    }
    const float zs = gate_scale(P.a_log, h), zc = gate_coef(zs);
    const size_t st_off = ((size_t)seq * P.H + h) * kState;

    // ---- forward: the state entering every kSub-token sub-block ----
    float s[8][4];
    if (P.initial_state) ld_state(P.initial_state + st_off, s, cgp, ng);
    else
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
    int par = 0;
    const int nsub = (len + kSub - 1) / kSub;
    for (int b0 = 0; b0 < len; b0 += kBlk) {
      const int bl = min(kBlk, len - b0);
      __syncthreads();  // the previous block's rows are no longer read
      stage_block<T, kZHead>(sm, P, h, bos + b0, bl, zc, false);
      __syncthreads();
      for (int i = 0; i < bl; ++i) {
        const int t = b0 + i;
        if (t % kSub == 0) {
          st_state(subck + (size_t)(t / kSub) * kState, s, cgp, ng);
          if (t / kSub == nsub - 1) break;  // the last sub-block is rebuilt in the sweep
        }
        fwd_token(sm, s, i, par, w, l, cgp, ng);
        par ^= 1;
      }
    }

    // ---- reverse sweep ----
    float ds[8][4];
    if (P.d_final) ld_state(P.d_final + st_off, ds, cgp, ng);
    else
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) ds[i][j] = 0.f;
    const int nblk = (len + kBlk - 1) / kBlk;
    for (int bi = nblk - 1; bi >= 0; --bi) {
      const int b0 = bi * kBlk, bl = min(kBlk, len - b0);
      __syncthreads();
      stage_block<T, kZHead>(sm, P, h, bos + b0, bl, zc, true);
      if (kZHead && tid < kBlk) sm.dzh[tid] = 0.f;
      __syncthreads();
      for (int j0 = ((bl - 1) / kSub) * kSub; j0 >= 0; j0 -= kSub) {
        const int sl = min(kSub, bl - j0);
        const float* const sub_in = subck + (size_t)((b0 + j0) / kSub) * kState;
        // rebuild S_t for the sub-block's tokens, and their e.  The ring keeps
        // S_t for all but the last token: the reverse step of token t reads only
        // S_{t-1}, and takes dq^ of token t - 1 (= S_{t-1} do_{t-1}) from it too.
        ld_state(sub_in, s, cgp, ng);
        for (int i = 0; i < sl; ++i) {
          const float4 e = fwd_token(sm, s, j0 + i, par, w, l, cgp, ng);
          par ^= 1;
          if (w < 4 && l < 8) st4(sm.e[i] + 4 * ng, e);  // cgp == 0: one writer per n
          if (i + 1 < sl) st_state(ring + (size_t)i * kState, s, cgp, ng);
        }
        {  // dq^ of the sub-block's last token from the state after it, still in s
          const float4 d4 = ld4(sm.dO[j0 + sl - 1] + 4 * ng);
          float p1[8];
#pragma unroll
          for (int r = 0; r < 8; ++r)
            p1[r] = s[r][0] * d4.x + s[r][1] * d4.y + s[r][2] * d4.z + s[r][3] * d4.w;
          fold<8>(p1, l & 4, 4);
          fold<4>(p1, l & 2, 2);
          fold<2>(p1, l & 1, 1);
          sm.redq[w & 3][8 * cgp + (l & 7)] = p1[0];
        }
        __syncthreads();  // e rows and the last token's dq^ parts visible
        if (tid < kD)
          sm.dqh[j0 + sl - 1][tid] =
              sm.redq[0][tid] + sm.redq[1][tid] + sm.redq[2][tid] + sm.redq[3][tid];
        for (int i = sl - 1; i >= 0; --i) {
          const int t = j0 + i;
          const float* const st_p = i > 0 ? ring + (size_t)(i - 1) * kState : sub_in;
          // (a) dS += q^ do^T; y = dS^T k^
          const float4 d4 = ld4(sm.dO[t] + 4 * ng);
          const float dov[4] = {d4.x, d4.y, d4.z, d4.w};
          const float* const qrow = sm.qh[t] + 8 * cgp;
          const float* const krow = sm.kh[t] + 8 * cgp;
          const float* const arow = sm.al[t] + 8 * cgp;
          float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const float qc = qrow[r], kc = krow[r];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              ds[r][j] = fmaf(qc, dov[j], ds[r][j]);
              y[j] = fmaf(ds[r][j], kc, y[j]);
            }
          }
          fold<4>(y, l & 16, 16);
          fold<2>(y, l & 8, 8);
          sm.redy[par][w >> 2][4 * ng + ((l >> 3) & 3)] = y[0];
          __syncthreads();
          // (b) de = beta y; dv; dbeta; dk^ = beta dS e - Sbar de; dSbar; dalpha;
          //     dS <- Diag(alpha) dSbar; dq^ of token t - 1 = S_{t-1} do_{t-1}
          float4 yy = ld4(sm.redy[par][0] + 4 * ng);
#pragma unroll
          for (int r = 1; r < 4; ++r) {
            const float4 x = ld4(sm.redy[par][r] + 4 * ng);
            yy.x += x.x; yy.y += x.y; yy.z += x.z; yy.w += x.w;
          }
          const float bt = sm.beta[t];
          const float4 e4 = ld4(sm.e[i] + 4 * ng);
          const float ev[4] = {e4.x, e4.y, e4.z, e4.w};
          const float de[4] = {bt * yy.x, bt * yy.y, bt * yy.z, bt * yy.w};
          if (w < 4 && l < 8) {  // cgp == 0: one writer per n
            st4(P.dv + ((size_t)(bos + b0 + t) * P.H + h) * kD + 4 * ng,
                make_float4(de[0], de[1], de[2], de[3]));
            float yb = yy.x * ev[0] + yy.y * ev[1] + yy.z * ev[2] + yy.w * ev[3];
            yb += __shfl_xor_sync(0x000000ffu, yb, 1);
            yb += __shfl_xor_sync(0x000000ffu, yb, 2);
            yb += __shfl_xor_sync(0x000000ffu, yb, 4);
            if (l == 0) atomicAdd(&sm.db[t], yb);
          }
          const float4 dp4 = ld4(sm.dO[t > 0 ? t - 1 : 0] + 4 * ng);
          const float dop[4] = {dp4.x, dp4.y, dp4.z, dp4.w};
          float p1[8], p2[8], p3[8];
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const float4 a = ld4(st_p + (size_t)(8 * cgp + r) * kD + 4 * ng);
            const float sp[4] = {a.x, a.y, a.z, a.w};
            const float ac = arow[r], kc = krow[r];
            float x2 = 0.f, x3 = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float sbar = ac * sp[j];
              x2 = fmaf(bt * ds[r][j], ev[j], x2);
              x2 = fmaf(-sbar, de[j], x2);
              const float dsb = fmaf(-kc, de[j], ds[r][j]);
              x3 = fmaf(dsb, sp[j], x3);
              ds[r][j] = ac * dsb;
            }
            p1[r] = sp[0] * dop[0] + sp[1] * dop[1] + sp[2] * dop[2] + sp[3] * dop[3];
            p2[r] = x2;
            p3[r] = x3;
          }
          fold<8>(p1, l & 4, 4);
          fold<4>(p1, l & 2, 2);
          fold<2>(p1, l & 1, 1);
          fold<8>(p2, l & 4, 4);
          fold<4>(p2, l & 2, 2);
          fold<2>(p2, l & 1, 1);
          fold<8>(p3, l & 4, 4);
          fold<4>(p3, l & 2, 2);
          fold<2>(p3, l & 1, 1);
          sm.red3[par][0][w & 3][8 * cgp + (l & 7)] = p1[0];
          sm.red3[par][1][w & 3][8 * cgp + (l & 7)] = p2[0];
          sm.red3[par][2][w & 3][8 * cgp + (l & 7)] = p3[0];
          __syncthreads();
          // (c) per key channel: dq^ of token t - 1 and dk^ kept for the block's norm
          //     pass (a sub-block's first token gets its dq^ from the sub-block before
          //     it, whose last token it is); dz out
          if (tid < kD) {
            const int c = tid;
            float dqh = 0.f, dkh = 0.f, dal = 0.f;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              dqh += sm.red3[par][0][r][c];
              dkh += sm.red3[par][1][r][c];
              dal += sm.red3[par][2][r][c];
            }
            if (i > 0) sm.dqh[t - 1][c] = dqh;
            sm.v[t][c] = dkh;  // this token's v is no longer read
            const float a = sm.al[t][c], g = __logf(a);
            const float dzc = dal * a * g * (1.f + g / 5.f) * zs;
            if (kZHead) {  // the head's one logit feeds every channel: sum the terms
              const float sum = warp_sum(dzc);
              if ((tid & 31) == 0) atomicAdd(&sm.dzh[t], sum);
            } else {
              P.dz[((size_t)(bos + b0 + t) * P.H + h) * kD + c] = dzc;
            }
          }
          par ^= 1;
        }
      }
      __syncthreads();
      // ---- the block's norm pass: dq = r_q (dq^ - q^ (q^ . dq^)), the same for k ----
      // Every lane takes part in the shuffles (rows past bl are zero in shared
      // memory); only live rows are stored.
      {
        const int t = tid >> 3, part = tid & 7, c0 = 16 * part;
        const bool live = t < bl;
        {
          const size_t row = ((size_t)(bos + b0 + t) * P.H + h) * kD + c0;
#pragma unroll
          for (int pass = 0; pass < 2; ++pass) {
            const float* xh = pass == 0 ? sm.qh[t] : sm.kh[t];
            const float* dxh = pass == 0 ? sm.dqh[t] : sm.v[t];
            float dot = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) dot = fmaf(xh[c0 + i], dxh[c0 + i], dot);
            dot += __shfl_xor_sync(0xffffffffu, dot, 1);
            dot += __shfl_xor_sync(0xffffffffu, dot, 2);
            dot += __shfl_xor_sync(0xffffffffu, dot, 4);
            const float r = pass == 0 ? sm.rq[t] : sm.rk[t];
            float* out = pass == 0 ? P.dq : P.dk;
            if (live)
#pragma unroll
            for (int i = 0; i < 16; i += 4)
              st4(out + row + i,
                  make_float4(r * (dxh[c0 + i] - xh[c0 + i] * dot),
                              r * (dxh[c0 + i + 1] - xh[c0 + i + 1] * dot),
                              r * (dxh[c0 + i + 2] - xh[c0 + i + 2] * dot),
                              r * (dxh[c0 + i + 3] - xh[c0 + i + 3] * dot)));
          }
          if (live && part == 0) {
            P.dbeta[(size_t)(bos + b0 + t) * P.H + h] = sm.db[t];
            if (kZHead) P.dz[(size_t)(bos + b0 + t) * P.H + h] = sm.dzh[t];
          }
        }
      }
    }
    if (P.d_initial) st_state(P.d_initial + st_off, ds, cgp, ng);
  }
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

int grid_for(const Problem& p) {
  const int sms = sm_count();
  return std::max(1, std::min(p.num_seqs * p.num_heads, sms));
}

long long states_per_cta(const Problem& p, const int32_t* cu_host) {
  int max_len = 0;
  for (int n = 0; n < p.num_seqs; ++n) max_len = std::max(max_len, cu_host[n + 1] - cu_host[n]);
  return (long long)(max_len + kSub - 1) / kSub + kSub;
}

}  // namespace bwd

namespace bwd {

// ---- dk or dv below 128: zero-padded to 128 channels around the kernel ----
//
// A key channel whose q, k are zero keeps a zero state row (its k never
// reaches the rank-one updates, and its decay acts on zeros); a value channel
// whose v is zero keeps a zero state column; zeros change no L2 norm.  So the
// 128 x 128 reverse mode over zero-padded inputs gives exactly the gradients of
// the real channels (those of the padded ones are zero and dropped).

template <typename T>
__global__ void pad_rows_kernel(T* __restrict__ dst, const T* __restrict__ src, long long rows,
                                int d) {
  const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (i >= rows * kD) return;
  const long long r = i / kD;
  const int c = (int)(i % kD);
  dst[i] = c < d ? src[r * d + c] : T(0.f);
}

__global__ void unpad_rows_kernel(float* __restrict__ dst, const float* __restrict__ src,
                                  long long rows, int d) {
  const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (i >= rows * d) return;
  dst[i] = src[(i / d) * kD + i % d];
}

// [NH][dk][dv] <-> [NH][128][128]
__global__ void pad_state_kernel(float* __restrict__ dst, const float* __restrict__ src,
                                 long long nh, int dk, int dv) {
  const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (i >= nh * kD * kD) return;
  const long long u = i / (kD * kD);
  const int c = (int)((i / kD) % kD), n = (int)(i % kD);
  dst[i] = (c < dk && n < dv) ? src[(u * dk + c) * dv + n] : 0.f;
}

__global__ void unpad_state_kernel(float* __restrict__ dst, const float* __restrict__ src,
                                   long long nh, int dk, int dv) {
  const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (i >= nh * dk * dv) return;
  const long long u = i / ((long long)dk * dv);
  const int c = (int)((i / dv) % dk), n = (int)(i % dv);
  dst[i] = src[(u * kD + c) * kD + n];
}

inline unsigned blocks_for(long long n) { return (unsigned)((n + 255) / 256); }

// Device layout of the padded inputs and outputs inside the workspace, ahead
// of the 128 x 128 kernel's own workspace.
struct PadLayout {
  size_t q, k, v, dout, z, s0, dfin, dq, dk, dv, dz, dini, inner, total;
};
inline size_t up256(size_t x) { return (x + 255) / 256 * 256; }
PadLayout pad_layout(const Problem& p) {
  const size_t th = (size_t)p.total_tokens * p.num_heads, es = p.io_bf16 ? 2 : 4;
  const size_t st = (size_t)p.num_seqs * p.num_heads * kD * kD * 4;
  PadLayout L;
  size_t o = 0;
  L.q = o; o += up256(th * kD * es);
  L.k = o; o += up256(th * kD * es);
  L.v = o; o += up256(th * kD * es);
  L.dout = o; o += up256(th * kD * es);
  L.z = o; o += up256(th * kD * 4);
  L.s0 = o; o += up256(st);
  L.dfin = o; o += up256(st);
  L.dq = o; o += up256(th * kD * 4);
  L.dk = o; o += up256(th * kD * 4);
  L.dv = o; o += up256(th * kD * 4);
  L.dz = o; o += up256(th * kD * 4);
  L.dini = o; o += up256(st);
  L.inner = o;
  L.total = o;
  return L;
}

}  // namespace bwd

static size_t bwd_inner_bytes(const Problem& p, const int32_t* cu_host) {
  if (p.num_seqs == 0 || p.num_heads == 0) return 0;
  return (size_t)bwd::grid_for(p) * (size_t)bwd::states_per_cta(p, cu_host) * bwd::kState *
         sizeof(float);
}

size_t recurrent_bwd_workspace_bytes(const Problem& p, const int32_t* cu_host) {
  if (p.num_seqs == 0 || p.num_heads == 0) return 0;
  if (p.dk == bwd::kD && p.dv == bwd::kD) return bwd_inner_bytes(p, cu_host);
  return bwd::pad_layout(p).total + bwd_inner_bytes(p, cu_host);
}

size_t chunk_bwd_workspace_bytes(const Problem& p, const int32_t* cu_host) {
  if (p.num_seqs == 0 || p.num_heads == 0) return 0;
  if (p.dk == bwd::kD && p.dv == bwd::kD) return chunk_bwd_inner_bytes(p, cu_host);
  return bwd::pad_layout(p).total + chunk_bwd_inner_bytes(p, cu_host);
}

static cudaError_t launch_bwd_128(const Problem& p, const BwdArgs& a, const int32_t* cu_host,
                                  void* ws, cudaStream_t st);

using Bwd128 = cudaError_t (*)(const Problem&, const BwdArgs&, const int32_t*, void*,
                               cudaStream_t);

// Either reverse mode (token by token or chunked) over inputs zero-padded to
// dk = dv = 128 when they are narrower.
static cudaError_t launch_bwd_padded(const Problem& p, const BwdArgs& a, const int32_t* cu_host,
                                     void* ws, cudaStream_t st, Bwd128 launch_128) {
  using namespace bwd;
  if (p.num_seqs == 0) return cudaSuccess;
  if (p.dk == kD && p.dv == kD) return launch_128(p, a, cu_host, ws, st);
  const PadLayout L = pad_layout(p);
  unsigned char* W = static_cast<unsigned char*>(ws);
  const long long th = (long long)p.total_tokens * p.num_heads;
  const long long nh = (long long)p.num_seqs * p.num_heads;
  Problem p128 = p;
  p128.dk = p128.dv = kD;
  BwdArgs b = a;
  auto pad = [&](size_t off, const void* src, int d) {
    if (p.io_bf16)
      pad_rows_kernel<__nv_bfloat16><<<blocks_for(th * kD), 256, 0, st>>>(
          reinterpret_cast<__nv_bfloat16*>(W + off), static_cast<const __nv_bfloat16*>(src), th, d);
    else
      pad_rows_kernel<float><<<blocks_for(th * kD), 256, 0, st>>>(
          reinterpret_cast<float*>(W + off), static_cast<const float*>(src), th, d);
    return reinterpret_cast<const void*>(W + off);
  };
  if (th > 0) {
    b.q = pad(L.q, a.q, p.dk);
    b.k = pad(L.k, a.k, p.dk);
    b.v = pad(L.v, a.v, p.dv);
    b.d_out = pad(L.dout, a.d_out, p.dv);
    if (!a.zhead) {
      pad_rows_kernel<float><<<blocks_for(th * kD), 256, 0, st>>>(
          reinterpret_cast<float*>(W + L.z), a.z, th, p.dk);
      b.z = reinterpret_cast<const float*>(W + L.z);
    }
  }
  auto pad_state = [&](size_t off, const float* src) -> const float* {
    if (!src) return nullptr;
    pad_state_kernel<<<blocks_for(nh * kD * kD), 256, 0, st>>>(
        reinterpret_cast<float*>(W + off), src, nh, p.dk, p.dv);
    return reinterpret_cast<const float*>(W + off);
  };
  b.initial_state = pad_state(L.s0, a.initial_state);
  b.d_final = pad_state(L.dfin, a.d_final);
  b.dq = reinterpret_cast<float*>(W + L.dq);
  b.dk = reinterpret_cast<float*>(W + L.dk);
  b.dv = reinterpret_cast<float*>(W + L.dv);
  if (!a.zhead) b.dz = reinterpret_cast<float*>(W + L.dz);  // one gate per head: [T, H] as is
  b.d_initial = a.d_initial ? reinterpret_cast<float*>(W + L.dini) : nullptr;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_128(p128, b, cu_host, W + L.inner, st);
  if (e != cudaSuccess) return e;
  if (th > 0) {
    unpad_rows_kernel<<<blocks_for(th * p.dk), 256, 0, st>>>(a.dq, b.dq, th, p.dk);
    unpad_rows_kernel<<<blocks_for(th * p.dk), 256, 0, st>>>(a.dk, b.dk, th, p.dk);
    unpad_rows_kernel<<<blocks_for(th * p.dv), 256, 0, st>>>(a.dv, b.dv, th, p.dv);
    if (!a.zhead) unpad_rows_kernel<<<blocks_for(th * p.dk), 256, 0, st>>>(a.dz, b.dz, th, p.dk);
  }
  if (a.d_initial)
    unpad_state_kernel<<<blocks_for(nh * p.dk * p.dv), 256, 0, st>>>(a.d_initial, b.d_initial,
                                                                    nh, p.dk, p.dv);
  return cudaGetLastError();
}

cudaError_t launch_recurrent_bwd(const Problem& p, const BwdArgs& a, const int32_t* cu_host,
                                 void* ws, cudaStream_t st) {
  return launch_bwd_padded(p, a, cu_host, ws, st, launch_bwd_128);
}

cudaError_t launch_chunk_bwd(const Problem& p, const BwdArgs& a, const int32_t* cu_host, void* ws,
                             cudaStream_t st) {
  return launch_bwd_padded(p, a, cu_host, ws, st, launch_chunk_bwd_128);
}

static cudaError_t launch_bwd_128(const Problem& p, const BwdArgs& a, const int32_t* cu_host,
                                  void* ws, cudaStream_t st) {
  using namespace bwd;
  if (p.num_seqs == 0) return cudaSuccess;
  static PerDeviceInit attrs;
  const cudaError_t attr = attrs.run([] {
    cudaError_t e = cudaSuccess;
    const void* kernels[] = {(const void*)bwd_kernel<float, false>,
                             (const void*)bwd_kernel<__nv_bfloat16, false>,
                             (const void*)bwd_kernel<float, true>,
                             (const void*)bwd_kernel<__nv_bfloat16, true>};
    for (const void* kf : kernels)
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(Smem));
    return e;
  });
  if (attr != cudaSuccess) return attr;
  static thread_local Params prm;  // large: keep off the stack
  prm.q = a.q;
  prm.k = a.k;
  prm.v = a.v;
  prm.z = a.z;
  prm.beta = a.beta;
  prm.initial_state = a.initial_state;
  prm.cu = a.cu_seqlens;
  prm.d_out = a.d_out;
  prm.d_final = a.d_final;
  prm.a_log = a.a_log;
  prm.dq = a.dq;
  prm.dk = a.dk;
  prm.dv = a.dv;
  prm.dz = a.dz;
  prm.dbeta = a.dbeta;
  prm.d_initial = a.d_initial;
  prm.ws = static_cast<float*>(ws);
  prm.ws_states = states_per_cta(p, cu_host);
  prm.err = a.err;
  prm.H = p.num_heads;
  prm.total = p.total_tokens;
  prm.num_seqs = p.num_seqs;
  prm.num_units = p.num_seqs * p.num_heads;
  prm.zhead = a.zhead;
  prm.use_order = 0;
  const int grid = grid_for(p);
  if (p.num_seqs <= kMaxOrder) {  // longest sequences first, each unit to the least-loaded CTA
    std::vector<int> idx(p.num_seqs);
    std::iota(idx.begin(), idx.end(), 0);
    std::stable_sort(idx.begin(), idx.end(), [&](int x, int y) {
      return cu_host[x + 1] - cu_host[x] > cu_host[y + 1] - cu_host[y];
    });
    auto tokens = [&](int sq) { return (long long)(cu_host[sq + 1] - cu_host[sq]); };
    const int n = build_unit_schedule(idx, p.num_heads, grid, tokens, prm.order, kMaxOrder);
    if (n > 0) {
      prm.num_units = n;
      prm.use_order = 2;
    } else {
      for (int i = 0; i < p.num_seqs; ++i) prm.order[i] = idx[i];
      prm.use_order = 1;
    }
  }
  if (p.io_bf16)
    prm.zhead ? bwd_kernel<__nv_bfloat16, true><<<grid, kNT, sizeof(Smem), st>>>(prm)
              : bwd_kernel<__nv_bfloat16, false><<<grid, kNT, sizeof(Smem), st>>>(prm);
  else
    prm.zhead ? bwd_kernel<float, true><<<grid, kNT, sizeof(Smem), st>>>(prm)
              : bwd_kernel<float, false><<<grid, kNT, sizeof(Smem), st>>>(prm);
  return cudaGetLastError();
}

}  // namespace kda
