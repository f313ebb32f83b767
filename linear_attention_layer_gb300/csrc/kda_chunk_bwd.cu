// kda_chunk_bwd.cu -- reverse mode of the KDA recurrence in the chunked (WY /
// UT) form, with the chunk products on the tensor cores.
//
// Forward of one chunk of C = 16 tokens (mhpq.cn/news/56770, section "KDA 到底
// 在算什么", evaluated chunkwise; the gate of blog.higcp.com "猜想：K3 可能是最适合
// TPU 的 MoE 架构", section "下界衰减"), with G the inclusive cumulative
// log-decay per channel inside the chunk and S the entering state [dk, dv]:
//     Q+ = q^ e^{G},  K+ = k^ e^{G},  K- = k^ e^{-G},  K~ = k^ e^{G_C - G}
//     A = diag(beta) strict_lower(K+ K-^T),  P = lower(Q+ K-^T)
//     T = (I + A)^{-1},  T' = T diag(beta),  R = V - K+ S,  U = T' R
//     O = Q+ S + P U,  S' = Diag(e^{G_C}) S + K~^T U.
// The pages print no gradient; the reverse mode is the chain rule through
// those lines, given dO and dS' (the gradient w.r.t. the leaving state):
//     dU = P^T dO + K~ dS',  dR = T'^T dU,  dV = dR
//     dQ+ = dO S^T + dP K-,  dK+ = -dR S^T + dAr K-,  dK~ = U dS'^T
//     dK- = dAr^T K+ + dP^T Q+,  dP = lower(dO U^T),  dT' = dU R^T
//     dbeta_j = sum_t T_tj dT'_tj + sum_s A_js dA_js / beta_j
//     dA = strict_lower(-T^T dT T^T) with dT = dT' diag(beta),  dAr = diag(beta) dA
//     dS = Diag(e^{G_C}) dS' + Q+^T dO - K+^T dR
// and through the exponentials of G: dq^ = dQ+ e^{G}, dk^ = dK+ e^{G} +
// (dK- + dK~ e^{G_C}) e^{-G}, while the gradient of the log-decay g_r (G the
// cumulative sum of g) is, per channel, summed so that no term cancels
// against another (a plain dG followed by its reverse cumulative sum loses
// every digit the two share):
//     dg_r = rowsum(S o dS') e^{G_C} + sum_{t >= r} (dO S^T o Q+ - dR S^T o K+)_t
//            + sum_{t < r} (dK~ o K~)_t
//            + sum_{t >= r > s} (dP_ts Q+_t + dAr_ts K+_t) K-_s.
// Then the gate (dz = dg g (1 + g/5) e^{A}) and the L2 norms
// (dq = r (dq^ - q^ (q^ . dq^))).  16-token chunks keep every factor
// e^{+-G} inside [e^{-80}, e^{80}] (the gate's lower bound), so no product
// leaves the fp32 range.
//
// Products: bf16 warp MMAs (m16n8k16, fp32 accumulation) on operands split
// into a high and a low bf16 part (x = hi + lo to 2^-17), three MMAs per
// product (hi hi + hi lo + lo hi): 16 significant bits per operand, with the
// fp32 range.  Every operand sits in shared memory as two bf16 planes whose
// 16-byte row chunks are permuted by row, so each fragment, plain or
// transposed, is one ldmatrix without bank conflicts.
//
// Schedule: one CTA of 16 warps per (sequence, head), persistent over units
// longest first.  S and dS stay fp32 in registers (each warp a 32 x 32 block),
// with bf16 hi / lo copies in shared memory as MMA operands.  A forward sweep
// writes the state entering every chunk to the workspace (as its hi / lo
// planes, the only form the reverse step reads), with the chunk's R, U, A and
// T; the reverse sweep walks the chunks backwards, copying each chunk's planes
// and record straight into shared memory (cp.async) and recomputing only what
// involves q and dO; each chunk's inputs, state and record are prefetched
// toward L2 one chunk ahead.
#include <algorithm>
#include <numeric>
#include <vector>

#include "kda_common.cuh"
#include "kda_launch.h"
#include "kda_schedule.h"
#include "tc_ptx.cuh"

namespace kda {
namespace cbwd {

using tc::ldmatrix_x4;
using tc::ldmatrix_x4_trans;
using tc::mma_16816;
using tc::pack_bf16;
using tc::smem_u32;

constexpr int kD = 128;    // key and value channels
constexpr int kC = 16;     // tokens per chunk
constexpr int kNT = 512;
constexpr int kMaxOrder = 4096;
constexpr size_t kState = (size_t)kD * kD;
constexpr float kLog2e = 1.4426950408889634f;

// ---- shared memory (bytes) ----
constexpr int kPlaneS = kD * kD * 2;  // a 128 x 128 bf16 plane
constexpr int kPlane = kC * kD * 2;   // a 16 x 128 bf16 plane
constexpr int kPlane16 = kC * kC * 2; // a 16 x 16 bf16 plane
constexpr int kF32 = kC * kD * 4;     // a 16 x 128 fp32 array
// each operand: its hi plane, then its lo plane
constexpr int OFF_S = 0;
constexpr int OFF_DS = OFF_S + 2 * kPlaneS;
constexpr int OFF_KP = OFF_DS + 2 * kPlaneS;  // K+
constexpr int OFF_KM = OFF_KP + 2 * kPlane;   // K-
constexpr int OFF_KT = OFF_KM + 2 * kPlane;   // K~
constexpr int OFF_QP = OFF_KT + 2 * kPlane;   // Q+
constexpr int OFF_R = OFF_QP + 2 * kPlane;    // R = V - K+ S
constexpr int OFF_U = OFF_R + 2 * kPlane;
constexpr int OFF_DO = OFF_U + 2 * kPlane;
constexpr int OFF_DU = OFF_DO + 2 * kPlane;
constexpr int OFF_DR = OFF_DU + 2 * kPlane;
constexpr int OFF_QH = OFF_DR + 2 * kPlane;   // q^ fp32
constexpr int OFF_EG = OFF_QH + kF32;         // e^{G} fp32
constexpr int OFF_ARAW = OFF_EG + kF32;       // fp32 16 x 16: strict_lower(K+ K-^T)
constexpr int OFF_T = OFF_ARAW + 1024;        // fp32 16 x 16: (I + A)^{-1}
constexpr int OFF_DTP = OFF_T + 1024;         // fp32 16 x 16: dT'
constexpr int OFF_DPF = OFF_DTP + 1024;       // fp32 16 x 16: dP
constexpr int OFF_TP = OFF_DPF + 1024;        // T' planes
constexpr int OFF_P = OFF_TP + 2 * kPlane16;  // P planes
constexpr int OFF_DP = OFF_P + 2 * kPlane16;  // dP planes
constexpr int OFF_DAR = OFF_DP + 2 * kPlane16;  // dAr planes
constexpr int OFF_EC = OFF_DAR + 2 * kPlane16;  // e^{G_C} [128]
constexpr int OFF_DEC = OFF_EC + 512;           // rowsum(S o dS') [128]
constexpr int OFF_VEC = OFF_DEC + 512;          // beta, rq, rk, db, dzh [16] each
constexpr int SMEM_BYTES = OFF_VEC + 5 * 64;
static_assert(SMEM_BYTES <= 232448, "shared memory");
// What the forward sweep keeps of each chunk besides its state, copied verbatim
// from / to shared memory: the R and U planes, A and T (fp32), the T' planes.
constexpr int kKeptRU = 4 * kPlane;          // R hi, lo, U hi, lo
constexpr int kKeptAT = 2048;                // A, T fp32
constexpr int kKeptTP = 2 * kPlane16;        // T' hi, lo
constexpr int kKeptBytes = kKeptRU + kKeptAT + kKeptTP;
constexpr int kKeptStride = 20480;
static_assert(OFF_U == OFF_R + 2 * kPlane && OFF_T == OFF_ARAW + 1024, "kept regions");
static_assert(kKeptBytes <= kKeptStride && kKeptBytes % (16 * 4) == 0, "kept layout");
// fp32 scratch laid over operands that are dead at the time:
//   staging: g (log2 units) on U, k^ on dR, v on dU, the scan's partial sums on R
//   reverse: the dg state terms on dU and dR, T^T dT and dAr (fp32) on R,
//            the norms' partial dots on U, dz on dO, dot totals on K~

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
  float* ws;            // per CTA: ws_states state plane images (64 KiB), one per chunk
                        // of the longest sequence, then as many kept records
  long long ws_states;
  int* err;
  int H;
  int total;
  int num_seqs;
  int num_units;
  int use_order;
  int order[kMaxOrder];
};

// Byte offset of element (r, c) in a 128-wide bf16 plane: 256-byte rows whose
// 16-byte chunks are permuted by c / 8 -> c / 8 ^ (r % 8).
__device__ __forceinline__ uint32_t boff(int r, int c) {
  return (uint32_t)((r << 8) + ((((c >> 3) ^ (r & 7)) << 4) | ((c & 7) << 1)));
}
// ... and in a 16-wide plane: 32-byte rows, chunk c / 8 -> c / 8 ^ (r / 4 % 2).
__device__ __forceinline__ uint32_t boff16(int r, int c) {
  return (uint32_t)((r << 5) + ((((c >> 3) ^ ((r >> 2) & 1)) << 4) | ((c & 7) << 1)));
}
template <bool kWide>
__device__ __forceinline__ uint32_t poff(int r, int c) {
  return kWide ? boff(r, c) : boff16(r, c);
}
// fp32 [rows][128]: element (r, c) at r * 128 + (c ^ (8 (r % 4) + (r & 4))).
__device__ __forceinline__ int swz(int r, int c) {
  return (r << 7) + (c ^ (((r & 3) << 3) | (r & 4)));
}

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 x) { *reinterpret_cast<float4*>(p) = x; }
__device__ __forceinline__ float2 ld2(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ void st2(float* p, float2 x) { *reinterpret_cast<float2*>(p) = x; }

template <typename T>
__device__ __forceinline__ float4 ld4_io(const T* p);
template <>
__device__ __forceinline__ float4 ld4_io<float>(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}
template <>
__device__ __forceinline__ float4 ld4_io<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 a = __ldg(reinterpret_cast<const uint2*>(p));
  return make_float4(__uint_as_float(a.x << 16), __uint_as_float(a.x & 0xffff0000u),
                     __uint_as_float(a.y << 16), __uint_as_float(a.y & 0xffff0000u));
}

// x0, x1 (columns c, c + 1) as bf16 hi and lo pairs at byte offset o of the hi
// and lo planes.
__device__ __forceinline__ void st_split(unsigned char* hi, unsigned char* lo, uint32_t o,
                                         float x0, float x1) {
  const uint32_t h = pack_bf16(x0, x1);
  const uint32_t l =
      pack_bf16(x0 - __uint_as_float(h << 16), x1 - __uint_as_float(h & 0xffff0000u));
  *reinterpret_cast<uint32_t*>(hi + o) = h;
  *reinterpret_cast<uint32_t*>(lo + o) = l;
}
// one element as bf16 hi / lo
__device__ __forceinline__ void st_split1(unsigned char* hi, unsigned char* lo, uint32_t o,
                                          float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  *reinterpret_cast<__nv_bfloat16*>(hi + o) = h;
  *reinterpret_cast<__nv_bfloat16*>(lo + o) = __float2bfloat16_rn(x - __bfloat162float(h));
}
// hi + lo of the pair at byte offset o
__device__ __forceinline__ float2 ld_split(const unsigned char* hi, const unsigned char* lo,
                                           uint32_t o) {
  const uint32_t h = *reinterpret_cast<const uint32_t*>(hi + o);
  const uint32_t l = *reinterpret_cast<const uint32_t*>(lo + o);
  return make_float2(__uint_as_float(h << 16) + __uint_as_float(l << 16),
                     __uint_as_float(h & 0xffff0000u) + __uint_as_float(l & 0xffff0000u));
}

// ---- MMA fragments (m16n8k16 bf16: a = rows g, g + 8 x column pairs 2q, 2q + 8;
// b = row pairs 2q, 2q + 8 x column g; c = rows g, g + 8 x columns 2q, 2q + 1) ----
// A (16 x 16) at rows m0.., columns k0.. of a [m][k] plane at shared address `base`
template <bool kWide>
__device__ __forceinline__ void lda(uint32_t base, int m0, int k0, uint32_t (&a)[4]) {
  const int l = threadIdx.x & 31, j = l >> 3, i = l & 7;
  ldmatrix_x4(base + poff<kWide>(m0 + ((j & 1) << 3) + i, k0 + ((j >> 1) << 3)), a[0], a[1], a[2],
              a[3]);
}
// A (16 x 16) with A[m][k] = X[k0 + k][m0 + m] (X a [k][m] plane)
template <bool kWide>
__device__ __forceinline__ void lda_t(uint32_t base, int m0, int k0, uint32_t (&a)[4]) {
  const int l = threadIdx.x & 31, j = l >> 3, i = l & 7;
  ldmatrix_x4_trans(base + poff<kWide>(k0 + ((j >> 1) << 3) + i, m0 + ((j & 1) << 3)), a[0], a[1],
                    a[2], a[3]);
}
// B of one n-tile (columns n0..n0+7) for k-steps k0 and k0 + 16, with
// B[k][n] = X[n][k] (X a [n][k] plane): b[0], b[1] for k0; b[2], b[3] for k0 + 16
__device__ __forceinline__ void ldb_nk2(uint32_t base, int k0, int n0, uint32_t (&b)[4]) {
  const int l = threadIdx.x & 31, j = l >> 3, i = l & 7;
  ldmatrix_x4(base + boff(n0 + i, k0 + (j << 3)), b[0], b[1], b[2], b[3]);
}
// ... with B[k][n] = X[k][n] (X a [k][n] plane)
__device__ __forceinline__ void ldb_kn2(uint32_t base, int k0, int n0, uint32_t (&b)[4]) {
  const int l = threadIdx.x & 31, j = l >> 3, i = l & 7;
  ldmatrix_x4_trans(base + boff(k0 + (j << 3) + i, n0), b[0], b[1], b[2], b[3]);
}
// B of one n-tile for the single k-step of a 16-token contraction, hi and lo
// together: b[0], b[1] hi; b[2], b[3] lo.  [k][n] planes (k = token):
__device__ __forceinline__ void ldb_kn_hl(uint32_t hi, uint32_t lo, int n0, uint32_t (&b)[4]) {
  const int l = threadIdx.x & 31, j = l >> 3, i = l & 7;
  ldmatrix_x4_trans((j < 2 ? hi : lo) + boff(((j & 1) << 3) + i, n0), b[0], b[1], b[2], b[3]);
}
// [n][k] planes (n = token, 16 rows; k = channel), k-step k0:
__device__ __forceinline__ void ldb_nk_hl(uint32_t hi, uint32_t lo, int k0, int n0,
                                          uint32_t (&b)[4]) {
  const int l = threadIdx.x & 31, j = l >> 3, i = l & 7;
  ldmatrix_x4((j < 2 ? hi : lo) + boff(n0 + i, k0 + ((j & 1) << 3)), b[0], b[1], b[2], b[3]);
}
// B of two n-tiles (n0, n0 + 8) for one k-step from a [k][n] plane: b[0], b[1]
// for n0; b[2], b[3] for n0 + 8
__device__ __forceinline__ void ldb_kn_2n(uint32_t base, int k0, int n0, uint32_t (&b)[4]) {
  const int l = threadIdx.x & 31, j = l >> 3, i = l & 7;
  ldmatrix_x4_trans(base + boff(k0 + ((j & 1) << 3) + i, n0 + ((j >> 1) << 3)), b[0], b[1], b[2],
                    b[3]);
}

// d += (ah + al)(bh + bl) without the al bl term
__device__ __forceinline__ void mma3(float (&d)[4], const uint32_t (&ah)[4],
                                     const uint32_t (&al)[4], uint32_t bh0, uint32_t bh1,
                                     uint32_t bl0, uint32_t bl1) {
  mma_16816(d, al, bh0, bh1);
  mma_16816(d, ah, bl0, bl1);
  mma_16816(d, ah, bh0, bh1);
}
// ... when A is exact in bf16 (al = 0)
__device__ __forceinline__ void mma2a(float (&d)[4], const uint32_t (&ah)[4], uint32_t bh0,
                                      uint32_t bh1, uint32_t bl0, uint32_t bl1) {
  mma_16816(d, ah, bl0, bl1);
  mma_16816(d, ah, bh0, bh1);
}
// ... when B is exact in bf16 (bl = 0)
__device__ __forceinline__ void mma2b(float (&d)[4], const uint32_t (&ah)[4],
                                      const uint32_t (&al)[4], uint32_t bh0, uint32_t bh1) {
  mma_16816(d, al, bh0, bh1);
  mma_16816(d, ah, bh0, bh1);
}
__device__ __forceinline__ void negate(uint32_t (&a)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) a[i] ^= 0x80008000u;
}

// A state in registers: this warp's 32 x 32 block at rows cb = 32 (w / 4),
// columns vb = 32 (w % 4); x[mt][nt][e] is row cb + 16 mt + g + 8 (e / 2),
// column vb + 8 nt + 2 q + e % 2.
struct Block {
  float x[2][4][4];
};

__device__ __forceinline__ void block_load(Block& s, const float* src) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, g = l >> 2, q = l & 3;
  const int cb = 32 * (w >> 2), vb = 32 * (w & 3);
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = cb + 16 * mt + g + 8 * hf, c = vb + 8 * nt + 2 * q;
        const float2 v = src ? __ldcg(reinterpret_cast<const float2*>(src + (size_t)r * kD + c))
                             : make_float2(0.f, 0.f);
        s.x[mt][nt][2 * hf] = v.x;
        s.x[mt][nt][2 * hf + 1] = v.y;
      }
}
__device__ __forceinline__ void block_store(const Block& s, float* dst) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, g = l >> 2, q = l & 3;
  const int cb = 32 * (w >> 2), vb = 32 * (w & 3);
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = cb + 16 * mt + g + 8 * hf, c = vb + 8 * nt + 2 * q;
        __stcg(reinterpret_cast<float2*>(dst + (size_t)r * kD + c),
               make_float2(s.x[mt][nt][2 * hf], s.x[mt][nt][2 * hf + 1]));
      }
}
// the block's bf16 hi / lo copy into the planes at `off`
__device__ __forceinline__ void block_planes(const Block& s, unsigned char* sm, int off) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, g = l >> 2, q = l & 3;
  const int cb = 32 * (w >> 2), vb = 32 * (w & 3);
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = cb + 16 * mt + g + 8 * hf, c = vb + 8 * nt + 2 * q;
        st_split(sm + off, sm + off + kPlaneS, boff(r, c), s.x[mt][nt][2 * hf],
                 s.x[mt][nt][2 * hf + 1]);
      }
}

// 16 bytes global -> shared without registers (cp.async; completed by cp_async_wait)
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
// The S planes (hi and lo, 64 KiB, as laid out in shared memory) to global memory
__device__ __forceinline__ void planes_out(const unsigned char* sm, float* dst) {
#pragma unroll
  for (int i = 0; i < 2 * kPlaneS / 16 / kNT; ++i) {
    const int b = 16 * (threadIdx.x + i * kNT);
    __stcg(reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(dst) + b),
           *reinterpret_cast<const uint4*>(sm + OFF_S + b));
  }
}

// byte i (multiple of 16) of a kept record <-> its place in shared memory
__device__ __forceinline__ int kept_smem_off(int i) {
  return i < kKeptRU ? OFF_R + i
                     : (i < kKeptRU + kKeptAT ? OFF_ARAW + (i - kKeptRU)
                                              : OFF_TP + (i - kKeptRU - kKeptAT));
}
constexpr int kKeptPerThread = (kKeptBytes / 16 + kNT - 1) / kNT;

// ---- steps shared by the forward rebuild and the reverse step of a chunk ----
// Tokens [ts, ts + n) of head h (n <= 16; rows at or past n are zero, with a
// zero log-decay, so they change nothing).  The S planes hold the entering
// state.  On return (after a block barrier): EG, K+, K-, K~, EC, beta, rk,
// Araw, T, T', R, U, and with kBack also q^, Q+, dO, rq and P.
// Lines of the inputs of tokens [ts, ts + 16) of head h toward L2 (k, v, z,
// and q, dO when kBack): one 128-byte line per thread.
template <typename T, bool kZHead>
__device__ __forceinline__ void prefetch_chunk(const Params& P, int h, int ts, bool back) {
  constexpr int L = (int)sizeof(T) * kD / 128;  // lines per io row
  const int t = threadIdx.x >> 5, li = threadIdx.x & 31;
  const int tok = ts + t;
  if (ts < 0 || tok >= P.total) return;
  const size_t row = (size_t)tok * P.H + h;
  const char* a = nullptr;
  if (li < 4) {
    if (!kZHead) a = reinterpret_cast<const char*>(P.z + row * kD) + 128 * li;
  } else if (li < 4 + L) {
    a = static_cast<const char*>(P.k) + row * kD * sizeof(T) + 128 * (li - 4);
  } else if (li < 4 + 2 * L) {
    a = static_cast<const char*>(P.v) + row * kD * sizeof(T) + 128 * (li - 4 - L);
  } else if (back && li < 4 + 3 * L) {
    a = static_cast<const char*>(P.q) + row * kD * sizeof(T) + 128 * (li - 4 - 2 * L);
  } else if (back && li < 4 + 4 * L) {
    a = static_cast<const char*>(P.d_out) + row * kD * sizeof(T) + 128 * (li - 4 - 3 * L);
  }
  if (a) asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
}

// Tokens [ts, ts + n) of head h; `s_src`, when given, is the entering
// state's planes as kept in global memory, copied into the S planes under the
// staging (`s_out`, when given: the S planes are written there);
// `ts_next` / `next_back` name the chunk processed next, whose inputs (and
// state `s_next`, when given) are prefetched toward L2 (ts_next < 0: none).
template <typename T, bool kZHead, bool kBack, bool kKept = false>
__device__ void chunk_common(unsigned char* sm, const Params& P, int h, int ts, int n, float zc,
                             const float* s_src, const float* s_next, float* s_out,
                             int ts_next, bool next_back, const unsigned char* kept = nullptr,
                             const unsigned char* kept_next = nullptr) {
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31, g = l >> 2, q = l & 3;
  const uint32_t sb = smem_u32(sm);
  float* const QH = reinterpret_cast<float*>(sm + OFF_QH);
  float* const EG = reinterpret_cast<float*>(sm + OFF_EG);
  float* const EC = reinterpret_cast<float*>(sm + OFF_EC);
  float* const vec = reinterpret_cast<float*>(sm + OFF_VEC);
  float* const beta = vec;
  float* const Gs = reinterpret_cast<float*>(sm + (kKept ? OFF_DU : OFF_U));  // scratch
  float* const KHs = reinterpret_cast<float*>(sm + OFF_DR);  // scratch
  float* const Vs = reinterpret_cast<float*>(sm + OFF_DU);   // scratch
  __syncthreads();  // the previous chunk no longer reads any chunk array
  if (s_src) {
#pragma unroll
    for (int i = 0; i < 2 * kPlaneS / 16 / kNT; ++i) {
      const int b = 16 * (tid + i * kNT);
      cp_async16(sm + OFF_S + b, reinterpret_cast<const unsigned char*>(s_src) + b);
    }
  }
  if (s_out) planes_out(sm, s_out);
  prefetch_chunk<T, kZHead>(P, h, ts_next, next_back);
  if (s_next)  // the next chunk's entering state toward L2: one 128-byte line per thread
    asm volatile("prefetch.global.L2 [%0];" ::"l"(s_next + 32 * threadIdx.x));
  if (kept_next && tid * 128 < kKeptBytes)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(kept_next + 128 * tid));
  if (kKept) {  // this chunk's kept record, in flight during the staging
#pragma unroll
    for (int i = 0; i < kKeptPerThread; ++i) {
      const int b = 16 * (tid + i * kNT);
      if (b < kKeptBytes) cp_async16(sm + kept_smem_off(b), kept + b);
    }
  }
  {  // staging: one warp per token, four channels per lane; every load issued first
    const int t = w, c = 4 * l;
    const bool live = t < n;
    const size_t row = ((size_t)(ts + t) * P.H + h) * kD + c;
    const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 xk = live ? ld4_io<T>(static_cast<const T*>(P.k) + row) : zero4;
    float4 xq = zero4, xo = zero4, xv = zero4, zz = zero4;
    if (kBack && live) {
      xq = ld4_io<T>(static_cast<const T*>(P.q) + row);
      xo = ld4_io<T>(static_cast<const T*>(P.d_out) + row);
    }
    if (!kKept && live) xv = ld4_io<T>(static_cast<const T*>(P.v) + row);
    if (live) {
      if (kZHead) {
        const float z1 = __ldg(P.z + (size_t)(ts + t) * P.H + h);
        zz = make_float4(z1, z1, z1, z1);
      } else {
        zz = __ldg(reinterpret_cast<const float4*>(P.z + row));
      }
    }
    const float bt = (live && l == 0) ? __ldg(P.beta + (size_t)(ts + t) * P.H + h) : 0.f;
    float r = warp_sum(xk.x * xk.x + xk.y * xk.y + xk.z * xk.z + xk.w * xk.w);
    const float rk = live ? rsqrtf(r + kNormEps) : 0.f;
    st4(KHs + swz(t, c), make_float4(xk.x * rk, xk.y * rk, xk.z * rk, xk.w * rk));
    float rq = 0.f;
    if (kBack) {
      r = warp_sum(xq.x * xq.x + xq.y * xq.y + xq.z * xq.z + xq.w * xq.w);
      rq = live ? rsqrtf(r + kNormEps) : 0.f;
      st4(QH + swz(t, c), make_float4(xq.x * rq, xq.y * rq, xq.z * rq, xq.w * rq));
      st_split(sm + OFF_DO, sm + OFF_DO + kPlane, boff(t, c), xo.x, xo.y);
      st_split(sm + OFF_DO, sm + OFF_DO + kPlane, boff(t, c + 2), xo.z, xo.w);
    }
    if (!kKept) st4(Vs + swz(t, c), xv);
    st4(Gs + swz(t, c),
        live ? make_float4(log_decay_c(zz.x, zc) * kLog2e, log_decay_c(zz.y, zc) * kLog2e,
                           log_decay_c(zz.z, zc) * kLog2e, log_decay_c(zz.w, zc) * kLog2e)
             : zero4);
    if (l == 0) {
      beta[t] = bt;
      vec[32 + t] = rk;  // rk
      vec[16 + t] = rq;  // rq
      vec[48 + t] = 0.f; // db
      vec[64 + t] = 0.f; // dzh
    }
    if (tid < kD) reinterpret_cast<float*>(sm + OFF_DEC)[tid] = 0.f;
    if (tid < kC * kC) {  // accumulated by atomics below
      if (!kKept) reinterpret_cast<float*>(sm + OFF_ARAW)[tid] = 0.f;
      reinterpret_cast<float*>(sm + OFF_DPF)[tid] = 0.f;
      reinterpret_cast<float*>(sm + OFF_DTP)[tid] = 0.f;
    }
  }
  if (s_src || kKept) cp_async_wait();
  __syncthreads();
  {  // cumulative log-decay and the decayed operands: two channels, two tokens
     // per thread; the eight threads of a channel pair are adjacent lanes
    const int c = 2 * (tid >> 3), p = tid & 7, t0 = 2 * p;
    const float2 g0 = ld2(Gs + swz(t0, c)), g1 = ld2(Gs + swz(t0 + 1, c));
    float sx = g0.x + g1.x, sy = g0.y + g1.y;  // inclusive prefix over the parts
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      const float ux = __shfl_up_sync(0xffffffffu, sx, o, 8);
      const float uy = __shfl_up_sync(0xffffffffu, sy, o, 8);
      if (p >= o) {
        sx += ux;
        sy += uy;
      }
    }
    const float cx = __shfl_sync(0xffffffffu, sx, 7, 8), cy = __shfl_sync(0xffffffffu, sy, 7, 8);
    float gx = sx - (g0.x + g1.x), gy = sy - (g0.y + g1.y);
    const float ecx = ex2_approx(cx), ecy = ex2_approx(cy);
    if (p == 0) st2(EC + c, make_float2(ecx, ecy));
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int t = t0 + i;
      const float2 gv = i ? g1 : g0;
      gx += gv.x;
      gy += gv.y;
      const float egx = ex2_approx(gx), egy = ex2_approx(gy);
      const float emx = ex2_approx(-gx), emy = ex2_approx(-gy);
      const float2 kh = ld2(KHs + swz(t, c));
      st2(EG + swz(t, c), make_float2(egx, egy));
      const uint32_t o = boff(t, c);
      st_split(sm + OFF_KP, sm + OFF_KP + kPlane, o, kh.x * egx, kh.y * egy);
      st_split(sm + OFF_KM, sm + OFF_KM + kPlane, o, kh.x * emx, kh.y * emy);
      st_split(sm + OFF_KT, sm + OFF_KT + kPlane, o, kh.x * emx * ecx, kh.y * emy * ecy);
      if (kBack) {
        const float2 qh = ld2(QH + swz(t, c));
        st_split(sm + OFF_QP, sm + OFF_QP + kPlane, o, qh.x * egx, qh.y * egy);
      }
    }
  }
  __syncthreads();
  // K+ K-^T on warps 0-3 and Q+ K-^T on warps 4-7: each warp one 16 x 8 tile
  // over half of the 128 channels, summed into fp32 by shared atomics (the
  // masks are applied where the products are read)
  if ((!kKept && w < 4) || (kBack && w >= 4 && w < 8)) {
    const int nt = w & 1, kh0 = 64 * ((w >> 1) & 1);
    const uint32_t ao = sb + (w < 4 ? OFF_KP : OFF_QP);
    float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k0 = kh0; k0 < kh0 + 64; k0 += 32) {
      uint32_t ah[4], al[4], b[4];
      lda<true>(ao, 0, k0, ah);
      lda<true>(ao + kPlane, 0, k0, al);
      ldb_nk_hl(sb + OFF_KM, sb + OFF_KM + kPlane, k0, 8 * nt, b);
      mma3(acc0, ah, al, b[0], b[1], b[2], b[3]);
      lda<true>(ao, 0, k0 + 16, ah);
      lda<true>(ao + kPlane, 0, k0 + 16, al);
      ldb_nk_hl(sb + OFF_KM, sb + OFF_KM + kPlane, k0 + 16, 8 * nt, b);
      mma3(acc1, ah, al, b[0], b[1], b[2], b[3]);
    }
    float* const M = reinterpret_cast<float*>(sm + (w < 4 ? OFF_ARAW : OFF_DPF));
#pragma unroll
    for (int e = 0; e < 4; ++e)
      atomicAdd(M + (g + 8 * (e >> 1)) * kC + 8 * nt + 2 * q + (e & 1), acc0[e] + acc1[e]);
  }
  // Y = K+ S on this warp's 8 value columns; R = v - Y
  if (!kKept) {
    const int n0 = 8 * w;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 2
    for (int k0 = 0; k0 < kD; k0 += 32) {
      uint32_t bh[4], bl[4];
      ldb_kn2(sb + OFF_S, k0, n0, bh);
      ldb_kn2(sb + OFF_S + kPlaneS, k0, n0, bl);
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        uint32_t ah[4], al[4];
        lda<true>(sb + OFF_KP, 0, k0 + 16 * s, ah);
        lda<true>(sb + OFF_KP + kPlane, 0, k0 + 16 * s, al);
        mma3(acc[s], ah, al, bh[2 * s], bh[2 * s + 1], bl[2 * s], bl[2 * s + 1]);
      }
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int r = g + 8 * hf, c = n0 + 2 * q;
      const float2 v = ld2(Vs + swz(r, c));
      st_split(sm + OFF_R, sm + OFF_R + kPlane, boff(r, c), v.x - acc[0][2 * hf] - acc[1][2 * hf],
               v.y - acc[0][2 * hf + 1] - acc[1][2 * hf + 1]);
    }
  }
  // T = (I + A)^{-1} (A = diag(beta) strict_lower(K+ K-^T)) by forward
  // substitution, one lane per column, column entries updated right-looking
  // (warp 0, once warps 0-3 have added their parts of A); T' = T diag(beta)
  if (!kKept && w < 4) asm volatile("bar.sync 1, 128;" ::: "memory");
  if (!kKept && w == 0) {
    const float* const Araw = reinterpret_cast<const float*>(sm + OFF_ARAW);
    float* const Tm = reinterpret_cast<float*>(sm + OFF_T);
    const int j = l & 15;
    float col[kC];
#pragma unroll
    for (int t = 0; t < kC; ++t) col[t] = t == j ? 1.f : 0.f;
#pragma unroll
    for (int m = 0; m < kC - 1; ++m) {
      const float cm = col[m];
#pragma unroll
      for (int u = m + 1; u < kC; ++u) col[u] = fmaf(-beta[u] * Araw[u * kC + m], cm, col[u]);
    }
    if (l < kC) {
      const float bj = beta[j];
#pragma unroll
      for (int t = 0; t < kC; ++t) {
        Tm[t * kC + j] = col[t];
        st_split1(sm + OFF_TP, sm + OFF_TP + kPlane16, boff16(t, j), col[t] * bj);
      }
    }
  }
  __syncthreads();
  // U = T' R on this warp's 8 value columns
  if (!kKept) {
    const int n0 = 8 * w;
    uint32_t ah[4], al[4], b[4];
    lda<false>(sb + OFF_TP, 0, 0, ah);
    lda<false>(sb + OFF_TP + kPlane16, 0, 0, al);
    ldb_kn_hl(sb + OFF_R, sb + OFF_R + kPlane, n0, b);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    mma3(acc, ah, al, b[0], b[1], b[2], b[3]);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
      st_split(sm + OFF_U, sm + OFF_U + kPlane, boff(g + 8 * hf, n0 + 2 * q), acc[2 * hf],
               acc[2 * hf + 1]);
  }
  if (kBack && tid < kC * kC) {  // P = lower(Q+ K-^T) to its planes; the sum area back to zero
    float* const PF = reinterpret_cast<float*>(sm + OFF_DPF);
    const int a = tid >> 4, b = tid & 15;
    st_split1(sm + OFF_P, sm + OFF_P + kPlane16, boff16(a, b), b <= a ? PF[tid] : 0.f);
    PF[tid] = 0.f;
  }
  __syncthreads();
}

// S <- Diag(e^{G_C}) S + K~^T U (registers, this warp's block), its planes
// rewritten.
__device__ void advance_state(unsigned char* sm, Block& S) {
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31, g = l >> 2;
  const uint32_t sb = smem_u32(sm);
  const float* const EC = reinterpret_cast<const float*>(sm + OFF_EC);
  const int cb = 32 * (w >> 2), vb = 32 * (w & 3);
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const int c0 = cb + 16 * mt;
    uint32_t ah[4], al[4];
    lda_t<true>(sb + OFF_KT, c0, 0, ah);
    lda_t<true>(sb + OFF_KT + kPlane, c0, 0, al);
    const float e_lo = EC[c0 + g], e_hi = EC[c0 + g + 8];
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      uint32_t bh[4], bl[4];
      ldb_kn_2n(sb + OFF_U, 0, vb + 16 * np, bh);
      ldb_kn_2n(sb + OFF_U + kPlane, 0, vb + 16 * np, bl);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float* x = S.x[mt][2 * np + i];
        float acc[4] = {e_lo * x[0], e_lo * x[1], e_hi * x[2], e_hi * x[3]};
        mma3(acc, ah, al, bh[2 * i], bh[2 * i + 1], bl[2 * i], bl[2 * i + 1]);
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = acc[e];
      }
    }
  }
  block_planes(S, sm, OFF_S);
}

// The reverse step of one chunk (after chunk_common<kBack = true>): the
// chunk's gradients to global memory; dS (registers) updated to the gradient
// w.r.t. the state entering the chunk, and its planes rewritten.
template <typename T, bool kZHead>
__device__ void chunk_reverse(unsigned char* sm, const Params& P, int h, int ts, int n, float zs,
                              float zc, Block& dS) {
  // dO is exact in bf16 for bf16 inputs: its low planes are zero
  constexpr bool kExactDO = sizeof(T) == 2;
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31, g = l >> 2, q = l & 3;
  const uint32_t sb = smem_u32(sm);
  const int n0 = 8 * w;  // this warp's 8 columns of the 16-row products
  const int cb = 32 * (w >> 2), vb = 32 * (w & 3);
  const float* const EG = reinterpret_cast<const float*>(sm + OFF_EG);
  const float* const QH = reinterpret_cast<const float*>(sm + OFF_QH);
  const float* const EC = reinterpret_cast<const float*>(sm + OFF_EC);
  float* const DEC = reinterpret_cast<float*>(sm + OFF_DEC);
  float* const vec = reinterpret_cast<float*>(sm + OFF_VEC);
  const float* const beta = vec;

  // dU = P^T dO + K~ dS' and dR = T'^T dU on value columns n0..; dv out
  {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    {
      uint32_t ah[4], al[4], b[4];
      lda_t<false>(sb + OFF_P, 0, 0, ah);
      lda_t<false>(sb + OFF_P + kPlane16, 0, 0, al);
      ldb_kn_hl(sb + OFF_DO, sb + OFF_DO + kPlane, n0, b);
      if (kExactDO) mma2b(acc, ah, al, b[0], b[1]);
      else mma3(acc, ah, al, b[0], b[1], b[2], b[3]);
    }
#pragma unroll 2
    for (int k0 = 0; k0 < kD; k0 += 32) {
      uint32_t bh[4], bl[4];
      ldb_kn2(sb + OFF_DS, k0, n0, bh);
      ldb_kn2(sb + OFF_DS + kPlaneS, k0, n0, bl);
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        uint32_t ah[4], al[4];
        lda<true>(sb + OFF_KT, 0, k0 + 16 * s, ah);
        lda<true>(sb + OFF_KT + kPlane, 0, k0 + 16 * s, al);
        mma3(acc, ah, al, bh[2 * s], bh[2 * s + 1], bl[2 * s], bl[2 * s + 1]);
      }
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
      st_split(sm + OFF_DU, sm + OFF_DU + kPlane, boff(g + 8 * hf, n0 + 2 * q), acc[2 * hf],
               acc[2 * hf + 1]);
    __syncwarp();
    float dr[4] = {0.f, 0.f, 0.f, 0.f};
    {
      uint32_t ah[4], al[4], b[4];
      lda_t<false>(sb + OFF_TP, 0, 0, ah);
      lda_t<false>(sb + OFF_TP + kPlane16, 0, 0, al);
      ldb_kn_hl(sb + OFF_DU, sb + OFF_DU + kPlane, n0, b);
      mma3(dr, ah, al, b[0], b[1], b[2], b[3]);
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int t = g + 8 * hf, c = n0 + 2 * q;
      st_split(sm + OFF_DR, sm + OFF_DR + kPlane, boff(t, c), dr[2 * hf], dr[2 * hf + 1]);
      if (t < n)
        *reinterpret_cast<float2*>(P.dv + ((size_t)(ts + t) * P.H + h) * kD + c) =
            make_float2(dr[2 * hf], dr[2 * hf + 1]);
    }
  }
  // dK~ = U dS'^T and dQ+_state = dO S^T on key columns n0..
  float dkt[4] = {0.f, 0.f, 0.f, 0.f}, dqp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
  for (int k0 = 0; k0 < kD; k0 += 32) {
    uint32_t bh[4], bl[4];
    ldb_nk2(sb + OFF_DS, k0, n0, bh);
    ldb_nk2(sb + OFF_DS + kPlaneS, k0, n0, bl);
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      uint32_t ah[4], al[4];
      lda<true>(sb + OFF_U, 0, k0 + 16 * s, ah);
      lda<true>(sb + OFF_U + kPlane, 0, k0 + 16 * s, al);
      mma3(dkt, ah, al, bh[2 * s], bh[2 * s + 1], bl[2 * s], bl[2 * s + 1]);
    }
    ldb_nk2(sb + OFF_S, k0, n0, bh);
    ldb_nk2(sb + OFF_S + kPlaneS, k0, n0, bl);
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      uint32_t ah[4], al[4];
      lda<true>(sb + OFF_DO, 0, k0 + 16 * s, ah);
      if (kExactDO) {
        mma2a(dqp, ah, bh[2 * s], bh[2 * s + 1], bl[2 * s], bl[2 * s + 1]);
      } else {
        lda<true>(sb + OFF_DO + kPlane, 0, k0 + 16 * s, al);
        mma3(dqp, ah, al, bh[2 * s], bh[2 * s + 1], bl[2 * s], bl[2 * s + 1]);
      }
    }
  }
  // rowsum(S o dS') over this warp's block, into DEC
  {
    float part[4] = {0.f, 0.f, 0.f, 0.f};  // rows cb + 16 mt + g + 8 hf, index 2 mt + hf
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int r = cb + 16 * mt + g + 8 * hf, c = vb + 8 * nt + 2 * q;
          const float2 s = ld_split(sm + OFF_S, sm + OFF_S + kPlaneS, boff(r, c));
          part[2 * mt + hf] += s.x * dS.x[mt][nt][2 * hf] + s.y * dS.x[mt][nt][2 * hf + 1];
        }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      part[i] += __shfl_xor_sync(0xffffffffu, part[i], 1);
      part[i] += __shfl_xor_sync(0xffffffffu, part[i], 2);
    }
    if (q == 0)
#pragma unroll
      for (int i = 0; i < 4; ++i) atomicAdd(DEC + cb + 16 * (i >> 1) + g + 8 * (i & 1), part[i]);
  }
  __syncthreads();  // dU, dR complete; every read of the dS' planes done
  // dR S^T (= -dK+_state) on key columns n0..
  float dkp[4] = {0.f, 0.f, 0.f, 0.f};  // holds -dK+ throughout
#pragma unroll 1
  for (int k0 = 0; k0 < kD; k0 += 32) {
    uint32_t bh[4], bl[4];
    ldb_nk2(sb + OFF_S, k0, n0, bh);
    ldb_nk2(sb + OFF_S + kPlaneS, k0, n0, bl);
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      uint32_t ah[4], al[4];
      lda<true>(sb + OFF_DR, 0, k0 + 16 * s, ah);
      lda<true>(sb + OFF_DR + kPlane, 0, k0 + 16 * s, al);
      mma3(dkp, ah, al, bh[2 * s], bh[2 * s + 1], bl[2 * s], bl[2 * s + 1]);
    }
  }
  // dT' = dU R^T (warps 0-3) and dO U^T (warps 4-7): each warp one 16 x 8 tile
  // over half of the 128 value channels, summed into fp32 by shared atomics
  if (w < 8) {
    const int nt = w & 1, kh0 = 64 * ((w >> 1) & 1);
    const bool dp = w >= 4;
    const uint32_t ao = sb + (dp ? OFF_DO : OFF_DU), bo = sb + (dp ? OFF_U : OFF_R);
    float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k0 = kh0; k0 < kh0 + 64; k0 += 16) {
      uint32_t ah[4], al[4], b[4];
      lda<true>(ao, 0, k0, ah);
      ldb_nk_hl(bo, bo + kPlane, k0, 8 * nt, b);
      float (&acc)[4] = (k0 & 16) ? acc1 : acc0;
      if (kExactDO && dp) {
        mma2a(acc, ah, b[0], b[1], b[2], b[3]);
      } else {
        lda<true>(ao + kPlane, 0, k0, al);
        mma3(acc, ah, al, b[0], b[1], b[2], b[3]);
      }
    }
    float* const M = reinterpret_cast<float*>(sm + (dp ? OFF_DPF : OFF_DTP));
#pragma unroll
    for (int e = 0; e < 4; ++e)
      atomicAdd(M + (g + 8 * (e >> 1)) * kC + 8 * nt + 2 * q + (e & 1), acc0[e] + acc1[e]);
  }
  // dS <- Diag(e^{G_C}) dS' + Q+^T dO - K+^T dR (registers), then its planes
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const int c0 = cb + 16 * mt;
    uint32_t qh_[4], ql_[4], kh_[4], kl_[4];
    lda_t<true>(sb + OFF_QP, c0, 0, qh_);
    lda_t<true>(sb + OFF_QP + kPlane, c0, 0, ql_);
    lda_t<true>(sb + OFF_KP, c0, 0, kh_);
    lda_t<true>(sb + OFF_KP + kPlane, c0, 0, kl_);
    negate(kh_);
    negate(kl_);
    const float e_lo = EC[c0 + g], e_hi = EC[c0 + g + 8];
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      uint32_t oh[4], ol[4], rh[4], rl[4];
      ldb_kn_2n(sb + OFF_DO, 0, vb + 16 * np, oh);
      if (!kExactDO) ldb_kn_2n(sb + OFF_DO + kPlane, 0, vb + 16 * np, ol);
      ldb_kn_2n(sb + OFF_DR, 0, vb + 16 * np, rh);
      ldb_kn_2n(sb + OFF_DR + kPlane, 0, vb + 16 * np, rl);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float* x = dS.x[mt][2 * np + i];
        float acc[4] = {e_lo * x[0], e_lo * x[1], e_hi * x[2], e_hi * x[3]};
        if (kExactDO) mma2b(acc, qh_, ql_, oh[2 * i], oh[2 * i + 1]);
        else mma3(acc, qh_, ql_, oh[2 * i], oh[2 * i + 1], ol[2 * i], ol[2 * i + 1]);
        mma3(acc, kh_, kl_, rh[2 * i], rh[2 * i + 1], rl[2 * i], rl[2 * i + 1]);
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = acc[e];
      }
    }
  }
  block_planes(dS, sm, OFF_DS);
  __syncthreads();  // dT', dP complete
  // the UT transform: X = T^T dT (dT = dT' diag(beta)); dA = strict_lower(-X T^T);
  // dAr = diag(beta) dA; dbeta
  {
    const float* const Tm = reinterpret_cast<const float*>(sm + OFF_T);
    const float* const dTp = reinterpret_cast<const float*>(sm + OFF_DTP);
    const float* const Araw = reinterpret_cast<const float*>(sm + OFF_ARAW);
    float* const X = reinterpret_cast<float*>(sm + OFF_R);  // scratch: R is no longer read
    float* const dArF = X + kC * kC;
    float* const db = vec + 48;
    if (tid < 256) {
      const int a = tid >> 4, b = tid & 15;
      float x = 0.f, d1 = 0.f;
#pragma unroll
      for (int t = 0; t < kC; ++t) {
        x = fmaf(Tm[t * kC + a], dTp[t * kC + b], x);
        d1 = fmaf(Tm[t * kC + b], dTp[t * kC + b], d1);
      }
      X[a * kC + b] = x * beta[b];
      if (a == 0) db[b] = d1;  // from T' = T diag(beta)
      float* const dPF = reinterpret_cast<float*>(sm + OFF_DPF);
      const float dpv = b <= a ? dPF[tid] : 0.f;  // dP = lower(dO U^T)
      dPF[tid] = dpv;
      st_split1(sm + OFF_DP, sm + OFF_DP + kPlane16, boff16(a, b), dpv);
    }
    __syncthreads();
    if (tid < 256) {
      const int a = tid >> 4, b = tid & 15;
      float da = 0.f;
      if (b < a) {
#pragma unroll
        for (int m = 0; m < kC; ++m) da = fmaf(X[a * kC + m], Tm[b * kC + m], da);
        da = -da;
      }
      const float dar = beta[a] * da;
      dArF[a * kC + b] = dar;
      st_split1(sm + OFF_DAR, sm + OFF_DAR + kPlane16, boff16(a, b), dar);
      float d2 = Araw[a * kC + b] * da;  // from A = diag(beta) strict_lower(K+ K-^T)
      d2 += __shfl_xor_sync(0xffffffffu, d2, 1);
      d2 += __shfl_xor_sync(0xffffffffu, d2, 2);
      d2 += __shfl_xor_sync(0xffffffffu, d2, 4);
      d2 += __shfl_xor_sync(0xffffffffu, d2, 8);
      if (b == 0 && a < n) P.dbeta[(size_t)(ts + a) * P.H + h] = db[a] + d2;
    }
    __syncthreads();  // dAr complete
  }
  // the dg state terms (before the chunk-internal parts join dQ+ and dK+),
  // then the rest of dQ+, dK+ and dK- on key columns n0..
  float* const As = reinterpret_cast<float*>(sm + OFF_DU);  // scratch: dU is no longer read
  float* const Bs = reinterpret_cast<float*>(sm + OFF_DR);  // scratch: dR is no longer read
  const int c = n0 + 2 * q;
  float eg[4], kh[4];
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const int t = g + 8 * hf;
    const float2 e2 = ld2(EG + swz(t, c)), q2 = ld2(QH + swz(t, c));
    const float2 km = ld_split(sm + OFF_KM, sm + OFF_KM + kPlane, boff(t, c));
    eg[2 * hf] = e2.x;
    eg[2 * hf + 1] = e2.y;
    kh[2 * hf] = km.x * e2.x;
    kh[2 * hf + 1] = km.y * e2.y;
    const float ec0 = EC[c], ec1 = EC[c + 1];
    // a = dO S^T o Q+ - dR S^T o K+ ; b = dK~ o K~
    st2(As + swz(t, c), make_float2(dqp[2 * hf] * q2.x * e2.x - dkp[2 * hf] * kh[2 * hf] * e2.x,
                                    dqp[2 * hf + 1] * q2.y * e2.y -
                                        dkp[2 * hf + 1] * kh[2 * hf + 1] * e2.y));
    st2(Bs + swz(t, c), make_float2(dkt[2 * hf] * km.x * ec0,  // k^ / e^{G} = K-
                                    dkt[2 * hf + 1] * km.y * ec1));
  }
  float dkm[4] = {0.f, 0.f, 0.f, 0.f};
  {
    uint32_t b[4], ah[4], al[4];
    ldb_kn_hl(sb + OFF_KM, sb + OFF_KM + kPlane, n0, b);
    lda<false>(sb + OFF_DP, 0, 0, ah);
    lda<false>(sb + OFF_DP + kPlane16, 0, 0, al);
    mma3(dqp, ah, al, b[0], b[1], b[2], b[3]);  // += dP K-
    lda<false>(sb + OFF_DAR, 0, 0, ah);
    lda<false>(sb + OFF_DAR + kPlane16, 0, 0, al);
    negate(ah);
    negate(al);
    mma3(dkp, ah, al, b[0], b[1], b[2], b[3]);  // -dK+ -= dAr K-
    ldb_kn_hl(sb + OFF_KP, sb + OFF_KP + kPlane, n0, b);
    lda_t<false>(sb + OFF_DAR, 0, 0, ah);
    lda_t<false>(sb + OFF_DAR + kPlane16, 0, 0, al);
    mma3(dkm, ah, al, b[0], b[1], b[2], b[3]);  // dAr^T K+
    ldb_kn_hl(sb + OFF_QP, sb + OFF_QP + kPlane, n0, b);
    lda_t<false>(sb + OFF_DP, 0, 0, ah);
    lda_t<false>(sb + OFF_DP + kPlane16, 0, 0, al);
    mma3(dkm, ah, al, b[0], b[1], b[2], b[3]);  // dP^T Q+
  }
  // dq^, dk^ and the norms' partial dots
  float dqh[4], dkh[4];
  {
    float* const part = reinterpret_cast<float*>(sm + OFF_U);  // scratch: U is no longer read
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float ec = EC[c + (e & 1)];
      dqh[e] = dqp[e] * eg[e];
      dkh[e] = -dkp[e] * eg[e] + __fdividef(dkm[e] + dkt[e] * ec, eg[e]);
    }
    float pq[2], pk[2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int t = g + 8 * hf;
      const float2 q2 = ld2(QH + swz(t, c));
      pq[hf] = q2.x * dqh[2 * hf] + q2.y * dqh[2 * hf + 1];
      pk[hf] = kh[2 * hf] * dkh[2 * hf] + kh[2 * hf + 1] * dkh[2 * hf + 1];
      pq[hf] += __shfl_xor_sync(0xffffffffu, pq[hf], 1);
      pq[hf] += __shfl_xor_sync(0xffffffffu, pq[hf], 2);
      pk[hf] += __shfl_xor_sync(0xffffffffu, pk[hf], 1);
      pk[hf] += __shfl_xor_sync(0xffffffffu, pk[hf], 2);
    }
    if (q == 0) {
      part[(w * kC + g) * 2 + 0] = pq[0];
      part[(w * kC + g) * 2 + 1] = pk[0];
      part[(w * kC + g + 8) * 2 + 0] = pq[1];
      part[(w * kC + g + 8) * 2 + 1] = pk[1];
    }
  }
  __syncthreads();  // the dg state terms, partial dots, DEC
  float* const dots = reinterpret_cast<float*>(sm + OFF_KT);  // scratch: K~ is no longer read
  if (tid < 2 * kC) {
    const float* const part = reinterpret_cast<const float*>(sm + OFF_U);
    float s = 0.f;
#pragma unroll
    for (int ww = 0; ww < 16; ++ww) s += part[ww * 2 * kC + tid];
    dots[tid] = s;
  }
  __syncthreads();
  // dq, dk (this thread's four positions)
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const int t = g + 8 * hf;
    if (t >= n) continue;
    const float dotq = dots[2 * t], dotk = dots[2 * t + 1];
    const float rq = vec[16 + t], rk = vec[32 + t];
    const float2 q2 = ld2(QH + swz(t, c));
    const size_t o = ((size_t)(ts + t) * P.H + h) * kD + c;
    *reinterpret_cast<float2*>(P.dq + o) = make_float2(rq * (dqh[2 * hf] - q2.x * dotq),
                                                       rq * (dqh[2 * hf + 1] - q2.y * dotq));
    *reinterpret_cast<float2*>(P.dk + o) =
        make_float2(rk * (dkh[2 * hf] - kh[2 * hf] * dotk),
                    rk * (dkh[2 * hf + 1] - kh[2 * hf + 1] * dotk));
  }
  // dg per channel: four threads per channel (s = p, p + 4, p + 8, p + 12 for
  // the chunk-internal rectangle sums; rows 4 p .. 4 p + 3 for the rest)
  float* const dzs = reinterpret_cast<float*>(sm + OFF_DO);  // scratch: dO is no longer read
  {
    const int ch = tid >> 2, p = tid & 3;
    float zrow[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // the gate logits of rows 4 p + i, early
      const int r = min(4 * p + i, n - 1);
      zrow[i] = kZHead ? __ldg(P.z + (size_t)(ts + r) * P.H + h)
                       : __ldg(P.z + ((size_t)(ts + r) * P.H + h) * kD + ch);
    }
    const float* const dPF = reinterpret_cast<const float*>(sm + OFF_DPF);
    const float* const dArF = reinterpret_cast<const float*>(sm + OFF_R) + kC * kC;
    float qp[kC], kp[kC], rs[kC];
#pragma unroll
    for (int t = 0; t < kC; ++t) {
      const float e = EG[swz(t, ch)];
      const uint32_t o = boff(t, ch);
      const float km = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + OFF_KM + o)) +
                       __bfloat162float(
                           *reinterpret_cast<const __nv_bfloat16*>(sm + OFF_KM + kPlane + o));
      qp[t] = QH[swz(t, ch)] * e;
      kp[t] = (km * e) * e;
      rs[t] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int s = p + 4 * i;
      const uint32_t o = boff(s, ch);
      const float km = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + OFF_KM + o)) +
                       __bfloat162float(
                           *reinterpret_cast<const __nv_bfloat16*>(sm + OFF_KM + kPlane + o));
      float acc = 0.f;
#pragma unroll
      for (int t = kC - 1; t > 0; --t) {
        if (t > s) {
          acc = fmaf(dPF[t * kC + s], qp[t], acc);
          acc = fmaf(dArF[t * kC + s], kp[t], acc);
          rs[t] = fmaf(km, acc, rs[t]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kC; ++t) {
      rs[t] += __shfl_xor_sync(0xffffffffu, rs[t], 1);
      rs[t] += __shfl_xor_sync(0xffffffffu, rs[t], 2);
    }
    // suffix sums of a, prefix sums of b, for rows 4 p .. 4 p + 3
    float sa = 0.f;
#pragma unroll
    for (int t = kC - 1; t >= 0; --t) {
      if (t >= 4 * p) sa += As[swz(t, ch)];
      if (t < 4 * p + 4) qp[t] = sa;  // reuse: qp[t] = sum_{t' >= t} a_t'
    }
    float pb = 0.f;
#pragma unroll
    for (int t = 0; t < kC; ++t) {
      if (t < 4 * p + 4) {
        kp[t] = pb;  // reuse: kp[t] = sum_{t' < t} b_t'
        pb += Bs[swz(t, ch)];
      }
    }
    const float base = DEC[ch] * EC[ch];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = 4 * p + i;
      float dgv = 0.f;
#pragma unroll
      for (int t = 0; t < kC; ++t)
        if (t == r) dgv = qp[t] + kp[t] + rs[t];
      dgv += base;
      const float gd = log_decay_c(zrow[i], zc);
      const float dzv = r < n ? dgv * gd * (1.f + gd * (1.f / 5.f)) * zs : 0.f;
      if (kZHead) {
        float sum = dzv;
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        sum += __shfl_xor_sync(0xffffffffu, sum, 8);
        sum += __shfl_xor_sync(0xffffffffu, sum, 16);
        if (l < 4) atomicAdd(vec + 64 + r, sum);
      } else {
        dzs[swz(r, ch)] = dzv;
      }
    }
  }
  __syncthreads();
  if (kZHead) {
    if (tid < kC && tid < n) P.dz[(size_t)(ts + tid) * P.H + h] = vec[64 + tid];
  } else {
    const int t = tid >> 5, c4 = 4 * (tid & 31);
    if (t < n)
      *reinterpret_cast<float4*>(P.dz + ((size_t)(ts + t) * P.H + h) * kD + c4) =
          ld4(dzs + swz(t, c4));
  }
}

template <typename T, bool kZHead>
__global__ void __launch_bounds__(kNT, 1) chunk_bwd_kernel(const __grid_constant__ Params P) {
  extern __shared__ __align__(128) unsigned char sm[];
  float* const states =
      P.ws + (size_t)blockIdx.x * P.ws_states * (kState + kKeptStride / 4);  // one per chunk
  unsigned char* const kept = reinterpret_cast<unsigned char*>(states + P.ws_states * kState);

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
    const int nch = (len + kC - 1) / kC;
    if (nch > P.ws_states) {  // workspace planned for shorter sequences
      report_error(P.err, kErrDeviceCheck);
      continue;
    }
    const float zs = gate_scale(P.a_log, h), zc = gate_coef(zs);
    const size_t st_off = ((size_t)seq * P.H + h) * kState;

    // ---- forward: the state entering every chunk ----
    __syncthreads();  // the previous unit no longer reads any plane
    Block S;
    block_load(S, P.initial_state ? P.initial_state + st_off : nullptr);
    block_planes(S, sm, OFF_S);
    for (int j = 0; j + 1 < nch; ++j) {
      const int ts = bos + j * kC;
      // next: the following chunk (after the last forward one, the reverse sweep's first);
      // the entering state's planes are kept
      chunk_common<T, kZHead, false>(sm, P, h, ts, kC, zc, nullptr, nullptr,
                                     states + (size_t)j * kState, ts + kC, j + 2 == nch);
#pragma unroll
      for (int i = 0; i < kKeptPerThread; ++i) {  // the chunk's kept record
        const int b = 16 * (threadIdx.x + i * kNT);
        if (b < kKeptBytes)
          __stcg(reinterpret_cast<uint4*>(kept + (size_t)j * kKeptStride + b),
                 *reinterpret_cast<const uint4*>(sm + kept_smem_off(b)));
      }
      advance_state(sm, S);
    }
    if (nch > 0) {  // the last chunk's entering state
      __syncthreads();
      planes_out(sm, states + (size_t)(nch - 1) * kState);
    }

    // ---- reverse sweep: each chunk from its stored entering state ----
    Block dS;
    block_load(dS, P.d_final ? P.d_final + st_off : nullptr);
    block_planes(dS, sm, OFF_DS);
    for (int j = nch - 1; j >= 0; --j) {
      const int ts = bos + j * kC, n = min(kC, len - j * kC);
      const float* const s_next = j > 0 ? states + (size_t)(j - 1) * kState : nullptr;
      const unsigned char* const k_next = j > 0 ? kept + (size_t)(j - 1) * kKeptStride : nullptr;
      if (j == nch - 1)  // the last chunk has no kept record: computed in full
        chunk_common<T, kZHead, true, false>(sm, P, h, ts, n, zc, states + (size_t)j * kState,
                                             s_next, nullptr, j > 0 ? ts - kC : -1, true,
                                             nullptr, k_next);
      else
        chunk_common<T, kZHead, true, true>(sm, P, h, ts, n, zc, states + (size_t)j * kState,
                                            s_next, nullptr, j > 0 ? ts - kC : -1, true,
                                            kept + (size_t)j * kKeptStride, k_next);
      chunk_reverse<T, kZHead>(sm, P, h, ts, n, zs, zc, dS);
    }
    if (P.d_initial) block_store(dS, P.d_initial + st_off);
  }
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

int grid_for(const Problem& p) {
  return std::max(1, std::min(p.num_seqs * p.num_heads, sm_count()));
}

long long states_per_cta(const Problem& p, const int32_t* cu_host) {
  int max_len = 0;
  for (int n = 0; n < p.num_seqs; ++n) max_len = std::max(max_len, cu_host[n + 1] - cu_host[n]);
  return std::max<long long>(1, (max_len + kC - 1) / kC);
}

}  // namespace cbwd

size_t chunk_bwd_inner_bytes(const Problem& p, const int32_t* cu_host) {
  if (p.num_seqs == 0 || p.num_heads == 0) return 0;
  return (size_t)cbwd::grid_for(p) * (size_t)cbwd::states_per_cta(p, cu_host) *
         (cbwd::kState * sizeof(float) + cbwd::kKeptStride);
}

cudaError_t launch_chunk_bwd_128(const Problem& p, const BwdArgs& a, const int32_t* cu_host,
                                 void* ws, cudaStream_t st) {
  using namespace cbwd;
  if (p.num_seqs == 0) return cudaSuccess;
  static PerDeviceInit attrs;
  const cudaError_t attr = attrs.run([] {
    cudaError_t e = cudaSuccess;
    const void* kernels[] = {(const void*)chunk_bwd_kernel<float, false>,
                             (const void*)chunk_bwd_kernel<__nv_bfloat16, false>,
                             (const void*)chunk_bwd_kernel<float, true>,
                             (const void*)chunk_bwd_kernel<__nv_bfloat16, true>};
    for (const void* kf : kernels)
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
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
  prm.use_order = 0;
  const int grid = grid_for(p);
  if (p.num_seqs <= kMaxOrder) {  // longest sequences first, each unit to the least-loaded CTA
    std::vector<int> idx(p.num_seqs);
    std::iota(idx.begin(), idx.end(), 0);
    std::stable_sort(idx.begin(), idx.end(), [&](int x, int y) {
      return cu_host[x + 1] - cu_host[x] > cu_host[y + 1] - cu_host[y];
    });
    auto chunks = [&](int sq) { return (long long)((cu_host[sq + 1] - cu_host[sq] + kC - 1) / kC); };
    const int n = build_unit_schedule(idx, p.num_heads, grid, chunks, prm.order, kMaxOrder);
    if (n > 0) {
      prm.num_units = n;
      prm.use_order = 2;
    } else {
      for (int i = 0; i < p.num_seqs; ++i) prm.order[i] = idx[i];
      prm.use_order = 1;
    }
  }
  if (p.io_bf16)
    a.zhead ? chunk_bwd_kernel<__nv_bfloat16, true><<<grid, kNT, SMEM_BYTES, st>>>(prm)
            : chunk_bwd_kernel<__nv_bfloat16, false><<<grid, kNT, SMEM_BYTES, st>>>(prm);
  else
    a.zhead ? chunk_bwd_kernel<float, true><<<grid, kNT, SMEM_BYTES, st>>>(prm)
            : chunk_bwd_kernel<float, false><<<grid, kNT, SMEM_BYTES, st>>>(prm);
  return cudaGetLastError();
}

}  // namespace kda
