// kda_chunk_tc.cu -- chunked KDA prefill on the Blackwell tensor cores
// (bf16 q/k/v, fp32 gates and state, dk = dv = 128).
//
// The operation is the recurrence of mhpq.cn/news/56770, section
// "KDA 到底在算什么", S_t = (I - b k k^T) Diag(alpha) S_{t-1} + b k v^T,
// o_t = S_t^T q_t, evaluated 64 tokens (one chunk) at a time.  With G_t the
// inclusive cumulative log-decay inside the chunk (per key channel), S the
// entry state, and hats for L2-normalised vectors:
//
//   A[t,j] = b_t sum_c k^_tc k^_jc e^{G_tc-G_jc}  (j < t),  T = (I + A)^{-1}
//   P[t,j] =     sum_c q^_tc k^_jc e^{G_tc-G_jc}  (j <= t)
//   T' = T diag(b),  W = T' K+,  U~ = T' V,  U = U~ - W S
//   O = Q+ S + P U,  S <- Diag(e^{G_C}) S + Khat^T U
//
// with Q+ = q^ e^{G}, K+ = k^ e^{G}, Khat = k^ e^{G_C - G}.  The factors
// e^{G_t - G_j} span e^{+-320} across a 64-token chunk, beyond fp32, so the
// pairwise (Gram) products use one reference per 16-token query subtile:
// with r_a the cumulative log-decay before subtile a,
//   Q~_t = q^_t e^{G_t - r_a} <= 1,  K~q_t = k^_t e^{G_t - r_a} <= 1   (t in a)
//   K^(a)_j = k^_j e^{r_a - G_j}: <= e^80 for j in a, <= 1 for earlier j,
// so P[t, j] = Q~_t . K^(a)_j and A[t, j] = b_t K~q_t . K^(a)_j for every
// j <= t, and no product ever leaves the fp32 range.  The e^80 bound is what
// the lower-bounded gate buys (blog.higcp.com "猜想：K3 可能是最适合 TPU 的
// MoE 架构", section "下界衰减": log alpha >= -5, so a 16-token tile decays by
// less than e^-80 and its reciprocal stays finite).  K^(a) is formed from
// K^(a-1) by the per-channel factor e^{r_a - r_{a-1}} (>= e^-80), so only
// values that are negligible in fact underflow.
//
// Everything else is kept in the transposed orientation so that the dense
// tcgen05 GEMMs have M = 128 and the state and U can feed the tensor core
// straight from Tensor Memory:
//   Y^T = S^T K+^T,  D^T = V^T - Y^T,  U^T = D^T T'^T,
//   O^T = S^T Q+^T + U^T P^T,  S^T <- S^T Diag(e^{G_C}) + U^T Khat.
// S^T (fp32, 128 lanes = value channel) stays resident in TMEM across
// chunks; its fp16 copy, D^T and U^T are A operands read from TMEM.  D is
// formed in fp32 before its one rounding: v - S^T k cancels when a key
// already holds its value.
//
// Precision: the Gram products run as tcgen05 kind::tf32 on operands rounded
// to tf32 once (the e^80 range rules out fp16 there); the dense products
// use fp16 operands (11-bit significand; all of them are bounded by 1 or by
// the data) with fp32 accumulation.  bf16 operands there would leave ~0.2%
// relative error on the largest outputs.  The inverse's 16x16 diagonal
// blocks are solved in fp32; its off-diagonal block products run as tf32
// warp MMAs (its fp16 rounding for the tensor core bounds it anyway).
//
// One CTA (16 warps) per SM walks (sequence, head) work units, longest
// sequence first.  Per chunk:
//   TMA   q, k, v (bf16, 128B swizzle) and z (fp32) tiles into shared memory;
//   CUDA  gate g = -5 sigmoid(z), per-channel cumulative sums, L2 norms, and
//         the decayed operands written in tensor-core layouts;
//   tcgen05 (tf32)  the Gram products: four M = 64 (keys) x N = 32 blocks,
//         one per query subtile, giving P^T and A^T in TMEM;
//   CUDA  T = (I + A)^{-1}: 16x16 diagonal inverses, then a four-level series;
//   tcgen05 (f16)   the five dense products above, accumulators in TMEM.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <array>
#include <cmath>
#include <mutex>
#include <numeric>
#include <queue>
#include <vector>

#include "kda_common.cuh"
#include "kda_launch.h"
#include "tc_ptx.cuh"

namespace kda {
namespace tcp {

using namespace kda::tc;

constexpr int kC = 64;     // chunk length
constexpr int kD = 128;    // dk = dv
constexpr int kNT = 512;   // threads per CTA (16 warps; warps w, w+4, w+8, w+12 share a TMEM lane quadrant)
constexpr int kMaxOrder = 6144;

// ---- shared memory map (offsets from a 1024-byte aligned base) ----
constexpr uint32_t OFF_Q = 0;         // q stage: [2 c-blk][64 t][64 c] bf16, SW128 (TMA)
constexpr uint32_t OFF_K = 16384;     // k stage, same
constexpr uint32_t OFF_Z = 32768;     // z stage: [64 t][128 c] fp32 (TMA); then G in place
constexpr uint32_t OFF_V = 65536;     // v stage: [2 n-blk][64 j][64 n] bf16 SW128 (TMA); read for D = V - Y
constexpr uint32_t OFF_G = 81920;     // 80K: Gram A operand, later A / T / T' / P / W^T
// Gram operands (tf32, K-major, 128-byte swizzle; one region per 32-channel atom):
//   G_M (A operand, M = 128) over the q / k / z stages: [4 atoms][128 rows][32 c],
//       row t = Q~_t, row 64 + t = K~q_t;
//   G_N (B operand, N = 160) in the Gram region: [4 atoms][160 rows][32 c], K^(a)
//       (keys of subtiles 0..a, reference r_a) at rows ka_row(a) .. ka_row(a) + 16(a+1) - 1.
constexpr uint32_t G_M = OFF_Q;
constexpr uint32_t kGMAtom = 128 * 128;
constexpr uint32_t G_N = OFF_G;
constexpr uint32_t kGNAtom = 160 * 128;
constexpr int kGN = 160;
__host__ __device__ constexpr int ka_row(int a) { return 8 * a * (a + 1); }  // 0, 16, 48, 96
constexpr int kLS = 68;                       // row stride (floats) of A and T: conflict-free
// in the Gram A region once the Gram products are done:
constexpr uint32_t S_AKK = OFF_G;             // A   fp32 [64][kLS]
constexpr uint32_t S_T32 = OFF_G + 17408;     // T   fp32 [64][kLS]
constexpr uint32_t S_TP = OFF_G + 34816;      // T'  fp16 [64 t][64 j] SW128: K-major B
constexpr uint32_t G_P = OFF_G + 43008;       // P   fp16 [64 t][64 j] SW128: K-major B
constexpr uint32_t S_TPL = OFF_G + 51200;     // T' - fp16(T'), fp16, same layout as S_TP
constexpr uint32_t OFF_QPT = 163840;  // Q+^T  fp16 [128 c][64 t] SW128: MN-major B
constexpr uint32_t OFF_KPT = 180224;  // K+^T  fp16 [128 c][64 j] SW128: K-major A
constexpr uint32_t OFF_KH = 196608;   // Khat^T fp16 [128 c][64 t] SW128: K-major B
constexpr uint32_t OFF_MISC = 212992;
// misc floats
constexpr int M_BETA = 0, M_RQK = 64, M_DECAY = 192, M_TOT = 320,
              M_END = 320 + 4 * 128;
constexpr uint32_t OFF_BAR = OFF_MISC + M_END * 4;  // 3 mbarriers + tmem slot
// (fused convolution) the last three raw inputs before the chunk, fp32
// [q, k][3 tokens, oldest first][128 channels]
constexpr uint32_t OFF_HALO = OFF_BAR + 64;
// (fused convolution) the head's taps, right-aligned: fp32 [q, k][128 channels][4]
constexpr uint32_t OFF_TAPS = OFF_HALO + 2 * 3 * 128 * 4;
constexpr uint32_t SMEM_BYTES = OFF_HALO + 1024;  // + alignment slack
constexpr uint32_t SMEM_BYTES_CONV = OFF_TAPS + 2 * 128 * 4 * 4 + 1024;  // kConv variant

// ---- Tensor Memory columns (all 128 lanes) ----
constexpr uint32_t TS32 = 0;    // S^T fp32   [n][c]   128 cols
constexpr uint32_t TS16 = 128;  // S^T fp16   [n][c/2]  64 cols (A operand)
constexpr uint32_t TG = 192;    // Gram [Q~; K~q] K^(a)^T  [t][key row] 160 cols, until read back
constexpr uint32_t TY16 = 192;  // D^T = V^T - Y^T fp16 [n][t/2] 32 cols (A operand), after the Gram
constexpr uint32_t TU = 256;    // U~^T / U^T [n][t]    64 cols
constexpr uint32_t TU16 = 320;  // U^T fp16   [n][t/2]  32 cols (A operand)
constexpr uint32_t TU16L = 352; // U^T - fp16(U^T), fp16 [n][t/2] 32 cols (A operand)
constexpr uint32_t TO = 384;    // O^T fp32   [n][t]    64 cols
constexpr uint32_t TY = 448;    // Y^T = S^T K+^T fp32 [n][t] 64 cols

// largest magnitude an fp16 operand may take
constexpr float kF16Max = 65504.0f;

// Work list.  mode 0: units are (sequence, head) pairs, list[i] = the i-th
// sequence to process (longest first) when use_order == 1, or list[u] =
// seq * H + head of unit u (-1: none) when use_order == 2 (a schedule built on
// the host: CTA b runs list[b], list[b + grid], ...); token ranges from the
// device cu_seqlens.  mode 1 (splitting long sequences): list holds entries
// of kEnt ints {seq, token begin, token end, in, out, flags}; in / out are
// state slots of `ws` (>= 0), or kSlotZero / kSlotIdentity / kSlotUser (the
// caller's initial / final state of `seq`), kSlotNone for no output state;
// flags & kFlagZeroV treats v as zero; flags & kFlagNoOut writes no outputs and
// no checkpoints (a run from a stand-in entry state).
constexpr int kEnt = 6;
// kSlotAux (out only): the caller's aux_state of `seq` (the transition M of an
// affine summary).
constexpr int kSlotNone = -1, kSlotZero = -1, kSlotIdentity = -2, kSlotUser = -3, kSlotAux = -4;
constexpr int kFlagZeroV = 1, kFlagNoOut = 2;

struct Params {
  const float* beta;
  const float* a_log;   // per-head gate log-scale [H], may be null
  float* ckpt;          // state checkpoints (null: none)
  const int32_t* ckpt_off;
  int ckpt_every;
  const float* zh;      // one gate logit per (token, head), [T, H] (null: z tiles per channel)
  const float* initial_state;
  const int32_t* cu;
  __nv_bfloat16* out;   // may be null (no output written)
  float* final_state;
  float* aux_state;     // [N][H][dk][dk]: output slot kSlotAux (mode 1)
  float* ws;            // state slots [slot][H][dk][dv] (mode 1)
  int* err;
  // fused Q/K convolution (kernel variant kConv): taps [H][128][W], incoming
  // states [N][H][128][W-1] (null: zeros), and the raw q, k from which a
  // segment that starts inside its sequence takes its first halo
  const float* conv_wq;
  const float* conv_wk;
  const float* conv_sq;
  const float* conv_sk;
  const __nv_bfloat16* qraw;
  const __nv_bfloat16* kraw;
  int conv_w;
  int H, total, num_seqs, num_units, use_order, mode;
  long long spin_cycles;
  int inject_timeout;   // testing: make the first input wait of each unit unsatisfiable
  int list[kMaxOrder];
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, long long limit) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// One 16 x 8 output tile (columns 8*nt .. of a 16-wide block) of X * Y as
// tf32 warp MMAs with fp32 accumulation, stored as s * result at
// M[r0 + row][c0 + 8*nt + col].  X(row, k) is produced by `xf` (so it may
// combine several stored blocks); Y starts at (yr, yc) of a row-stride-kLS
// matrix.  One warp.  (The inverse these tiles build is rounded to fp16 for
// its MMA right after, which bounds its precision more tightly than tf32
// inputs do.)
template <typename XF>
__device__ __forceinline__ void warp_tile_tf32(XF xf, const float* Y, int yr, int yc, int K, int nt,
                                               float* M, int r0, int c0, float s, int g, int q) {
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int k0 = 0; k0 < K; k0 += 8) {
    const uint32_t a[4] = {to_tf32(xf(g, k0 + q)), to_tf32(xf(g + 8, k0 + q)),
                           to_tf32(xf(g, k0 + q + 4)), to_tf32(xf(g + 8, k0 + q + 4))};
    mma_1688_tf32(acc, a, to_tf32(Y[(yr + k0 + q) * kLS + yc + 8 * nt + g]),
                  to_tf32(Y[(yr + k0 + q + 4) * kLS + yc + 8 * nt + g]));
  }
  float* m = M + (r0 + g) * kLS + c0 + 8 * nt + 2 * q;
  m[0] = s * acc[0];
  m[1] = s * acc[1];
  m[8 * kLS] = s * acc[2];
  m[8 * kLS + 1] = s * acc[3];
}

// Store 16 consecutive values of row `row`, starting at column `col` (a
// multiple of 16, < 64), as fp16 into a 128-byte-row SW128 tile.
__device__ __forceinline__ void st_row16_f16(unsigned char* tile, int row, int col,
                                             const float (&v)[16]) {
  uint4 a, b;
  a.x = pack_f16(v[0], v[1]);   a.y = pack_f16(v[2], v[3]);
  a.z = pack_f16(v[4], v[5]);   a.w = pack_f16(v[6], v[7]);
  b.x = pack_f16(v[8], v[9]);   b.y = pack_f16(v[10], v[11]);
  b.z = pack_f16(v[12], v[13]); b.w = pack_f16(v[14], v[15]);
  const uint32_t c0 = (uint32_t)(col >> 3);
  *reinterpret_cast<uint4*>(tile + row * 128 + (((c0) ^ (row & 7)) << 4)) = a;
  *reinterpret_cast<uint4*>(tile + row * 128 + (((c0 + 1) ^ (row & 7)) << 4)) = b;
}

// Store 8 consecutive values of row `row`, starting at column `col` (a
// multiple of 8, < 64), as fp16 into a 128-byte-row SW128 tile.
__device__ __forceinline__ void st_row8_f16(unsigned char* tile, int row, int col,
                                            const float (&v)[8]) {
  const uint4 a = make_uint4(pack_f16(v[0], v[1]), pack_f16(v[2], v[3]), pack_f16(v[4], v[5]),
                             pack_f16(v[6], v[7]));
  *reinterpret_cast<uint4*>(tile + row * 128 + ((((uint32_t)col >> 3) ^ (row & 7)) << 4)) = a;
}

// Byte offset of fp32 element (row, c) of a K-major tf32 operand with the
// 128-byte swizzle: 32 channels per 128-byte row, one region of `atom`
// bytes per 32-channel group, 16-byte chunk index XOR (row % 8).
__device__ __forceinline__ uint32_t tf32_off(int row, int c, uint32_t atom) {
  return (uint32_t)(c >> 5) * atom + (uint32_t)row * 128u +
         ((((uint32_t)(c & 31) >> 2) ^ ((uint32_t)row & 7)) << 4) + ((uint32_t)(c & 3) << 2);
}

// Descriptors of 128-byte-swizzled operands at byte offset `off` from the
// base described by `base` (a 1024-byte aligned, K-major descriptor):
// K-major (8-row groups 1024 bytes apart) or MN-major (64-element atoms
// 8192 bytes apart, 8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t desc_k(uint64_t base, uint32_t off) {
  return base + (uint64_t)(off >> 4);
}
__device__ __forceinline__ uint64_t desc_mn(uint64_t base, uint32_t off) {
  return base + (uint64_t)(off >> 4) + ((uint64_t)(8192 >> 4) << 16);
}

// x rounded to tf32 (nearest, ties away), kept as an fp32 bit pattern
// The Gram's fp32 operands go to the tensor core as they are; it reads them as
// tf32, keeping the top 10 fraction bits (truncation toward zero, a mean error
// of -1/2 tf32 ulp).  Scaling them by 1 + ln(2)/2048 beforehand lifts a value
// of significand m by m ln(2)/2 ulp, which centres that error for significands
// spread log-uniformly over [1, 2) (their mean is 1/ln 2); the error stays
// within one ulp.  The lift rides on the token norms; the fp16 operands made
// from the same values take it back out.
constexpr float kTf32Lift = 1.0003384f;
constexpr float kTf32Unlift = 0.9996617f;

// Barrier of warps 0-11 (the ones inverting I + A), id 1.
__device__ __forceinline__ void inv_sync() { asm volatile("bar.sync 1, 384;" ::: "memory"); }

__device__ __forceinline__ void sync_tc() {
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

__device__ __forceinline__ bool f16_ok(float x) { return fabsf(x) < kF16Max; }

// S^T (fp32 in TMEM; lane n = value channel n) to dst[c][n], a [dk][dv]
// fp32 state; warp part cq covers key channels 32 cq .. 32 cq + 31.
__device__ __forceinline__ void write_state(float* dst, uint32_t my_lane, int row, int cq) {
  dst += row;
#pragma unroll
  for (int c0 = 32 * cq; c0 < 32 * cq + 32; c0 += 16) {
    float v[16];
    tmem_ld16(my_lane + TS32 + c0, v);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) dst[(size_t)(c0 + i) * kD] = v[i];
  }
}

// The end of a chunk, once its last products have landed in TMEM: O^T (lane
// n = value channel, column t) to out[t0 + t][h][n] in bf16 for t < len.
// Warp part cq covers 16 columns.
__device__ __forceinline__ void write_o(__nv_bfloat16* out, int H, int h, int t0, int len,
                                        uint32_t my_lane, int row, int cq) {
  __nv_bfloat16* ocol = out + ((size_t)t0 * H + h) * kD + row;
  const int col = 16 * cq;
  float v[16];
  tmem_ld16(my_lane + TO + col, v);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if (col + i < len) ocol[(size_t)(col + i) * H * kD] = __float2bfloat16_rn(v[i]);
}

// The state entering a chunk, in one TMEM read of S^T (fp32; this warp's lane
// quadrant, key channels 32 cq .. 32 cq + 31): its fp16 copy (the A operand
// of the chunk's state products) and S^T <- S^T Diag(e^{G_C}) (dec = e^{G_C}
// per key channel) ahead of the chunk's update.
__device__ __forceinline__ void prep_state(uint32_t my_lane, const float* dec, int cq,
                                           float& absmax) {
#pragma unroll
  for (int c0 = 32 * cq; c0 < 32 * cq + 32; c0 += 16) {
    float v[16];
    tmem_ld16(my_lane + TS32 + c0, v);
    tmem_ld_wait();
    uint32_t hp[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      hp[i] = pack_f16(v[2 * i], v[2 * i + 1]);
      absmax = fmaxf(absmax, fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1])));
    }
    tmem_st8(my_lane + TS16 + (c0 >> 1), hp);
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
      const float4 d4 = *reinterpret_cast<const float4*>(dec + c0 + i);
      v[i] *= d4.x; v[i + 1] *= d4.y; v[i + 2] *= d4.z; v[i + 3] *= d4.w;
    }
    tmem_st16(my_lane + TS32 + c0, v);
  }
  tmem_st_wait();
}

// q / k tile words: bf16 pairs as loaded, fp16 pairs once the fused
// convolution has rewritten them (kConv).
template <bool kF16>
__device__ __forceinline__ float tile_lo(uint32_t x) {
  if (kF16) return __half2float(__ushort_as_half((unsigned short)(x & 0xFFFFu)));
  return bf16_lo(x);
}
template <bool kF16>
__device__ __forceinline__ float tile_hi(uint32_t x) {
  if (kF16) return __half2float(__ushort_as_half((unsigned short)(x >> 16)));
  return bf16_hi(x);
}

// The fused short convolution + Swish of the chunk's raw q and k tiles (in
// the input stages, 128-byte swizzled bf16), in place, before the token norms.
// Warp w takes tensor w % 2 (q, k), 64-channel block (w / 2) % 2 and tokens
// 16 (w / 4) .. + 15; lane l the channel pair 2l, 2l + 1 of the block.  The
// three raw inputs before the chunk come from the halo area, which quarter 3
// refills with the chunk's last three raw inputs for the next chunk.  All
// threads take part (two block barriers).  Taps are right-aligned: width W
// uses the last W of four (the others zero).  The results are stored as fp16
// (11-bit significand; the raw inputs were bf16), so the tiles lose less than
// an output stored in the io dtype would; absmax tracks the fp16 range.
// Swish is evaluated as u / (1 + e^-u): the form through tanh(u/2) costs one
// multi-function op less but loses |u| 2^-12 absolutely to cancellation in
// 1 + tanh for negative u.
__device__ __forceinline__ void conv_tiles(unsigned char* sm, const Params& P, int h, int warp,
                                           int lane, float& absmax) {
  const int tens = warp & 1, blk = (warp >> 1) & 1, qt = warp >> 2;
  const int c0 = 64 * blk + 2 * lane;
  unsigned char* tile = sm + (tens ? OFF_K : OFF_Q) + blk * 8192;
  float* halo = reinterpret_cast<float*>(sm + OFF_HALO) + tens * 384;
  const float4 t4a = reinterpret_cast<const float4*>(sm + OFF_TAPS)[tens * 128 + c0];
  const float4 t4b = reinterpret_cast<const float4*>(sm + OFF_TAPS)[tens * 128 + c0 + 1];
  const float ta[4] = {t4a.x, t4a.y, t4a.z, t4a.w};
  const float tb[4] = {t4b.x, t4b.y, t4b.z, t4b.w};
  const uint32_t xo = (((uint32_t)lane & 3) << 2);
  auto word = [&](int t) -> uint32_t* {
    return reinterpret_cast<uint32_t*>(tile + t * 128 + (((((uint32_t)lane >> 2)) ^ (uint32_t)(t & 7)) << 4) + xo);
  };
  float xa[19], xb[19];  // raw inputs of tokens 16 qt - 3 .. 16 qt + 15
#pragma unroll
  for (int j = 0; j < 19; ++j) {
    const int t = 16 * qt - 3 + j;
    if (j < 3 && qt == 0) {
      xa[j] = halo[j * 128 + c0];
      xb[j] = halo[j * 128 + c0 + 1];
    } else {
      const uint32_t w = *word(t);
      xa[j] = bf16_lo(w);
      xb[j] = bf16_hi(w);
    }
  }
  __syncthreads();  // every raw input is read before any is overwritten
  if (qt == 3) {
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      halo[j * 128 + c0] = xa[16 + j];
      halo[j * 128 + c0 + 1] = xb[16 + j];
    }
  }
  __half2 hmax = __float2half2_rn(0.f);  // largest |y| of the pair, for the fp16 range check
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float ua = fmaf(ta[0], xa[i], fmaf(ta[1], xa[i + 1], fmaf(ta[2], xa[i + 2], ta[3] * xa[i + 3])));
    const float ub = fmaf(tb[0], xb[i], fmaf(tb[1], xb[i + 1], fmaf(tb[2], xb[i + 2], tb[3] * xb[i + 3])));
    // swish u sigmoid(u) = u / (1 + e^-u)
    const __half2 y2 = __floats2half2_rn(__fdividef(ua, 1.f + __expf(-ua)),
                                         __fdividef(ub, 1.f + __expf(-ub)));
    hmax = __hmax2(hmax, __habs2(y2));
    *word(16 * qt + i) = *reinterpret_cast<const uint32_t*>(&y2);
  }
  absmax = fmaxf(absmax, fmaxf(__low2float(hmax), __high2float(hmax)));
  // the converted tiles are complete for warps 0-7, which compute the token
  // norms next; warps 8-15 only signal (the next block barrier orders them)
  if (warp < 8) asm volatile("bar.sync 2, 512;" ::: "memory");
  else asm volatile("bar.arrive 2, 512;" ::: "memory");
}

// kZHead: one gate logit per (token, head) (P.zh) instead of z tiles per channel.
// kConv: q and k pass the fused short convolution + Swish first.
template <bool kZHead, bool kConv>
__global__ void __launch_bounds__(kNT, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_z,
                const __grid_constant__ Params P) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* misc = reinterpret_cast<float*>(sm + OFF_MISC);
  uint64_t* bar_qkz = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* bar_v = bar_qkz + 1;
  uint64_t* bar_mma = bar_qkz + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar_qkz + 3);
  uint64_t* bar_mma2 = bar_qkz + 4;  // the state products issued with the Gram

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = P.H;

  if (warp == 0) {
    tmem_alloc(s_tmem, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar_qkz, 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_mma2, 1);
    mbar_fence_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_z);
  }
  sync_tc();
  const uint32_t tmem = *s_tmem;
  // descriptor of the shared-memory base; per-operand descriptors add offsets
  const uint64_t dbase = make_sdesc(smem_u32(sm), 0, 1024, kSwizzle128);
  // TMEM lane quadrant w % 4 (row = tid % 128); the kWQ warps sharing a
  // quadrant split the columns of every TMEM pass (part cq)
  const uint32_t my_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  const int row = tid & 127, cq = warp >> 2;
  uint32_t ph_qkz = 0, ph_v = 0, ph_mma = 0, ph_mma2 = 0;
  bool pend_qkz = false, pend_v = false;  // TMA copies in flight (uniform)
  bool pend_mma = false, pend_mma2 = false;  // MMA commits not yet observed
  bool aborted = false;
  float absmax = 0.f;  // largest |value| this thread converted to fp16

  for (int u = blockIdx.x; u < P.num_units && !aborted; u += gridDim.x) {
    int si = u / H, h = u % H;
    int seq, bos, eos, in_slot = kSlotUser, out_slot = kSlotUser, flags = 0;
    if (P.mode == 0) {
      if (P.use_order == 2) {  // the host's schedule
        const int pk = P.list[u];
        if (pk < 0) continue;  // this CTA has no unit at this position
        si = pk / H;
        h = pk % H;
        seq = si;
      } else {
        seq = P.use_order ? P.list[si] : si;
      }
      bos = P.cu[seq];
      eos = P.cu[seq + 1];
    } else {
      const int* e = P.list + kEnt * si;
      seq = e[0]; bos = e[1]; eos = e[2]; in_slot = e[3]; out_slot = e[4]; flags = e[5];
    }
    const bool zero_v = (flags & kFlagZeroV) != 0;
    const bool no_out = (flags & kFlagNoOut) != 0;
    const int sbeg = P.mode == 0 ? bos : __ldg(P.cu + seq);  // start of the sequence
    const float zcoef = gate_coef(gate_scale(P.a_log, h));  // -e^{A_h} log2(e)
    if (bos < 0 || eos < bos || eos > P.total) {
      if (tid == 0) report_error(P.err, kErrDeviceCheck);
      continue;
    }
    const int nchunks = (eos - bos + kC - 1) / kC;
    if (tid == 0 && nchunks > 0) {
      // (testing) 16 expected bytes that no copy delivers: the wait below expires
      mbar_arrive_expect_tx(bar_qkz, (kZHead ? 32768u : 65536u) + (P.inject_timeout ? 16u : 0u));
      tma_load_3d(sm + OFF_Q, &tm_q, 0, h, bos, bar_qkz);
      tma_load_3d(sm + OFF_Q + 8192, &tm_q, 64, h, bos, bar_qkz);
      tma_load_3d(sm + OFF_K, &tm_k, 0, h, bos, bar_qkz);
      tma_load_3d(sm + OFF_K + 8192, &tm_k, 64, h, bos, bar_qkz);
      if (!kZHead) tma_load_3d(sm + OFF_Z, &tm_z, 0, h, bos, bar_qkz);
      if (!zero_v) {
        mbar_arrive_expect_tx(bar_v, 16384u);
        tma_load_3d(sm + OFF_V, &tm_v, 0, h, bos, bar_v);
        tma_load_3d(sm + OFF_V + 8192, &tm_v, 64, h, bos, bar_v);
      }
    }
    pend_qkz = nchunks > 0;
    pend_v = nchunks > 0 && !zero_v;
    // beta of the first chunk (later chunks are prefetched one chunk ahead)
    float beta_pf = 0.f;
    if (tid < min(kC, eos - bos)) beta_pf = __ldg(P.beta + (size_t)(bos + tid) * H + h);

    // ---- entry state S^T: lane n holds column n of S (fp32 and fp16) ----
    {
      const int n = row;
      const float* src = nullptr;
      if (in_slot == kSlotUser) {
        if (P.initial_state) src = P.initial_state + ((size_t)seq * H + h) * kD * kD + n;
      } else if (in_slot >= 0) {
        src = P.ws + ((size_t)in_slot * H + h) * kD * kD + n;
      }
      const float diag = in_slot == kSlotIdentity ? 1.f : 0.f;
#pragma unroll
      for (int c0 = 32 * cq; c0 < 32 * cq + 32; c0 += 16) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          v[i] = src ? __ldg(src + (size_t)(c0 + i) * kD) : (c0 + i == n ? diag : 0.f);
        tmem_st16(my_lane + TS32 + c0, v);
        uint32_t hp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          hp[i] = pack_f16(v[2 * i], v[2 * i + 1]);
          absmax = fmaxf(absmax, fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1])));
        }
        tmem_st8(my_lane + TS16 + (c0 >> 1), hp);
      }
      tmem_st_wait();
    }
    if (kConv && tid < 256) {
      // the head's taps, right-aligned (width W uses the last W of four)
      {
        const int tens = tid >> 7, c = tid & 127;
        const float* wsrc = (tens ? P.conv_wk : P.conv_wq) + ((size_t)h * kD + c) * P.conv_w;
        float t4[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int tj = j - (4 - P.conv_w);
          t4[j] = tj >= 0 ? __ldg(wsrc + tj) : 0.f;
        }
        reinterpret_cast<float4*>(sm + OFF_TAPS)[tens * 128 + c] =
            make_float4(t4[0], t4[1], t4[2], t4[3]);
      }
      // the halo before the unit's first chunk: raw inputs bos-3 .. bos-1 of the
      // sequence where they exist (a segment starting inside it), else its
      // incoming convolution state (last W-1 inputs before it), else zeros
      const int tens = tid >> 7, c = tid & 127;
      const __nv_bfloat16* raw = tens ? P.kraw : P.qraw;
      const float* cst = tens ? P.conv_sk : P.conv_sq;
      float* halo = reinterpret_cast<float*>(sm + OFF_HALO) + tens * 384;
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        const int pos = bos - 3 + j;
        float x = 0.f;
        if (pos >= sbeg) {
          x = __bfloat162float(raw[((size_t)pos * H + h) * kD + c]);
        } else if (cst) {
          const int si = pos - sbeg + (P.conv_w - 1);  // index into the W-1 kept inputs
          if (si >= 0) x = __ldg(cst + (((size_t)seq * H + h) * kD + c) * (P.conv_w - 1) + si);
        }
        halo[j * 128 + c] = x;
      }
    }
    sync_tc();

    // ---------------- B: token norms and beta of the chunk at tc0 (lenc tokens) ----------------
    // (from the q / k stages, once they hold that chunk).  Warps 0-7 only, so
    // that warp 8 can issue the U products meanwhile.
    auto norms_and_beta = [&](int tc0, int lenc) {
      if (tid >= 256) return;
      // four threads per token, one half row (32 channels, four 16-byte chunks)
      // of one 64-channel block each; the sum over a row does not depend on
      // which chunk holds which channels.  Chunk x of row t is read at
      // x ^ (t % 8), and the second block walks its chunks in the order j ^ 2,
      // so the eight lanes of a quarter warp hit eight different bank groups.
      const int t = tid >> 2, e = tid & 3;
      const int boff = (e >> 1) * 8192 + t * 128;
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int x = (((e & 1) * 4 + (j ^ ((e >> 1) << 1))) ^ (t & 7)) << 4;
        const uint4 a = *reinterpret_cast<const uint4*>(sm + OFF_Q + boff + x);
        const uint4 b = *reinterpret_cast<const uint4*>(sm + OFF_K + boff + x);
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float u = tile_lo<kConv>(aw[i]), w = tile_hi<kConv>(aw[i]);
          sq += u * u + w * w;
          u = tile_lo<kConv>(bw[i]); w = tile_hi<kConv>(bw[i]);
          sk += u * u + w * w;
        }
      }
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
      }
      if (e == 0) {
        // (rq, rk) per token, both times kTf32Lift (see the Gram operands)
        *reinterpret_cast<float2*>(misc + M_RQK + 2 * t) =
            t < lenc ? make_float2(rsqrtf(sq + kNormEps) * kTf32Lift,
                                  rsqrtf(sk + kNormEps) * kTf32Lift)
                    : make_float2(0.f, 0.f);
      }
      if (tid < kC) {
        misc[M_BETA + tid] = beta_pf;
        beta_pf = 0.f;
        if (tid < min(kC, eos - tc0 - kC)) beta_pf = __ldg(P.beta + (size_t)(tc0 + kC + tid) * H + h);
      }
    };

    bool pend_l = false;  // the previous chunk still has to write O and convert S^T
    int l_t0 = 0, l_len = 0;
    long long l_ck = -1;  // its state checkpoint slot, if it ends one
    for (int ci = 0; ci < nchunks; ++ci) {
      const int t0 = bos + ci * kC;
      const int len = min(kC, eos - t0);
      // ---------------- A: inputs ----------------
      // (from the second chunk on, A and B ran during the previous chunk's U products)
      bool ok = true;
      if (ci == 0) {
        ok = wait_bar(bar_qkz, ph_qkz, P.spin_cycles);
        if (ok) {
          ph_qkz ^= 1;
          pend_qkz = false;
        }
        if (__syncthreads_or(!ok)) { aborted = true; break; }
        if (kConv) conv_tiles(sm, P, h, warp, lane, absmax);
        norms_and_beta(t0, len);
      }

      // ---------------- C: gate and cumulative decay ----------------
      // thread = (subtile a, key channel c) with its 16 tokens t = 16a + i; a
      // warp covers 32 channels of one subtile.  With G[i] the cumulative
      // log-decay from the start of the subtile through token t (G_t - r_a),
      // F[i] = e^{G[i]} is the running product of the per-token retentions
      // alpha = e^g and E[i] = e^{-G[i]} = (1 / F[15]) prod_{j > i} alpha_j, so
      // one exponential per token gives both (no factor leaves [e^-80, e^80]).
      const int c = tid & 127, a = tid >> 7;
      float F[16], E[16];
      {
        const float* Z = reinterpret_cast<const float*>(sm + OFF_Z);
        if (kZHead) {  // one logit per (token, head): every channel gets the same gate
#pragma unroll
          for (int i = 0; i < 16; ++i)
            F[i] = 16 * a + i < len ? __ldg(P.zh + (size_t)(t0 + 16 * a + i) * H + h) : 0.f;
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) F[i] = Z[(16 * a + i) * kD + c];
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)  // alpha = e^g = 2^{g log2 e}; 1 past the sequence end
          F[i] = (16 * a + i < len) ? ex2_approx(log_decay_c(F[i], zcoef) * 1.4426950408889634f)
                                    : 1.f;
        E[15] = 1.f;
#pragma unroll
        for (int i = 14; i >= 0; --i) E[i] = E[i + 1] * F[i + 1];
#pragma unroll
        for (int i = 1; i < 16; ++i) F[i] *= F[i - 1];
        const float inv = __frcp_rn(F[15]);
#pragma unroll
        for (int i = 0; i < 16; ++i) E[i] *= inv;
        misc[M_TOT + a * kD + c] = F[15];  // e^{tot_a}, the subtile's whole decay
      }
      tc_fence_before();
      if (__syncthreads_or(!ok)) { aborted = true; break; }  // subtile totals, token norms
      tc_fence_after();

      // ---------------- D: decayed operands ----------------
      // Pass 1 reads q and k (input stages) into registers; pass 2, after a
      // barrier, writes the Gram operands over the stages and the fp16
      // operands of the dense products.
      {
        float et[4];  // e^{tot_b}: each subtile's decay
#pragma unroll
        for (int b = 0; b < 4; ++b) et[b] = misc[M_TOT + b * kD + c];
        if (a == 0) misc[M_DECAY + c] = et[0] * et[1] * et[2] * et[3];
        float qt[16], kq[16], kt[16];  // Q~, K~q (<= 1) and K~ = K^(a) (<= e^80)
        // Row t = 16a + i of a 128-byte-swizzled tile holds this thread's element in
        // 16-byte chunk (x ^ (i % 8)) with x its unswizzled chunk, so the address is
        // a per-thread base for i % 8 plus 128 i.
        {
          const unsigned char* qk = sm + OFF_Q + (c >> 6) * 8192 + 2048 * a + (c & 7) * 2;
          const uint32_t x = ((uint32_t)c & 63) >> 3;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint32_t off = 128u * i + ((x ^ (uint32_t)(i & 7)) << 4);
            const float2 rqk = *reinterpret_cast<const float2*>(misc + M_RQK + 2 * (16 * a + i));
            const uint16_t qw = *reinterpret_cast<const uint16_t*>(qk + off);
            const uint16_t kw = *reinterpret_cast<const uint16_t*>(qk + OFF_K - OFF_Q + off);
            const float q = (kConv ? __half2float(__ushort_as_half(qw))
                                   : __uint_as_float((uint32_t)qw << 16)) * rqk.x;
            const float k = (kConv ? __half2float(__ushort_as_half(kw))
                                   : __uint_as_float((uint32_t)kw << 16)) * rqk.y;
            qt[i] = q * F[i];
            kq[i] = k * F[i];
            kt[i] = k * E[i];
          }
        }
        // The previous chunk's last products read Khat, overwritten below: wait for them.
        bool okl = true;
        if (pend_l) {
          okl = wait_bar(bar_mma, ph_mma, P.spin_cycles);
          if (okl) {
            ph_mma ^= 1;
            pend_mma = false;
          }
          ok = ok && okl;
        }
        // adjacent-subtile factors e^{r_{b+1} - r_b} = e^{tot_b} (r_4 = G_C), each >= e^-80
        float ed[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) ed[b] = b >= a ? et[b] : 1.f;
        // fp16 dense operands (outside the input stages, so before the barrier), row c
        // of [c][t] (tokens 16a .. 16a+15): Q+ = Q~ e^{r_a}, K+ = K~q e^{r_a}, Khat
        // (the fp16 operands drop the tf32 lift carried by qt, kq and kt)
        const float er = (a > 0 ? et[0] : 1.f) * (a > 1 ? et[1] : 1.f) * (a > 2 ? et[2] : 1.f) *
                         kTf32Unlift;
        const float ed3 = ed[3] * kTf32Unlift;
        const uint32_t rowoff = (uint32_t)c * 128u;
#pragma unroll
        for (int h8 = 0; h8 < 2; ++h8) {
          const uint32_t off = rowoff + ((((uint32_t)(2 * a + h8)) ^ ((uint32_t)c & 7)) << 4);
          const int i0 = 8 * h8;
          float kh[8];  // Khat = K^(3) e^{G_C - r_3}, along the same chain
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float x = kt[i0 + i];
#pragma unroll
            for (int b = 0; b < 3; ++b)
              if (b >= a) x *= ed[b];
            kh[i] = x * ed3;
          }
          *reinterpret_cast<uint4*>(sm + OFF_QPT + off) = make_uint4(
              pack_f16(qt[i0] * er, qt[i0 + 1] * er), pack_f16(qt[i0 + 2] * er, qt[i0 + 3] * er),
              pack_f16(qt[i0 + 4] * er, qt[i0 + 5] * er), pack_f16(qt[i0 + 6] * er, qt[i0 + 7] * er));
          *reinterpret_cast<uint4*>(sm + OFF_KPT + off) = make_uint4(
              pack_f16(kq[i0] * er, kq[i0 + 1] * er), pack_f16(kq[i0 + 2] * er, kq[i0 + 3] * er),
              pack_f16(kq[i0 + 4] * er, kq[i0 + 5] * er), pack_f16(kq[i0 + 6] * er, kq[i0 + 7] * er));
          *reinterpret_cast<uint4*>(sm + OFF_KH + off) = make_uint4(
              pack_f16(kh[0], kh[1]), pack_f16(kh[2], kh[3]), pack_f16(kh[4], kh[5]),
              pack_f16(kh[6], kh[7]));
        }
        __syncthreads();  // every thread is done with the q / k / z stages
        {
          // A warp holds 32 consecutive channels (lane = c % 32) of 16 tokens; four
          // tokens go out per stmatrix: matrix j = token i0 + j, its row r = channels
          // 4r .. 4r+3, one 16-byte chunk of that token's 128-byte swizzled row.
          const uint32_t lj = (uint32_t)lane >> 3, lr = (uint32_t)lane & 7;
          const uint32_t so0 = 128u * lj + ((lr ^ lj) << 4);
          const uint32_t so4 = 128u * lj + ((lr ^ (4u | lj)) << 4);
          const uint32_t gm = smem_u32(sm) + G_M + (c >> 5) * kGMAtom + 2048 * a;
          const uint32_t gn = smem_u32(sm) + G_N + (c >> 5) * kGNAtom + 2048 * a;
#pragma unroll
          for (int i0 = 0; i0 < 16; i0 += 4) {
            const uint32_t so = 128u * i0 + ((i0 & 4) ? so4 : so0);
            // M-side rows: Q~ at t, K~q at 64 + t
            stmatrix_x4(gm + so, __float_as_uint(qt[i0]), __float_as_uint(qt[i0 + 1]),
                        __float_as_uint(qt[i0 + 2]), __float_as_uint(qt[i0 + 3]));
            stmatrix_x4(gm + 64 * 128 + so, __float_as_uint(kq[i0]), __float_as_uint(kq[i0 + 1]),
                        __float_as_uint(kq[i0 + 2]), __float_as_uint(kq[i0 + 3]));
            // N side: K^(a') = k^ e^{r_a' - G} for a' = a .. 3, rows ka_row(a') + t, by
            // the chain K^(a'+1) = K^(a') e^{r_a'+1 - r_a'} (no factor below e^-80)
            float v0 = kt[i0], v1 = kt[i0 + 1], v2 = kt[i0 + 2], v3 = kt[i0 + 3];
#pragma unroll
            for (int ap = 0; ap < 4; ++ap) {
              if (ap < a) continue;
              if (ap > a) {
                const float e = ed[ap - 1];
                v0 *= e; v1 *= e; v2 *= e; v3 *= e;
              }
              stmatrix_x4(gn + ka_row(ap) * 128 + so, __float_as_uint(v0), __float_as_uint(v1),
                          __float_as_uint(v2), __float_as_uint(v3));
            }
          }
        }
      }
      fence_proxy_async_smem();
      sync_tc();
      if (tid == kNT - 32) {
        // Gram, tf32: D[r][p] = M_r . N_p over the 128 channels, M = [Q~; K~q]
        // (128 rows), N = the packed K^(a) (160 rows).  Issued from the last warp,
        // the one with the least work until the Gram has landed.
        const uint32_t id_g = make_idesc_tf32(128, kGN);
#pragma unroll
        for (int kb = 0; kb < kD / 32; ++kb)
#pragma unroll
          for (int k8 = 0; k8 < 4; ++k8)
            mma_tf32_ss(tmem + TG, desc_k(dbase, G_M + kb * kGMAtom + k8 * 32),
                        desc_k(dbase, G_N + kb * kGNAtom + k8 * 32), id_g, (kb | k8) != 0);
        mma_commit(bar_mma);
      }

      // ---------------- L: the previous chunk's O; this chunk's entering state ----------------
      // While the Gram runs: the previous chunk's O to HBM (and its checkpoint), then in
      // one TMEM read of S^T (fp32) its fp16 copy (the A operand of this chunk's state
      // products) and S^T <- S^T Diag(e^{G_C}) ahead of this chunk's update.
      if (ok) {
        if (pend_l) {
          if (P.out && !no_out) write_o(P.out, H, h, l_t0, l_len, my_lane, row, cq);
          if (l_ck >= 0) write_state(P.ckpt + ((size_t)l_ck * H + h) * kD * kD, my_lane, row, cq);
        }
        prep_state(my_lane, misc + M_DECAY, cq, absmax);
      }
      pend_l = false;

      // ---------------- E: v -> fp16 while the Gram runs; read back P and A ----------------
      {
        if (!zero_v) {
          const bool okv = wait_bar(bar_v, ph_v, P.spin_cycles);
          if (okv) {
            ph_v ^= 1;
            pend_v = false;
          }
          ok = ok && okv;
        }
        const bool okg = wait_bar(bar_mma, ph_mma, P.spin_cycles);
        if (okg) ph_mma ^= 1;
        pend_mma = !okg;
        ok = ok && okg;
      }
      if (__syncthreads_or(!ok)) { aborted = true; break; }
      tc_fence_after();
      if (tid == 0 && ci + 1 < nchunks) {  // q / k / z stages are free: prefetch the next chunk
        const int tn = t0 + kC;
        mbar_arrive_expect_tx(bar_qkz, kZHead ? 32768u : 65536u);
        tma_load_3d(sm + OFF_Q, &tm_q, 0, h, tn, bar_qkz);
        tma_load_3d(sm + OFF_Q + 8192, &tm_q, 64, h, tn, bar_qkz);
        tma_load_3d(sm + OFF_K, &tm_k, 0, h, tn, bar_qkz);
        tma_load_3d(sm + OFF_K + 8192, &tm_k, 64, h, tn, bar_qkz);
        if (!kZHead) tma_load_3d(sm + OFF_Z, &tm_z, 0, h, tn, bar_qkz);
      }
      pend_qkz = ci + 1 < nchunks;
      {
        // TMEM row r = 32 (w % 4) + lane: P row t = r (r < 64) or A row t = r - 64.
        // Warp w / 4 takes key subtile b; row t (query subtile a) finds key j =
        // 16b + i of K^(a) at column ka_row(a) + j.  The two query subtiles of a
        // warp read their columns in two loads.
        const int s = warp & 3, b = warp >> 2;
        const int r = 32 * s + lane, t = r & 63, a = t >> 4;
        const int alo = 2 * (s & 1), ahi = alo + 1;  // subtiles of lanes 0-15 / 16-31
        float v[16], w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) { v[i] = 0.f; w[i] = 0.f; }
        const uint32_t tl = tmem + ((uint32_t)(32 * s) << 16) + TG;
        if (b <= alo) tmem_ld16(tl + ka_row(alo) + 16 * b, v);
        if (b <= ahi) tmem_ld16(tl + ka_row(ahi) + 16 * b, w);
        tmem_ld_wait();
        if (a == ahi) {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = w[i];
        }
        if (r < 64) {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = (b <= a && 16 * b + i <= t) ? v[i] : 0.f;
          st_row16_f16(sm + G_P, t, 16 * b, v);
        } else if (b <= a) {
          float* Akk = reinterpret_cast<float*>(sm + S_AKK) + t * kLS + 16 * b;
          const float bt = misc[M_BETA + t];
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            *reinterpret_cast<float4*>(Akk + i) =
                make_float4(16 * b + i < t ? bt * v[i] : 0.f, 16 * b + i + 1 < t ? bt * v[i + 1] : 0.f,
                            16 * b + i + 2 < t ? bt * v[i + 2] : 0.f,
                            16 * b + i + 3 < t ? bt * v[i + 3] : 0.f);
        }
      }
      __syncthreads();

      // ---------------- F: T = (I + A)^{-1},  T' = T diag(beta) ----------------
      {
        const int g = lane >> 2, q4 = lane & 3;
        float* Akk = reinterpret_cast<float*>(sm + S_AKK);
        float* T = reinterpret_cast<float*>(sm + S_T32);
        // T' (fp16, [t][j] rows) = T diag(beta), zero above the block diagonal, for
        // task k = (row 16 br + k / 8, columns 8 (k % 8) .. + 7) of block row br, once
        // that block row of T is final
        auto build_tp = [&](int br, int k) {
          const int t = 16 * br + (k >> 3), j0 = (k & 7) * 8;
          const int bj = j0 >> 4;
          const float* src = (bj == br ? T : Akk) + t * kLS + j0;
          float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
          if (bj <= br) {
            x0 = *reinterpret_cast<const float4*>(src);
            x1 = *reinterpret_cast<const float4*>(src + 4);
          }
          const float4 b0 = *reinterpret_cast<const float4*>(misc + M_BETA + j0);
          const float4 b1 = *reinterpret_cast<const float4*>(misc + M_BETA + j0 + 4);
          const float v[8] = {x0.x * b0.x, x0.y * b0.y, x0.z * b0.z, x0.w * b0.w,
                              x1.x * b1.x, x1.y * b1.y, x1.z * b1.z, x1.w * b1.w};
          st_row8_f16(sm + S_TP, t, j0, v);
          float lo[8];  // what the fp16 rounding of T' dropped
#pragma unroll
          for (int i = 0; i < 8; ++i) lo[i] = v[i] - __half2float(__float2half_rn(v[i]));
          st_row8_f16(sm + S_TPL, t, j0, lo);
        };
        // Warps 0-11 invert.  Meanwhile warps 12-15 run the state products
        // O^T = S^T Q+^T and Y^T = S^T K+^T (M=128 value channels, N=64 tokens,
        // K=128 key channels; they only need the entry state) and convert Y^T to
        // fp16, and warps 4-11, idle during the diagonal solves, decay S^T (fp32)
        // by e^{G_C} ahead of this chunk's update.
        pend_mma2 = true;
        if (warp < 4) {
          if (lane < 16) {
            // diagonal block `warp`, column `lane` of its inverse: forward
            // substitution, each solved entry swept into the rows below it
            const int base = 16 * warp, cc = lane;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = (i == cc) ? 1.f : 0.f;
#pragma unroll
            for (int i = 0; i < 15; ++i) {
#pragma unroll
              for (int k = i + 1; k < 16; ++k) x[k] -= Akk[(base + k) * kLS + base + i] * x[i];
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) T[(base + i) * kLS + base + cc] = x[i];
          }
        } else if (warp >= 12) {
          if (warp == 12 && lane == 0) {
            const uint32_t id_o = make_idesc_f16(128, kC, false, true);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
              mma_ts(tmem + TO, tmem + TS16 + kk * 8, desc_mn(dbase, OFF_QPT + kk * 2048), id_o,
                     kk > 0);
              mma_ts(tmem + TY, tmem + TS16 + kk * 8, desc_mn(dbase, OFF_KPT + kk * 2048), id_o,
                     kk > 0);
            }
            mma_commit(bar_mma2);
          }
          __syncwarp();
          const bool okm = wait_bar(bar_mma2, ph_mma2, P.spin_cycles);
          tc_fence_after();
          if (okm) {
            // D^T = V^T - Y^T (lane n = value channel, column t = token), formed in
            // fp32 and rounded to fp16 once: the delta rule's correction v - S^T k
            // cancels when a key already holds its value, so rounding Y first
            // would cost 2^-12 |Y| rather than 2^-12 |D|.  V[t][n] is read from
            // the bf16 stage (row t, 16-byte chunk (n % 64) / 8 XOR t % 8).
            const int n = row;
            const unsigned char* vb = sm + OFF_V + (n >> 6) * 8192 + ((n & 7) << 1);
            const uint32_t xn = ((uint32_t)n & 63) >> 3;
#pragma unroll
            for (int col = 0; col < kC; col += 16) {
              float v[16];
              tmem_ld16(my_lane + TY + col, v);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int t = col + i;
                const float vt = zero_v ? 0.f
                                        : __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t*>(
                                                              vb + t * 128 + ((xn ^ (uint32_t)(t & 7)) << 4))
                                                          << 16);
                v[i] = vt - v[i];
              }
              uint32_t hp[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                hp[i] = pack_f16(v[2 * i], v[2 * i + 1]);
                absmax = fmaxf(absmax, fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1])));
              }
              tmem_st8(my_lane + TY16 + (col >> 1), hp);
            }
            tmem_st_wait();
          }
          ok = ok && okm;
        }
        if (warp < 12) {
          inv_sync();
          // Off-diagonal blocks.  With D = blockdiag(I + A_aa) (inverses T_aa above)
          // and L the blocks below it, I + A = D (I + N), N = D^{-1} L, N^4 = 0, so
          //   T = (I - N + N^2 - N^3) D^{-1},   T_ab = X_ab T_bb.
          // Four levels of 16x16 products in 16x8 tiles (one per warp).  N lives
          // in T's lower blocks, N^2 / N^3 in T's unused upper blocks, and the
          // final off-diagonal T_ab overwrite A's lower blocks.
          {
            float* Afin = Akk;
            auto blk = [&](const float* M, int r0, int c0) {
              return [M, r0, c0](int r, int k) { return M[(r0 + r) * kLS + c0 + k]; };
            };
            // level A: N_ab = T_aa A_ab for the six blocks a > b
            if (warp < 12) {
              const int bi = warp >> 1, nt = warp & 1;
              const int a = bi < 3 ? bi + 1 : (bi < 5 ? bi - 1 : 3);
              const int b = bi < 3 ? bi : (bi < 5 ? bi - 3 : 0);
              warp_tile_tf32(blk(T, 16 * a, 16 * a), Akk, 16 * a, 16 * b, 16, nt, T, 16 * a, 16 * b,
                              1.f, g, q4);
            }
            inv_sync();
            // level B: N^2_20, N^2_31, N^2_30 (upper blocks 02, 13, 03) and T_10, T_21, T_32
            if (warp < 12) {
              const int nt = warp & 1;
              switch (warp >> 1) {
                case 0: warp_tile_tf32(blk(T, 32, 16), T, 16, 0, 16, nt, T, 0, 32, 1.f, g, q4); break;
                case 1: warp_tile_tf32(blk(T, 48, 32), T, 32, 16, 16, nt, T, 16, 48, 1.f, g, q4); break;
                case 2: warp_tile_tf32(blk(T, 48, 16), T, 16, 0, 32, nt, T, 0, 48, 1.f, g, q4); break;
                case 3: warp_tile_tf32(blk(T, 16, 0), T, 0, 0, 16, nt, Afin, 16, 0, -1.f, g, q4); break;
                case 4: warp_tile_tf32(blk(T, 32, 16), T, 16, 16, 16, nt, Afin, 32, 16, -1.f, g, q4); break;
                default: warp_tile_tf32(blk(T, 48, 32), T, 32, 32, 16, nt, Afin, 48, 32, -1.f, g, q4); break;
              }
            }
            inv_sync();
            // level C: N^3_30 = N_32 N^2_20 (upper block 23); T_20 = (N^2_20 - N_20) T_00;
            // T_31 = (N^2_31 - N_31) T_11
            if (warp < 6) {
              const int task = warp >> 1, nt = warp & 1;
              if (task == 0) {
                warp_tile_tf32(blk(T, 48, 32), T, 0, 32, 16, nt, T, 32, 48, 1.f, g, q4);
              } else if (task == 1) {
                auto xf = [T](int r, int k) { return T[r * kLS + 32 + k] - T[(32 + r) * kLS + k]; };
                warp_tile_tf32(xf, T, 0, 0, 16, nt, Afin, 32, 0, 1.f, g, q4);
              } else {
                auto xf = [T](int r, int k) {
                  return T[(16 + r) * kLS + 48 + k] - T[(48 + r) * kLS + 16 + k];
                };
                warp_tile_tf32(xf, T, 16, 16, 16, nt, Afin, 48, 16, 1.f, g, q4);
              }
            } else if (warp >= 8) {
              build_tp(0, tid - 256);  // T' block row 0 (T_00 is final)
            }
            inv_sync();
            // level D: T_30 = (N^2_30 - N_30 - N^3_30) T_00
            if (warp < 2) {
              auto xf = [T](int r, int k) {
                return T[r * kLS + 48 + k] - T[(48 + r) * kLS + k] - T[(32 + r) * kLS + 48 + k];
              };
              warp_tile_tf32(xf, T, 0, 0, 16, warp, Afin, 48, 0, 1.f, g, q4);
            } else if (tid >= 64 && tid < 320) {
              build_tp(1 + ((tid - 64) >> 7), (tid - 64) & 127);  // T' block rows 1, 2
            }
          }
        }
        __syncthreads();  // T, the final off-diagonal blocks and the side work are done
        if (tid < 128) build_tp(3, tid);  // T' block row 3
      }
      fence_proxy_async_smem();
      tc_fence_before();
      if (__syncthreads_or(!ok)) { aborted = true; break; }
      tc_fence_after();
      ph_mma2 ^= 1;
      pend_mma2 = false;

      // ---------------- G: U^T = D^T T'^T,  D = V - Y ----------------
      if (tid == 256) {  // warp 8: no norm work below
        const uint32_t id_u = make_idesc_f16(128, kC, false, false);
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_ts(tmem + TU, tmem + TY16 + kk * 8, desc_k(dbase, S_TP + kk * 32), id_u, kk > 0);
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)  // + the part of T' its fp16 rounding dropped
          mma_ts(tmem + TU, tmem + TY16 + kk * 8, desc_k(dbase, S_TPL + kk * 32), id_u, true);
        mma_commit(bar_mma);
      }
      pend_mma = true;
      // A and B of the next chunk (its q / k / z landed during this one) while
      // the U products run
      bool okq = true;
      if (ci + 1 < nchunks) {
        okq = wait_bar(bar_qkz, ph_qkz, P.spin_cycles);
        if (okq) {
          ph_qkz ^= 1;
          pend_qkz = false;
        }
        // every lane runs it (its shuffles need the whole warp); after a timeout
        // the values are not used
        if (kConv) conv_tiles(sm, P, h, warp, lane, absmax);
        norms_and_beta(t0 + kC, min(kC, eos - t0 - kC));
      }
      ok = wait_bar(bar_mma, ph_mma, P.spin_cycles);
      if (ok) {
        ph_mma ^= 1;
        pend_mma = false;
      }
      if (__syncthreads_or(!ok || !okq)) { aborted = true; break; }
      tc_fence_after();
      if (tid == 0 && ci + 1 < nchunks && !zero_v) {  // v stage consumed: prefetch
        const int tn = t0 + kC;
        mbar_arrive_expect_tx(bar_v, 16384u);
        tma_load_3d(sm + OFF_V, &tm_v, 0, h, tn, bar_v);
        tma_load_3d(sm + OFF_V + 8192, &tm_v, 64, h, tn, bar_v);
      }
      pend_v = (ci + 1 < nchunks) && !zero_v;

      // ---------------- J: U^T -> fp16 in TMEM, and what that rounding drops ----------------
      {
        float v[16];
        tmem_ld16(my_lane + TU + 16 * cq, v);
        tmem_ld_wait();
        uint32_t hp[8], lp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          hp[i] = pack_f16(v[2 * i], v[2 * i + 1]);
          absmax = fmaxf(absmax, fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1])));
          const float2 h2 = __half22float2(*reinterpret_cast<const __half2*>(&hp[i]));
          lp[i] = pack_f16(v[2 * i] - h2.x, v[2 * i + 1] - h2.y);
        }
        tmem_st8(my_lane + TU16 + 8 * cq, hp);
        tmem_st8(my_lane + TU16L + 8 * cq, lp);
        tmem_st_wait();
      }
      sync_tc();

      // ---------------- K: O^T += U^T P^T;  S^T += U^T Khat ----------------
      if (tid == 0) {
        const uint32_t id_o = make_idesc_f16(128, kC, false, false);
        const uint32_t id_s = make_idesc_f16(128, kD, false, false);
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk) {
          const uint32_t au = tmem + TU16 + kk * 8, al = tmem + TU16L + kk * 8;
          mma_ts(tmem + TO, au, desc_k(dbase, G_P + kk * 32), id_o, true);
          mma_ts(tmem + TS32, au, desc_k(dbase, OFF_KH + kk * 32), id_s, true);
          mma_ts(tmem + TO, al, desc_k(dbase, G_P + kk * 32), id_o, true);
          mma_ts(tmem + TS32, al, desc_k(dbase, OFF_KH + kk * 32), id_s, true);
        }
        mma_commit(bar_mma);
      }
      // O and S^T are finished (L) while the next chunk computes its gates
      pend_mma = true;
      pend_l = true;
      l_t0 = t0;
      l_len = len;
      l_ck = -1;
      if (P.ckpt && !no_out && (t0 + len - sbeg) % P.ckpt_every == 0)
        l_ck = (long long)__ldg(P.ckpt_off + seq) + (t0 + len - sbeg) / P.ckpt_every - 1;
    }
    if (aborted) break;
    if (pend_l) {
      // ---------------- L (last chunk): write O ----------------
      const bool okl = wait_bar(bar_mma, ph_mma, P.spin_cycles);
      if (okl) {
        ph_mma ^= 1;
        pend_mma = false;
        tc_fence_after();
        if (P.out && !no_out) write_o(P.out, H, h, l_t0, l_len, my_lane, row, cq);
        if (l_ck >= 0) write_state(P.ckpt + ((size_t)l_ck * H + h) * kD * kD, my_lane, row, cq);
      }
      pend_l = false;
      tc_fence_before();
      if (__syncthreads_or(!okl)) { aborted = true; break; }
    }
    if (aborted) break;

    // ---- final state: lane n holds column n ----
    float* dst = nullptr;
    if (out_slot == kSlotUser) {
      if (P.final_state) dst = P.final_state + ((size_t)seq * H + h) * kD * kD;
    } else if (out_slot == kSlotAux) {
      if (P.aux_state) dst = P.aux_state + ((size_t)seq * H + h) * kD * kD;
    } else if (out_slot >= 0) {
      dst = P.ws + ((size_t)out_slot * H + h) * kD * kD;
    }
    if (dst) write_state(dst, my_lane, row, cq);
    sync_tc();
  }

  if (!(absmax < kF16Max)) report_error(P.err, kErrDeviceCheck);
  if (aborted) {
    if (tid == 0) {
      report_error(P.err, kErrTimeout);
      // let copies already in flight land before the shared memory goes away
      if (pend_qkz) {
        if (P.inject_timeout) mbar_complete_tx(bar_qkz, 16u);  // cancel the injected bytes
        wait_bar(bar_qkz, ph_qkz, P.spin_cycles);
      }
      if (pend_v) wait_bar(bar_v, ph_v, P.spin_cycles);
      if (pend_mma) wait_bar(bar_mma, ph_mma, P.spin_cycles);
      if (pend_mma2) wait_bar(bar_mma2, ph_mma2, P.spin_cycles);
    }
  }
  sync_tc();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------- host -----

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

#pragma GCC diagnostic push
#pragma GCC diagnostic ignored "-Wdeprecated-declarations"
EncodeFn get_encode() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}
#pragma GCC diagnostic pop

bool make_map(CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, int esize, int H, int T,
              int box_c, CUtensorMapSwizzle sw) {
  EncodeFn enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)T};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * esize, (cuuint64_t)H * kD * esize};
  const cuuint32_t box[3] = {(cuuint32_t)box_c, 1u, (cuuint32_t)kC};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return enc(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------- splitting long sequences --
//
// When there are fewer (sequence, head) units than SMs, a long sequence is cut
// into segments that run in parallel (the intra-device counterpart of the
// context-parallel scheme of blog.higcp.com "猜想：K3 可能是最适合 TPU 的 MoE
// 架构", section "第二层"): the state after a segment is affine in the state
// before it, S_out = M S_in + S~, with M the product of the segment's
// per-token transitions (the final state of the segment run from S_in = I
// with v = 0) and S~ the final state run from S_in = 0.  Pass 1 computes
// (S~, M) for the inner segments, while the first segment runs from the true
// initial state and writes its outputs; a prefix scan S_in(p+1) = M_p S_in(p)
// + S~_p yields every segment's entry state, and pass 2 runs every other
// segment from its entry state, writing the outputs and, for the last
// segment, the final state.

constexpr int kScanThreads = 256;
constexpr int kMaxScanSeqs = 512;
constexpr int kScanLd = 132;  // padded row (floats) of the scan's shared tiles
// dynamic shared memory of the scan: Mt and Ss (padded), and M as copied in
constexpr size_t kScanSmem = (2 * (size_t)kD * kScanLd + (size_t)kD * kD) * sizeof(float);

struct ScanSeq {
  int seq, base, nseg;
};
struct ScanParams {
  const float* initial_state;  // caller's, may be null
  float* ws;
  int H, E;
  ScanSeq s[kMaxScanSeqs];
};

// One CTA per (sequence, head), fp32: entry state of segment 0 (a copy of
// the initial state, so that the final state may alias it), then
// S_in(p+1) = M_p S_in(p) + S~_p for the inner segments.  Thread (ty, tx)
// owns rows 8ty.. and columns 8tx.. of the 128 x 128 state.
__global__ void __launch_bounds__(kScanThreads)
state_scan_kernel(const __grid_constant__ ScanParams Q) {
  extern __shared__ __align__(16) float scan_smem[];
  float* Mt = scan_smem;                 // M transposed: Mt[k][c]
  float* Ss = scan_smem + kD * kScanLd;  // current state: Ss[k][j]
  float* Mr = scan_smem + 2 * kD * kScanLd;  // M as stored, [c][k]
  const ScanSeq sq = Q.s[blockIdx.x / Q.H];
  const int h = blockIdx.x % Q.H, tid = threadIdx.x;
  const int r0 = (tid >> 4) * 8, c0 = (tid & 15) * 8;
  const size_t st = (size_t)kD * kD;
  auto slot = [&](int s) { return Q.ws + ((size_t)s * Q.H + h) * st; };
  {
    float* dst = slot(sq.base);
    const float* src = Q.initial_state ? Q.initial_state + ((size_t)sq.seq * Q.H + h) * st : nullptr;
    for (int i = 0; i < 8; ++i)
      for (int j = 0; j < 8; j += 4) {
        const size_t o = (size_t)(r0 + i) * kD + c0 + j;
        *reinterpret_cast<float4*>(dst + o) =
            src ? *reinterpret_cast<const float4*>(src + o) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
  }
  if (sq.nseg < 3) return;
  float s[8][8];
  {
    const float* src = slot(sq.base + 1);
    for (int i = 0; i < 8; ++i)
      for (int j = 0; j < 8; ++j) s[i][j] = src[(size_t)(r0 + i) * kD + c0 + j];
  }
  for (int p = 1; p + 1 < sq.nseg; ++p) {
    const float* M = slot(2 * Q.E + sq.base + p);
    const float* St = slot(Q.E + sq.base + p);
    __syncthreads();
    // M into shared memory in one round trip (16-byte cp.async pieces), then
    // transposed there
#pragma unroll
    for (int i = 0; i < kD * kD / 4 / kScanThreads; ++i) {
      const int e = 4 * (tid + i * kScanThreads);
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(Mr + e)),
                   "l"(M + e)
                   : "memory");
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    for (int idx = tid; idx < kD * kD; idx += kScanThreads) {
      const int c = idx >> 7, k = idx & 127;
      Mt[k * kScanLd + c] = Mr[idx];
    }
    for (int i = 0; i < 8; ++i)
      for (int j = 0; j < 8; ++j) Ss[(r0 + i) * kScanLd + c0 + j] = s[i][j];
    __syncthreads();
    float acc[8][8];
    for (int i = 0; i < 8; ++i)
      for (int j = 0; j < 8; ++j) acc[i][j] = St[(size_t)(r0 + i) * kD + c0 + j];
#pragma unroll 4
    for (int k = 0; k < kD; ++k) {
      const float4 m0 = *reinterpret_cast<const float4*>(Mt + k * kScanLd + r0);
      const float4 m1 = *reinterpret_cast<const float4*>(Mt + k * kScanLd + r0 + 4);
      const float4 s0 = *reinterpret_cast<const float4*>(Ss + k * kScanLd + c0);
      const float4 s1 = *reinterpret_cast<const float4*>(Ss + k * kScanLd + c0 + 4);
      const float mv[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
      const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(mv[i], sv[j], acc[i][j]);
    }
    float* dst = slot(sq.base + p + 1);
    for (int i = 0; i < 8; ++i)
      for (int j = 0; j < 8; ++j) {
        s[i][j] = acc[i][j];
        dst[(size_t)(r0 + i) * kD + c0 + j] = acc[i][j];
      }
  }
}

struct SplitPlan {
  bool use = false;
  int seg_len = 0, seg0_len = 0, E = 0;  // tokens of segments 1, 2, .. and of segment 0
  int s0_at = -1;  // pass 1: position of the block of segment-0 entries among the inner
                   // entries, or -1 for each before its own sequence's
  std::vector<int> nseg, base;
  size_t bytes = 0;
};

constexpr int kMaxEntries = kMaxOrder / kEnt;

// launches (from this host thread) that still get an unsatisfiable input wait
thread_local int g_inject_wait_timeout = 0;

// Token range of segment q of sequence n.
void seg_range(const SplitPlan& pl, const int32_t* cu, int n, int q, int& tb, int& te) {
  tb = q == 0 ? cu[n] : cu[n] + pl.seg0_len + (q - 1) * pl.seg_len;
  te = std::min(cu[n + 1], tb + (q == 0 ? pl.seg0_len : pl.seg_len));
}

struct RunEntry {
  int n, tb, te, in, out, flags;
};

// Pass 1: segment 0 of every split sequence, from the true initial state, and
// the two runs (S~ from zero, M from the identity) of every inner segment.
std::vector<RunEntry> pass1_entries(const SplitPlan& pl, const int32_t* cu, int num_seqs) {
  std::vector<RunEntry> inner, first, all;
  for (int n = 0; n < num_seqs; ++n) {
    const int k = pl.nseg[n], b = pl.base[n];
    if (k < 2) continue;
    int tb, te;
    seg_range(pl, cu, n, 0, tb, te);
    const RunEntry e0{n, tb, te, kSlotUser, b + 1, 0};
    if (pl.s0_at < 0) all.push_back(e0);
    else first.push_back(e0);
    for (int q = 1; q + 1 < k; ++q) {
      seg_range(pl, cu, n, q, tb, te);
      const RunEntry es{n, tb, te, kSlotZero, pl.E + b + q, kFlagNoOut};
      const RunEntry em{n, tb, te, kSlotIdentity, 2 * pl.E + b + q, kFlagZeroV | kFlagNoOut};
      if (pl.s0_at < 0) {
        all.push_back(es);
        all.push_back(em);
      } else {
        inner.push_back(es);
        inner.push_back(em);
      }
    }
  }
  if (pl.s0_at < 0) return all;
  const size_t at = std::min<size_t>((size_t)pl.s0_at, inner.size());
  all.assign(inner.begin(), inner.begin() + at);
  all.insert(all.end(), first.begin(), first.end());
  all.insert(all.end(), inner.begin() + at, inner.end());
  return all;
}

// Pass 2: every segment but a split sequence's first (and every unsplit
// sequence), from its entry state, longest first.
std::vector<RunEntry> pass2_entries(const SplitPlan& pl, const int32_t* cu, int num_seqs) {
  std::vector<std::array<int, 4>> segs;  // {len, n, q, k}
  for (int n = 0; n < num_seqs; ++n)
    for (int q = pl.nseg[n] >= 2 ? 1 : 0; q < pl.nseg[n]; ++q) {
      int tb, te;
      seg_range(pl, cu, n, q, tb, te);
      segs.push_back({te - tb, n, q, pl.nseg[n]});
    }
  std::stable_sort(segs.begin(), segs.end(),
                   [](const std::array<int, 4>& x, const std::array<int, 4>& y) { return x[0] > y[0]; });
  std::vector<RunEntry> all;
  for (const auto& sg : segs) {
    int tb, te;
    seg_range(pl, cu, sg[1], sg[2], tb, te);
    all.push_back({sg[1], tb, te, pl.base[sg[1]] + sg[2], sg[2] + 1 == sg[3] ? kSlotUser : kSlotNone,
                   0});
  }
  return all;
}

// Chunk-times until the last of a launch's units ends, given its entries'
// lengths in chunks: unit u is entry u / H, and CTA b of the min(units, sms)
// runs units b, b + grid, ...
double static_makespan(const std::vector<int>& len, int H, int sms, std::vector<double>& t) {
  const long units = (long)len.size() * H;
  if (units == 0) return 0.0;
  const long grid = std::min<long>(units, sms);
  t.assign(grid, 0.0);
  long b = 0;  // the CTA of unit i * H + h
  for (size_t i = 0; i < len.size(); ++i)
    for (int h = 0; h < H; ++h) {
      t[b] += len[i];
      if (++b == grid) b = 0;
    }
  return *std::max_element(t.begin(), t.end());
}

double static_makespan(const std::vector<RunEntry>& es, int H, int sms) {
  std::vector<int> len(es.size());
  for (size_t i = 0; i < es.size(); ++i) len[i] = (es[i].te - es[i].tb + kC - 1) / kC;
  std::vector<double> t;
  return static_makespan(len, H, sms, t);
}

// Choose the segment lengths by the launches' makespans; split only when it
// beats the unsplit launch by a clear margin.  Segment 0 runs once (in pass 1,
// beside the inner segments' two runs each), every later segment also runs
// in pass 2, so segment 0 may be longer than the rest; where the block of
// segment-0 entries goes in pass 1 is chosen so that no CTA holding one gets a
// second entry.  Plans whose segment summaries need more than max_bytes of
// scratch are not considered.  (The entry lengths below follow the order of
// pass1_entries and pass2_entries.)
SplitPlan plan_split_search(const Problem& p, const int32_t* cu, int sms, size_t max_bytes) {
  SplitPlan best;
  if (!cu || p.num_seqs == 0 || p.num_seqs > kMaxScanSeqs) return best;
  const long units = (long)p.num_seqs * p.num_heads;
  if (units >= 2L * sms) return best;
  std::vector<long> cs(p.num_seqs);
  long maxc = 0, sumc = 0;
  for (int n = 0; n < p.num_seqs; ++n) {
    cs[n] = (cu[n + 1] - cu[n] + kC - 1) / kC;
    maxc = std::max(maxc, cs[n]);
    sumc += cs[n];
  }
  const double unsplit = std::max<double>(maxc, std::ceil((double)sumc * p.num_heads / sms));
  double best_cost = 0.85 * unsplit;
  static const double kFirst[] = {1.0, 1.5, 2.0, 2.5, 3.0};  // segment 0 / the rest
  std::vector<int> nat, inner, first, order, p2;
  std::vector<double> t;
  for (int target = 2; target <= 64; ++target) {
    for (double f : kFirst) {
      const long segc = (long)std::ceil((double)maxc / (f + target - 1));  // chunks per segment
      if (segc < 4) continue;
      const long seg0c = std::min<long>(maxc, (long)std::lround(f * segc));
      nat.clear();
      inner.clear();
      first.clear();
      p2.clear();
      long steps = 0, e = 0;
      for (int n = 0; n < p.num_seqs; ++n) {
        const long c = cs[n];
        const int k = c <= seg0c ? 1 : (int)(1 + (c - seg0c + segc - 1) / segc);
        e += k;
        steps = std::max<long>(steps, k - 2);
        if (k < 2) {
          p2.push_back((int)c);
          continue;
        }
        nat.push_back((int)seg0c);
        first.push_back((int)seg0c);
        for (int q = 1; q + 1 < k; ++q) {
          nat.push_back((int)segc);
          nat.push_back((int)segc);
          inner.push_back((int)segc);
          inner.push_back((int)segc);
          p2.push_back((int)segc);
        }
        p2.push_back((int)(c - seg0c - (k - 2) * segc));  // the last segment
      }
      if (e > kMaxEntries || nat.empty() || (long)nat.size() > kMaxEntries ||
          (long)p2.size() > kMaxEntries)
        continue;
      if (3 * (size_t)e * p.num_heads * kD * kD * sizeof(float) > max_bytes) continue;
      if ((long)nat.size() * p.num_heads > 4L * sms) continue;  // pass 1 in more than 4 waves
      // pass 1 in the order with the smallest makespan: natural, or the
      // segment-0 block first, last, or where its units end the first wave
      // on CTAs that get no second unit
      double ms1 = static_makespan(nat, p.num_heads, sms, t);
      int best_at = -1;
      const int n_inner = (int)inner.size();
      const long u1 = (long)nat.size() * p.num_heads, grid = std::min<long>(u1, sms);
      const int ideal = (int)std::min<long>(
          n_inner, (std::max<long>(0, u1 - grid) + p.num_heads - 1) / p.num_heads);
      for (int at : {0, n_inner, ideal}) {
        order.assign(inner.begin(), inner.begin() + at);
        order.insert(order.end(), first.begin(), first.end());
        order.insert(order.end(), inner.begin() + at, inner.end());
        const double m = static_makespan(order, p.num_heads, sms, t);
        if (m < ms1) {
          ms1 = m;
          best_at = at;
        }
      }
      std::sort(p2.begin(), p2.end(), std::greater<int>());  // pass 2 runs longest first
      const double cost = ms1 + static_makespan(p2, p.num_heads, sms, t) + (double)steps;
      if (cost < best_cost) {
        best_cost = cost;
        best.use = true;
        best.seg_len = (int)(segc * kC);
        best.seg0_len = (int)(seg0c * kC);
        best.s0_at = best_at;
        best.E = (int)e;
      }
    }
  }
  if (best.use) {
    const long segc = best.seg_len / kC, seg0c = best.seg0_len / kC;
    best.nseg.resize(p.num_seqs);
    best.base.resize(p.num_seqs);
    int b = 0;
    for (int n = 0; n < p.num_seqs; ++n) {
      best.nseg[n] = cs[n] <= seg0c ? 1 : (int)(1 + (cs[n] - seg0c + segc - 1) / segc);
      best.base[n] = b;
      b += best.nseg[n];
    }
    best.bytes = 3 * (size_t)best.E * p.num_heads * kD * kD * sizeof(float);
  }
  return best;
}

// plan_split_search for the last arguments seen on this host thread (a
// workspace query and the launch that follows ask for the same plan).
SplitPlan plan_split(const Problem& p, const int32_t* cu, int sms,
                     size_t max_bytes = ~(size_t)0) {
  thread_local std::vector<int32_t> key_cu;
  thread_local int key[3] = {-1, -1, -1};
  thread_local size_t key_bytes = 0;
  thread_local SplitPlan plan;
  if (!cu || p.num_seqs == 0 || p.num_seqs > kMaxScanSeqs) return SplitPlan{};
  const int k3[3] = {p.num_seqs, p.num_heads, sms};
  if (std::equal(k3, k3 + 3, key) && key_bytes == max_bytes &&
      key_cu.size() == (size_t)p.num_seqs + 1 && std::equal(cu, cu + p.num_seqs + 1, key_cu.begin()))
    return plan;
  plan = plan_split_search(p, cu, sms, max_bytes);
  std::copy(k3, k3 + 3, key);
  key_bytes = max_bytes;
  key_cu.assign(cu, cu + p.num_seqs + 1);
  return plan;
}

// The (sequence, head) units of an unsplit launch, longest first, each given
// to the CTA with the least work so far (chunks), written so that CTA b's
// k-th unit is list[b + k * grid] (use_order 2).  False when the schedule
// does not fit the list (the caller keeps the plain longest-first order).
bool unit_schedule(const std::vector<int>& by_len, const int32_t* cu, int H, int grid,
                   Params& prm) {
  if (grid <= 0) return false;
  std::vector<long> load(grid, 0);
  std::vector<std::vector<int>> mine(grid);
  using Slot = std::pair<long, int>;  // (chunks so far, CTA)
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> free_first;
  for (int b = 0; b < grid; ++b) free_first.push({0, b});
  for (int seq : by_len) {
    const long c = std::max<long>(1, (cu[seq + 1] - cu[seq] + kC - 1) / kC);
    for (int h = 0; h < H; ++h) {
      const Slot sl = free_first.top();
      free_first.pop();
      mine[sl.second].push_back(seq * H + h);
      free_first.push({sl.first + c, sl.second});
    }
  }
  size_t depth = 0;
  for (const auto& m : mine) depth = std::max(depth, m.size());
  if (depth * (size_t)grid > (size_t)kMaxOrder) return false;
  for (size_t k = 0; k < depth; ++k)
    for (int b = 0; b < grid; ++b)
      prm.list[k * grid + b] = k < mine[b].size() ? mine[b][k] : -1;
  prm.num_units = (int)(depth * grid);
  prm.use_order = 2;
  return true;
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

}  // namespace tcp

bool chunk_tc_supported(const Problem& p, const Args& a) {
  if (!p.io_bf16 || p.dk != 128 || p.dv != 128) return false;
  auto al = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
  return al(a.q) && al(a.k) && al(a.v) && al(a.z) && al(a.out) &&
         (!a.initial_state || al(a.initial_state)) && (!a.final_state || al(a.final_state));
}

size_t chunk_tc_workspace_bytes(const Problem& p, const int32_t* cu_host) {
  if (!p.io_bf16 || p.dk != 128 || p.dv != 128) return 0;
  const int sms = tcp::sm_count();
  if (sms <= 0) return 0;
  const tcp::SplitPlan plan = tcp::plan_split(p, cu_host, sms);
  return plan.use ? (plan.bytes + 255) / 256 * 256 : 0;
}

namespace tcp {

// What every tensor-core launch needs: the kernels' shared-memory limit set
// on this device, the TMA maps of q, k, v and z, and the common parameters.
struct TcLaunch {
  CUtensorMap mq, mk, mv, mz;
  bool per_head = false;
  int sms = 0;
  cudaStream_t st = nullptr;

  cudaError_t init(const Problem& p, const Args& a, Params& prm, cudaStream_t stream) {
    st = stream;
    per_head = a.gate_per_head != 0;
    sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    static PerDeviceInit attrs;
    const cudaError_t attr_err = attrs.run([] {
      cudaError_t e = cudaSuccess;
      const void* kernels[] = {(const void*)chunk_tc_kernel<false, false>,
                               (const void*)chunk_tc_kernel<true, false>,
                               (const void*)chunk_tc_kernel<false, true>,
                               (const void*)chunk_tc_kernel<true, true>};
      for (const void* kf : kernels)
        if (e == cudaSuccess)
          e = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)SMEM_BYTES_CONV);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(state_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kScanSmem);
      return e;
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int T = std::max(p.total_tokens, 1);
    if (!make_map(&mq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.num_heads, T, 64,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.num_heads, T, 64,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.num_heads, T, 64,
                  CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    if (per_head) {
      mz = mq;  // z is [T, H] and read directly; the z tile map is never used
    } else if (!make_map(&mz, a.z, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.num_heads, T, 128,
                         CU_TENSOR_MAP_SWIZZLE_NONE)) {
      return cudaErrorInvalidValue;
    }
    prm.beta = a.beta;
    prm.a_log = a.a_log;
    prm.ckpt = a.ckpt;
    prm.ckpt_off = a.ckpt_off;
    prm.ckpt_every = a.ckpt_every;
    prm.zh = per_head ? a.z : nullptr;
    prm.initial_state = a.initial_state;
    prm.cu = a.cu_seqlens;
    prm.out = static_cast<__nv_bfloat16*>(a.out);
    prm.final_state = a.final_state;
    prm.aux_state = nullptr;
    prm.ws = nullptr;
    prm.err = a.err;
    prm.H = p.num_heads;
    prm.total = p.total_tokens;
    prm.num_seqs = p.num_seqs;
    prm.spin_cycles = 4000000000LL;  // ~2 s at 2 GHz
    prm.inject_timeout = 0;
    if (g_inject_wait_timeout > 0) {  // testing aid, see kda_testing_inject_wait_timeout
      --g_inject_wait_timeout;
      prm.inject_timeout = 1;
      prm.spin_cycles = 20000000LL;  // ~10 ms
    }
    prm.conv_w = a.conv_w;
    prm.conv_wq = a.conv_wq;
    prm.conv_wk = a.conv_wk;
    prm.conv_sq = a.conv_sq;
    prm.conv_sk = a.conv_sk;
    prm.qraw = static_cast<const __nv_bfloat16*>(a.q);
    prm.kraw = static_cast<const __nv_bfloat16*>(a.k);
    prm.use_order = 0;
    prm.mode = 0;
    return cudaSuccess;
  }

  void launch(const Params& prm, int grid) const {
    if (prm.conv_w > 0) {
      if (per_head)
        chunk_tc_kernel<true, true><<<grid, kNT, SMEM_BYTES_CONV, st>>>(mq, mk, mv, mz, prm);
      else
        chunk_tc_kernel<false, true><<<grid, kNT, SMEM_BYTES_CONV, st>>>(mq, mk, mv, mz, prm);
    } else if (per_head) {
      chunk_tc_kernel<true, false><<<grid, kNT, SMEM_BYTES, st>>>(mq, mk, mv, mz, prm);
    } else {
      chunk_tc_kernel<false, false><<<grid, kNT, SMEM_BYTES, st>>>(mq, mk, mv, mz, prm);
    }
  }
};

}  // namespace tcp

cudaError_t launch_chunk_tc(const Problem& p, const Args& a, const int32_t* cu_host, void* ws,
                            size_t ws_bytes, cudaStream_t st) {
  using namespace tcp;
  if (p.num_seqs == 0) return cudaSuccess;
  static thread_local Params prm;  // large: keep off the stack
  TcLaunch tl;
  const cudaError_t se = tl.init(p, a, prm, st);
  if (se != cudaSuccess) return se;
  const int sms = tl.sms;
  auto launch_tc = [&](int grid) { tl.launch(prm, grid); };

  SplitPlan plan;  // the best split whose summaries fit in the workspace, if any
  if (ws && (reinterpret_cast<uintptr_t>(ws) & 255) == 0) plan = plan_split(p, cu_host, sms, ws_bytes);
  if (!plan.use) {
    prm.num_units = p.num_seqs * p.num_heads;
    if (cu_host && p.num_seqs <= kMaxOrder) {
      std::vector<int> idx(p.num_seqs);
      std::iota(idx.begin(), idx.end(), 0);
      std::stable_sort(idx.begin(), idx.end(), [&](int x, int y) {
        return cu_host[x + 1] - cu_host[x] > cu_host[y + 1] - cu_host[y];
      });
      const int grid = std::min(prm.num_units, sms);
      if (!unit_schedule(idx, cu_host, p.num_heads, grid, prm)) {
        for (int i = 0; i < p.num_seqs; ++i) prm.list[i] = idx[i];
        prm.use_order = 1;
      }
    }
    launch_tc(std::min(prm.num_units, sms));
    return cudaGetLastError();
  }

  // ---- split: pass 1 (inner segments' S~ and M, segment 0 from the true state) ----
  const int E = plan.E;
  prm.ws = static_cast<float*>(ws);
  prm.mode = 1;
  int ne = 0;
  auto put = [&](const RunEntry& r) {
    int* e = prm.list + kEnt * ne++;
    e[0] = r.n; e[1] = r.tb; e[2] = r.te; e[3] = r.in; e[4] = r.out; e[5] = r.flags;
  };
  for (const RunEntry& r : pass1_entries(plan, cu_host, p.num_seqs)) put(r);
  // segment 0 runs from the true initial state, so it writes its outputs and
  // checkpoints here; the inner segments' runs from stand-in states do not
  prm.out = static_cast<__nv_bfloat16*>(a.out);
  prm.ckpt = a.ckpt;
  if (ne > 0) {
    prm.num_units = ne * p.num_heads;
    launch_tc(std::min(prm.num_units, sms));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // ---- scan ----
  {
    static thread_local ScanParams sp;
    sp.initial_state = a.initial_state;
    sp.ws = static_cast<float*>(ws);
    sp.H = p.num_heads;
    sp.E = E;
    for (int n = 0; n < p.num_seqs; ++n) sp.s[n] = ScanSeq{n, plan.base[n], plan.nseg[n]};
    state_scan_kernel<<<p.num_seqs * p.num_heads, kScanThreads, kScanSmem, st>>>(sp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // ---- pass 2: every other segment from its entry state, longest first ----
  ne = 0;
  for (const RunEntry& r : pass2_entries(plan, cu_host, p.num_seqs)) put(r);
  prm.out = static_cast<__nv_bfloat16*>(a.out);
  prm.ckpt = a.ckpt;
  prm.num_units = ne * p.num_heads;
  launch_tc(std::min(prm.num_units, sms));
  return cudaGetLastError();
}

// ------------------------------------------------- affine summaries --------
//
// The summary (M, S~) of a sequence is the final state of two runs of the
// same kernel: from zeros (S~) and from the identity with v = 0 (M; its
// "value" axis is the identity's column).  When there are fewer than one
// such run per SM, each sequence is cut into k segments whose summaries run
// side by side and are then composed in order,
//   S~ = M_{k-1}(... (M_1 S~_0 + S~_1) ...) + S~_{k-1},   M = M_{k-1} ... M_0.

namespace tcp {

struct SummaryPlan {
  bool use = false;
  int seg_len = 0, E = 0;       // segment length (tokens); slots per summary part
  std::vector<int> k, base;     // segments per sequence; first slot of a split sequence
  size_t bytes = 0;
};

SummaryPlan plan_summary(const Problem& p, const int32_t* cu, int sms,
                         size_t max_bytes = ~(size_t)0) {
  SummaryPlan best;
  if (!cu || p.num_seqs == 0) return best;
  const long runs = 2L * p.num_seqs * p.num_heads;
  if (runs >= sms) return best;
  long maxc = 0;
  for (int n = 0; n < p.num_seqs; ++n) maxc = std::max<long>(maxc, (cu[n + 1] - cu[n] + kC - 1) / kC);
  for (long kmax = sms / runs; kmax >= 2; --kmax) {
    const long segc = std::max<long>(4, (maxc + kmax - 1) / kmax);
    if (segc >= maxc) break;  // nothing would split
    SummaryPlan pl;
    pl.k.resize(p.num_seqs);
    pl.base.resize(p.num_seqs);
    for (int n = 0; n < p.num_seqs; ++n) {
      const long c = (cu[n + 1] - cu[n] + kC - 1) / kC;
      pl.k[n] = (int)std::max<long>(1, (c + segc - 1) / segc);
      pl.base[n] = pl.E;
      if (pl.k[n] >= 2) pl.E += pl.k[n];
    }
    pl.bytes = 2 * (size_t)pl.E * p.num_heads * kD * kD * sizeof(float);
    if (pl.bytes > max_bytes) continue;
    pl.use = true;
    pl.seg_len = (int)(segc * kC);
    return pl;
  }
  return best;
}

}  // namespace tcp

size_t chunk_tc_summary_workspace_bytes(const Problem& p, const int32_t* cu_host) {
  if (!p.io_bf16 || p.dk != 128 || p.dv != 128) return 0;
  const int sms = tcp::sm_count();
  if (sms <= 0) return 0;
  const tcp::SummaryPlan plan = tcp::plan_summary(p, cu_host, sms);
  return plan.use ? (plan.bytes + 255) / 256 * 256 : 0;
}

cudaError_t launch_chunk_tc_summary(const Problem& p, const Args& a, const int32_t* cu_host,
                                    float* m_out, void* ws, size_t ws_bytes, cudaStream_t st) {
  using namespace tcp;
  if (p.num_seqs == 0) return cudaSuccess;
  static thread_local Params prm;  // large: keep off the stack
  TcLaunch tl;
  cudaError_t e = tl.init(p, a, prm, st);
  if (e != cudaSuccess) return e;
  SummaryPlan plan;
  if (ws && (reinterpret_cast<uintptr_t>(ws) & 255) == 0)
    plan = plan_summary(p, cu_host, tl.sms, ws_bytes);
  prm.mode = 1;
  prm.out = nullptr;
  prm.ckpt = nullptr;
  prm.final_state = a.final_state;  // S~ of unsplit sequences
  prm.aux_state = m_out;            // M of unsplit sequences
  prm.ws = static_cast<float*>(ws);
  const int E = plan.use ? plan.E : 0;
  // every run, longest first: {length, seq, tb, te, in, out, flags}
  std::vector<std::array<int, 7>> runs;
  for (int n = 0; n < p.num_seqs; ++n) {
    const int k = plan.use ? plan.k[n] : 1;
    for (int q = 0; q < k; ++q) {
      const int tb = k == 1 ? cu_host[n] : cu_host[n] + q * plan.seg_len;
      const int te = k == 1 ? cu_host[n + 1] : std::min(cu_host[n + 1], tb + plan.seg_len);
      const int s_slot = k == 1 ? kSlotUser : plan.base[n] + q;
      const int m_slot = k == 1 ? kSlotAux : E + plan.base[n] + q;
      runs.push_back({te - tb, n, tb, te, kSlotZero, s_slot, 0});
      runs.push_back({te - tb, n, tb, te, kSlotIdentity, m_slot, kFlagZeroV});
    }
  }
  std::stable_sort(runs.begin(), runs.end(),
                   [](const std::array<int, 7>& x, const std::array<int, 7>& y) { return x[0] > y[0]; });
  for (size_t r0 = 0; r0 < runs.size(); r0 += kMaxEntries) {
    const int ne = (int)std::min<size_t>(kMaxEntries, runs.size() - r0);
    for (int i = 0; i < ne; ++i) {
      const auto& r = runs[r0 + i];
      int* en = prm.list + kEnt * i;
      en[0] = r[1]; en[1] = r[2]; en[2] = r[3]; en[3] = r[4]; en[4] = r[5]; en[5] = r[6];
    }
    prm.num_units = ne * p.num_heads;
    tl.launch(prm, std::min(prm.num_units, tl.sms));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (!plan.use) return cudaSuccess;
  // compose the segments of every split sequence
  std::vector<FoldEntry> fs, fm;
  for (int n = 0; n < p.num_seqs; ++n) {
    const int k = plan.k[n], b = plan.base[n];
    if (k < 2) continue;
    fs.push_back(FoldEntry{b, E + b + 1, b + 1, n, k - 1});
    fm.push_back(FoldEntry{E + b, E + b + 1, 0, n, k - 1});
  }
  const float* w = static_cast<const float*>(ws);
  e = launch_state_fold(kD, kD, p.num_heads, w, w, w, a.final_state, 1, fs.data(),
                        (int)fs.size(), st);
  if (e != cudaSuccess) return e;
  return launch_state_fold(kD, kD, p.num_heads, w, w, nullptr, m_out, 1, fm.data(),
                           (int)fm.size(), st);
}

}  // namespace kda

extern "C" void kda_testing_inject_wait_timeout(int launches) {
  kda::tcp::g_inject_wait_timeout = launches > 0 ? launches : 0;
}
