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
// e^{G_t - G_j} span e^{+-320} across a 64-token chunk, beyond fp32/bf16, so
// the pairwise (Gram) products use one reference per 16-token subtile: with
// r_a the cumulative log-decay before subtile a, Q~ = q^ e^{G - r_a} <= 1,
// K~ = k^ e^{r_a - G} <= e^80 and D_ab = e^{r_a - r_b}, a block (a, b) of P
// is (Q~_a D_ab) K~_b^T.  The e^80 bound is what the lower-bounded gate buys
// (blog.higcp.com "猜想：K3 可能是最适合 TPU 的 MoE 架构", section "下界衰减":
// log alpha >= -5, so a 16-token tile decays by less than e^-80 and its
// reciprocal stays finite), and it lets the diagonal blocks go through the
// tensor cores like the others.
//
// Everything else is kept in the transposed orientation so that every
// tcgen05 GEMM has M = 128 and the state and U can feed the tensor core
// straight from Tensor Memory:
//   W^T = K+^T T'^T,  U~^T = V^T T'^T,  U^T = U~^T - S^T W^T,
//   O^T = S^T Q+^T + U^T P^T,  S^T <- S^T Diag(e^{G_C}) + U^T Khat.
// S^T (fp32, 128 lanes = value channel) stays resident in TMEM across
// chunks; its fp16 copy and U^T's are A operands read from TMEM.
//
// Precision: the Gram products run as tf32 warp MMAs on fp32 operands (the
// e^80 range rules out fp16 there); the dense products use fp16 operands
// (11-bit significand; all of them are bounded by 1 or by the data) with
// fp32 accumulation.  bf16 operands there would leave ~0.2% relative error
// on the largest outputs.
//
// One CTA (4 warps) per SM walks (sequence, head) work units, longest
// sequence first.  Per chunk:
//   TMA   q, k, v (bf16, 128B swizzle) and z (fp32) tiles into shared memory;
//   CUDA  gate g = -5 sigmoid(z), per-channel cumulative sums, L2 norms, and
//         the decayed operands written in tensor-core layouts;
//   mma.sync (tf32)  the ten 16x16 Gram blocks of P and A;
//   CUDA  T = (I + A)^{-1} by block forward substitution (fp32);
//   tcgen05   the five dense products above, accumulators in TMEM.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>
#include <numeric>
#include <vector>

#include "kda_common.cuh"
#include "kda_launch.h"
#include "tc_ptx.cuh"

namespace kda {
namespace tcp {

using namespace kda::tc;

constexpr int kC = 64;     // chunk length
constexpr int kD = 128;    // dk = dv
constexpr int kNT = 128;   // threads per CTA
constexpr int kMaxOrder = 6144;

// ---- shared memory map (offsets from a 1024-byte aligned base) ----
constexpr uint32_t OFF_Q = 0;         // q stage: [2 c-blk][64 t][64 c] bf16, SW128 (TMA)
constexpr uint32_t OFF_K = 16384;     // k stage, same
constexpr uint32_t OFF_Z = 32768;     // z stage: [64 t][128 c] fp32 (TMA); then G in place
constexpr uint32_t OFF_V = 65536;     // v stage: [2 n-blk][64 j][64 n] SW128; fp16 in place = MN-major A
constexpr uint32_t OFF_G = 81920;     // 80K: Gram operands, later A / T / P / T' / W^T
constexpr uint32_t G_QT = OFF_G;              // Q~  fp32 [64 t][128 c] (xor-swizzled)
constexpr uint32_t G_KT = OFF_G + 32768;      // K~  fp32 [64 j][128 c] (xor-swizzled)
constexpr uint32_t G_KPT = OFF_G + 65536;     // K~+ bf16 [64 t][128 c] (xor-swizzled)
constexpr uint32_t G_AKK = OFF_G;             // A   fp32 [64][64]          (after the Gram)
constexpr uint32_t G_T32 = OFF_G + 16384;     // T   fp32 [64][64]
constexpr uint32_t G_P = OFF_G + 32768;       // P   fp16 [64 t][64 j] SW128: K-major B
constexpr uint32_t G_TP = OFF_G + 40960;      // T'  fp16 [64 t][64 j] SW128: K-major B
constexpr uint32_t G_WT = OFF_G + 49152;      // W^T fp16 [128 c][64 t] SW128: MN-major B
constexpr uint32_t OFF_QPT = 163840;  // Q+^T  fp16 [128 c][64 t] SW128: MN-major B
constexpr uint32_t OFF_KPT = 180224;  // K+^T  fp16 [128 c][64 j] SW128: K-major A
constexpr uint32_t OFF_KH = 196608;   // Khat^T fp16 [128 c][64 t] SW128: K-major B
constexpr uint32_t OFF_MISC = 212992;
// misc floats
constexpr int M_BETA = 0, M_RQ = 64, M_RK = 128, M_DECAY = 192, M_ER = 320, M_EGR = 832,
              M_DAB = 1344, M_END = 1344 + 6 * 128;
constexpr uint32_t OFF_BAR = OFF_MISC + M_END * 4;  // 3 mbarriers + tmem slot
constexpr uint32_t SMEM_BYTES = OFF_BAR + 64 + 1024;  // + alignment slack

// ---- Tensor Memory columns (all 128 lanes) ----
constexpr uint32_t TS32 = 0;    // S^T fp32   [n][c]   128 cols
constexpr uint32_t TS16 = 128;  // S^T fp16   [n][c/2]  64 cols (A operand)
constexpr uint32_t TW = 192;    // W^T fp32   [c][t]    64 cols
constexpr uint32_t TU = 256;    // U~^T / U^T [n][t]    64 cols
constexpr uint32_t TU16 = 320;  // U^T fp16   [n][t/2]  32 cols (A operand)
constexpr uint32_t TO = 384;    // O^T fp32   [n][t]    64 cols

// largest magnitude an fp16 operand may take
constexpr float kF16Max = 65504.0f;

struct Params {
  const float* beta;
  const float* initial_state;
  const int32_t* cu;
  __nv_bfloat16* out;
  float* final_state;
  int* err;
  int H, total, num_seqs, num_units, use_order;
  long long spin_cycles;
  int order[kMaxOrder];
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, long long limit) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// fp32 element (t, c) of a [64][128] tile, 32-bit word index xor (row % 8) * 4
__device__ __forceinline__ uint32_t f32_off(int t, int c) {
  return (uint32_t)t * 512u + ((uint32_t)(c ^ ((t & 7) << 2)) << 2);
}
// bf16 element (t, c) of a [64][128] tile, element index xor (row % 8) * 8
__device__ __forceinline__ uint32_t b16_off(int t, int c) {
  return (uint32_t)t * 256u + ((uint32_t)(c ^ ((t & 7) << 3)) << 1);
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

__device__ __forceinline__ void sync_tc() {
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

// Gram blocks (query subtile a, key subtile b), a >= b, and zero blocks a < b.
__constant__ int8_t c_blk_a[10] = {0, 1, 1, 2, 2, 2, 3, 3, 3, 3};
__constant__ int8_t c_blk_b[10] = {0, 0, 1, 0, 1, 2, 0, 1, 2, 3};
__constant__ int8_t c_zero_a[6] = {0, 0, 0, 1, 1, 2};
__constant__ int8_t c_zero_b[6] = {1, 2, 3, 2, 3, 3};

__device__ __forceinline__ int dab_index(int a, int b) {  // a > b
  return a == 1 ? 0 : (a == 2 ? 1 + b : 3 + b);
}

__device__ __forceinline__ bool f16_ok(float x) { return fabsf(x) < kF16Max; }

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
    mbar_fence_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_z);
  }
  sync_tc();
  const uint32_t tmem = *s_tmem;
  // this thread's TMEM lane (row): warp w owns lanes 32w .. 32w+31
  const uint32_t my_lane = tmem + ((uint32_t)(warp * 32) << 16);
  uint32_t ph_qkz = 0, ph_v = 0, ph_mma = 0;
  bool pend_qkz = false, pend_v = false;  // TMA copies in flight (uniform)
  bool aborted = false;
  bool range_ok = true;  // fp16 operand range held (this thread)

  for (int u = blockIdx.x; u < P.num_units && !aborted; u += gridDim.x) {
    const int si = u / H, h = u % H;
    const int seq = P.use_order ? P.order[si] : si;
    const int bos = P.cu[seq], eos = P.cu[seq + 1];
    if (bos < 0 || eos < bos || eos > P.total) {
      if (tid == 0) report_error(P.err, kErrDeviceCheck);
      continue;
    }
    const int nchunks = (eos - bos + kC - 1) / kC;
    if (tid == 0 && nchunks > 0) {
      mbar_arrive_expect_tx(bar_qkz, 65536u);
      tma_load_3d(sm + OFF_Q, &tm_q, 0, h, bos, bar_qkz);
      tma_load_3d(sm + OFF_Q + 8192, &tm_q, 64, h, bos, bar_qkz);
      tma_load_3d(sm + OFF_K, &tm_k, 0, h, bos, bar_qkz);
      tma_load_3d(sm + OFF_K + 8192, &tm_k, 64, h, bos, bar_qkz);
      tma_load_3d(sm + OFF_Z, &tm_z, 0, h, bos, bar_qkz);
      mbar_arrive_expect_tx(bar_v, 16384u);
      tma_load_3d(sm + OFF_V, &tm_v, 0, h, bos, bar_v);
      tma_load_3d(sm + OFF_V + 8192, &tm_v, 64, h, bos, bar_v);
    }
    pend_qkz = pend_v = nchunks > 0;

    // ---- entry state S^T: lane n holds column n of S (fp32 and fp16) ----
    {
      const int n = tid;
      const float* src = P.initial_state ? P.initial_state + ((size_t)seq * H + h) * kD * kD + n
                                         : nullptr;
#pragma unroll 1
      for (int c0 = 0; c0 < kD; c0 += 16) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = src ? __ldg(src + (size_t)(c0 + i) * kD) : 0.f;
        tmem_st16(my_lane + TS32 + c0, v);
        uint32_t hp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          hp[i] = pack_f16(v[2 * i], v[2 * i + 1]);
          range_ok &= f16_ok(v[2 * i]) & f16_ok(v[2 * i + 1]);
        }
        tmem_st8(my_lane + TS16 + (c0 >> 1), hp);
      }
      tmem_st_wait();
    }
    sync_tc();

    for (int ci = 0; ci < nchunks; ++ci) {
      const int t0 = bos + ci * kC;
      const int len = min(kC, eos - t0);
      // ---------------- A: inputs ----------------
      bool ok = wait_bar(bar_qkz, ph_qkz, P.spin_cycles);
      ph_qkz ^= 1;
      pend_qkz = false;
      if (__syncthreads_or(!ok)) { aborted = true; break; }

      // ---------------- B: token norms and beta ----------------
      {
        const int t = tid >> 1, hh = tid & 1;
        const unsigned char* qrow = sm + OFF_Q + hh * 8192 + t * 128;
        const unsigned char* krow = sm + OFF_K + hh * 8192 + t * 128;
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 a = *reinterpret_cast<const uint4*>(qrow + (j << 4));
          const uint4 b = *reinterpret_cast<const uint4*>(krow + (j << 4));
          const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float x = bf16_lo(aw[i]), y = bf16_hi(aw[i]);
            sq += x * x + y * y;
            x = bf16_lo(bw[i]); y = bf16_hi(bw[i]);
            sk += x * x + y * y;
          }
        }
        sq += __shfl_xor_sync(0xffffffffu, sq, 1);
        sk += __shfl_xor_sync(0xffffffffu, sk, 1);
        if (hh == 0) {
          misc[M_RQ + t] = t < len ? rsqrtf(sq + kNormEps) : 0.f;
          misc[M_RK + t] = t < len ? rsqrtf(sk + kNormEps) : 0.f;
        }
        if (tid < kC) misc[M_BETA + tid] = tid < len ? __ldg(P.beta + (size_t)(t0 + tid) * H + h) : 0.f;
      }
      __syncthreads();

      // ---------------- C: gate, cumulative decay, per-channel tables ----------------
      const int c = tid;
      float r[4];
      float* Z = reinterpret_cast<float*>(sm + OFF_Z);
      {
        float G = 0.f;
        r[0] = 0.f;
#pragma unroll
        for (int t = 0; t < kC; ++t) {
          if ((t & 15) == 0 && t > 0) r[t >> 4] = G;
          const float g = t < len ? log_decay(Z[t * kD + c]) : 0.f;
          G += g;
          Z[t * kD + c] = G;
        }
        misc[M_DECAY + c] = __expf(G);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          misc[M_ER + a * kD + c] = __expf(r[a]);
          misc[M_EGR + a * kD + c] = __expf(G - r[a]);
        }
        misc[M_DAB + 0 * kD + c] = __expf(r[1] - r[0]);
        misc[M_DAB + 1 * kD + c] = __expf(r[2] - r[0]);
        misc[M_DAB + 2 * kD + c] = __expf(r[2] - r[1]);
        misc[M_DAB + 3 * kD + c] = __expf(r[3] - r[0]);
        misc[M_DAB + 4 * kD + c] = __expf(r[3] - r[1]);
        misc[M_DAB + 5 * kD + c] = __expf(r[3] - r[2]);
      }

      // ---------------- D: decayed operands (thread = key channel c) ----------------
      {
        const float* er = misc + M_ER;
        const float* egr = misc + M_EGR;
        const unsigned char* qs = sm + OFF_Q;
        const unsigned char* ks = sm + OFF_K;
        const uint32_t sw = (uint32_t)(c & 7);
#pragma unroll
        for (int t8 = 0; t8 < kC; t8 += 8) {
          uint32_t qp_pack[4], kp_pack[4], kh_pack[4];
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            float qpv[2], kpv[2], khv[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int t = t8 + i + e, a = t >> 4;
              const float Gt = Z[t * kD + c];
              const float F = __expf(Gt - r[a]);
              const float E = __fdividef(1.0f, F);
              const uint32_t off = (uint32_t)(c >> 6) * 8192u + sw128_offset(t, c & 63);
              const float qh = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(qs + off)) * misc[M_RQ + t];
              const float kh = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(ks + off)) * misc[M_RK + t];
              const float qt = qh * F, kpt = kh * F, kt = kh * E;
              *reinterpret_cast<float*>(sm + G_QT + f32_off(t, c)) = qt;
              *reinterpret_cast<float*>(sm + G_KT + f32_off(t, c)) = kt;
              *reinterpret_cast<__nv_bfloat16*>(sm + G_KPT + b16_off(t, c)) = __float2bfloat16_rn(kpt);
              qpv[e] = qt * er[a * kD + c];
              kpv[e] = kpt * er[a * kD + c];
              khv[e] = kt * egr[a * kD + c];
            }
            qp_pack[i >> 1] = pack_f16(qpv[0], qpv[1]);
            kp_pack[i >> 1] = pack_f16(kpv[0], kpv[1]);
            kh_pack[i >> 1] = pack_f16(khv[0], khv[1]);
          }
          const uint32_t chunk_off = (uint32_t)c * 128u + ((((uint32_t)t8 >> 3) ^ sw) << 4);
          *reinterpret_cast<uint4*>(sm + OFF_QPT + chunk_off) =
              make_uint4(qp_pack[0], qp_pack[1], qp_pack[2], qp_pack[3]);
          *reinterpret_cast<uint4*>(sm + OFF_KPT + chunk_off) =
              make_uint4(kp_pack[0], kp_pack[1], kp_pack[2], kp_pack[3]);
          *reinterpret_cast<uint4*>(sm + OFF_KH + chunk_off) =
              make_uint4(kh_pack[0], kh_pack[1], kh_pack[2], kh_pack[3]);
        }
      }
      fence_proxy_async_smem();
      sync_tc();
      if (tid == 0) {
        // q/k/z stage consumed: prefetch the next chunk
        if (ci + 1 < nchunks) {
          const int tn = t0 + kC;
          mbar_arrive_expect_tx(bar_qkz, 65536u);
          tma_load_3d(sm + OFF_Q, &tm_q, 0, h, tn, bar_qkz);
          tma_load_3d(sm + OFF_Q + 8192, &tm_q, 64, h, tn, bar_qkz);
          tma_load_3d(sm + OFF_K, &tm_k, 0, h, tn, bar_qkz);
          tma_load_3d(sm + OFF_K + 8192, &tm_k, 64, h, tn, bar_qkz);
          tma_load_3d(sm + OFF_Z, &tm_z, 0, h, tn, bar_qkz);
        }
        // O^T = S^T Q+^T  (M=128 value channels, N=64 tokens, K=128 key channels)
        const uint32_t id_o = make_idesc_f16(128, kC, false, true);
        const uint32_t bq = smem_u32(sm + OFF_QPT);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_ts(tmem + TO, tmem + TS16 + kk * 8,
                 make_sdesc(bq + kk * 2048, 8192, 1024, kSwizzle128), id_o, kk > 0);
      }
      pend_qkz = (ci + 1 < nchunks);

      // ---------------- E: Gram blocks, tf32 mma.sync ----------------
      float accP[3][2][4], accA[3][2][4];
      {
        const int g = lane >> 2, q4 = lane & 3;
        const float* Qt = reinterpret_cast<const float*>(sm + G_QT);
        const float* Kt = reinterpret_cast<const float*>(sm + G_KT);
        const unsigned char* Kpt = sm + G_KPT;
#pragma unroll
        for (int bi = 0; bi < 3; ++bi) {
#pragma unroll
          for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) accP[bi][n][i] = accA[bi][n][i] = 0.f;
          const int blk = warp + 4 * bi;
          if (blk >= 10) continue;
          const int a = c_blk_a[blk], b = c_blk_b[blk];
          const float* dab = misc + M_DAB + (a > b ? dab_index(a, b) : 0) * kD;
          const int ta = 16 * a + g, jb = 16 * b + g;
#pragma unroll 4
          for (int c0 = 0; c0 < kD; c0 += 8) {
            const int ca = c0 + q4, cb = c0 + q4 + 4;
            float s0 = 1.f, s1 = 1.f;
            if (a != b) { s0 = dab[ca]; s1 = dab[cb]; }
            uint32_t fq[4], fk[4];
            fq[0] = to_tf32(Qt[f32_off(ta, ca) >> 2] * s0);
            fq[1] = to_tf32(Qt[f32_off(ta + 8, ca) >> 2] * s0);
            fq[2] = to_tf32(Qt[f32_off(ta, cb) >> 2] * s1);
            fq[3] = to_tf32(Qt[f32_off(ta + 8, cb) >> 2] * s1);
            const float k0 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(Kpt + b16_off(ta, ca)));
            const float k1 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(Kpt + b16_off(ta + 8, ca)));
            const float k2 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(Kpt + b16_off(ta, cb)));
            const float k3 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(Kpt + b16_off(ta + 8, cb)));
            fk[0] = to_tf32(k0 * s0);
            fk[1] = to_tf32(k1 * s0);
            fk[2] = to_tf32(k2 * s1);
            fk[3] = to_tf32(k3 * s1);
            const uint32_t b00 = to_tf32(Kt[f32_off(jb, ca) >> 2]);
            const uint32_t b01 = to_tf32(Kt[f32_off(jb, cb) >> 2]);
            const uint32_t b10 = to_tf32(Kt[f32_off(jb + 8, ca) >> 2]);
            const uint32_t b11 = to_tf32(Kt[f32_off(jb + 8, cb) >> 2]);
            mma_1688_tf32(accP[bi][0], fq, b00, b01);
            mma_1688_tf32(accP[bi][1], fq, b10, b11);
            mma_1688_tf32(accA[bi][0], fk, b00, b01);
            mma_1688_tf32(accA[bi][1], fk, b10, b11);
          }
        }
      }
      __syncthreads();  // Gram operands no longer read
      {
        const int g = lane >> 2, q4 = lane & 3;
        float* Akk = reinterpret_cast<float*>(sm + G_AKK);
        unsigned char* Pm = sm + G_P;
#pragma unroll
        for (int bi = 0; bi < 3; ++bi) {
          const int blk = warp + 4 * bi;
          if (blk >= 10) continue;
          const int a = c_blk_a[blk], b = c_blk_b[blk];
#pragma unroll
          for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
              const int t = 16 * a + g + 8 * hr, j = 16 * b + 8 * n + 2 * q4;
              const float p0 = j <= t ? accP[bi][n][2 * hr] : 0.f;
              const float p1 = j + 1 <= t ? accP[bi][n][2 * hr + 1] : 0.f;
              *reinterpret_cast<uint32_t*>(Pm + sw128_offset(t, j)) = pack_f16(p0, p1);
              const float bt = misc[M_BETA + t];
              Akk[t * kC + j] = j < t ? bt * accA[bi][n][2 * hr] : 0.f;
              Akk[t * kC + j + 1] = j + 1 < t ? bt * accA[bi][n][2 * hr + 1] : 0.f;
            }
        }
        for (int zb = warp; zb < 6; zb += 4) {
          const int a = c_zero_a[zb], b = c_zero_b[zb];
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            const int e = lane * 8 + i, t = 16 * a + (e >> 4), j = 16 * b + (e & 15);
            *reinterpret_cast<uint32_t*>(Pm + sw128_offset(t, j)) = 0u;
            Akk[t * kC + j] = 0.f;
            Akk[t * kC + j + 1] = 0.f;
          }
        }
      }
      __syncthreads();

      // ---------------- F: T = (I + A)^{-1}, T' = T diag(beta); V -> fp16 ----------------
      {
        const float* Akk = reinterpret_cast<const float*>(sm + G_AKK);
        float* T = reinterpret_cast<float*>(sm + G_T32);
        if (lane < 16) {  // diagonal block `warp`, column `lane`, forward substitution
          const int base = 16 * warp, cc = lane;
          float x[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float s = (i == cc) ? 1.f : 0.f;
#pragma unroll
            for (int j = 0; j < i; ++j) s -= Akk[(base + i) * kC + base + j] * x[j];
            x[i] = s;
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) T[(base + i) * kC + base + cc] = x[i];
        }
        __syncthreads();
#pragma unroll 1
        for (int d = 1; d < 4; ++d) {
          const int nelem = (4 - d) * 256;
          // Y_ab = sum_{j in blocks b..a-1} A[a rows][j] T[j][b cols], kept in block (b, a)
          for (int e = tid; e < nelem; e += kNT) {
            const int b = e >> 8, a = b + d, rr = (e >> 4) & 15, cc = e & 15;
            float y = 0.f;
            for (int j = 16 * b; j < 16 * a; ++j) y += Akk[(16 * a + rr) * kC + j] * T[j * kC + 16 * b + cc];
            T[(16 * b + rr) * kC + 16 * a + cc] = y;
          }
          __syncthreads();
          // T_ab = -T_aa Y_ab
          for (int e = tid; e < nelem; e += kNT) {
            const int b = e >> 8, a = b + d, rr = (e >> 4) & 15, cc = e & 15;
            float s = 0.f;
            for (int m = 0; m <= rr; ++m)
              s -= T[(16 * a + rr) * kC + 16 * a + m] * T[(16 * b + m) * kC + 16 * a + cc];
            T[(16 * a + rr) * kC + 16 * b + cc] = s;
          }
          __syncthreads();
        }
        // T' (fp16, [t][j] rows) = T diag(beta), zero above the block diagonal
        {
          const int t = tid >> 1, j0 = (tid & 1) * 32;
#pragma unroll
          for (int jj = 0; jj < 32; jj += 16) {
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int j = j0 + jj + i;
              v[i] = ((j >> 4) <= (t >> 4)) ? T[t * kC + j] * misc[M_BETA + j] : 0.f;
            }
            st_row16_f16(sm + G_TP, t, j0 + jj, v);
          }
        }
      }
      ok = wait_bar(bar_v, ph_v, P.spin_cycles);
      ph_v ^= 1;
      pend_v = false;
      if (__syncthreads_or(!ok)) { aborted = true; break; }
      {  // v stage bf16 -> fp16 in place (same layout: the MN-major A operand of U~^T)
        uint4* vv = reinterpret_cast<uint4*>(sm + OFF_V) + tid * 8;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint4 x = vv[i];
          uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float lo = bf16_lo(w[j]), hi = bf16_hi(w[j]);
            range_ok &= f16_ok(lo) & f16_ok(hi);
            w[j] = pack_f16(lo, hi);
          }
          vv[i] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async_smem();
      sync_tc();

      // ---------------- G: W^T = K+^T T'^T,  U~^T = V^T T'^T ----------------
      if (tid == 0) {
        const uint32_t ak = smem_u32(sm + OFF_KPT), av = smem_u32(sm + OFF_V),
                       bt = smem_u32(sm + G_TP);
        const uint32_t id_w = make_idesc_f16(128, kC, false, false);
        const uint32_t id_u = make_idesc_f16(128, kC, true, false);
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk) {
          const uint64_t bd = make_sdesc(bt + kk * 32, 0, 1024, kSwizzle128);
          mma_bf16_ss(tmem + TW, make_sdesc(ak + kk * 32, 0, 1024, kSwizzle128), bd, id_w, kk > 0);
          mma_bf16_ss(tmem + TU, make_sdesc(av + kk * 2048, 8192, 1024, kSwizzle128), bd, id_u,
                      kk > 0);
        }
        mma_commit(bar_mma);
      }
      ok = wait_bar(bar_mma, ph_mma, P.spin_cycles);
      ph_mma ^= 1;
      if (__syncthreads_or(!ok)) { aborted = true; break; }
      tc_fence_after();
      if (tid == 0 && ci + 1 < nchunks) {  // v stage consumed
        const int tn = t0 + kC;
        mbar_arrive_expect_tx(bar_v, 16384u);
        tma_load_3d(sm + OFF_V, &tm_v, 0, h, tn, bar_v);
        tma_load_3d(sm + OFF_V + 8192, &tm_v, 64, h, tn, bar_v);
      }
      pend_v = (ci + 1 < nchunks);

      // ---------------- H: W^T -> fp16 (MN-major B, row c) ----------------
#pragma unroll
      for (int col = 0; col < kC; col += 16) {
        float v[16];
        tmem_ld16(my_lane + TW + col, v);
        tmem_ld_wait();
        st_row16_f16(sm + G_WT, tid, col, v);
      }
      fence_proxy_async_smem();
      sync_tc();

      // ---------------- I: U^T = U~^T - S^T W^T ----------------
      if (tid == 0) {
        const uint32_t bw = smem_u32(sm + G_WT);
        const uint32_t idn = make_idesc_f16(128, kC, false, true, true);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_ts(tmem + TU, tmem + TS16 + kk * 8,
                 make_sdesc(bw + kk * 2048, 8192, 1024, kSwizzle128), idn, true);
        mma_commit(bar_mma);
      }
      ok = wait_bar(bar_mma, ph_mma, P.spin_cycles);
      ph_mma ^= 1;
      if (__syncthreads_or(!ok)) { aborted = true; break; }
      tc_fence_after();

      // ---------------- J: U^T -> fp16 in TMEM; S^T <- S^T Diag(e^{G_C}) ----------------
      {
#pragma unroll
        for (int col = 0; col < kC; col += 16) {
          float v[16];
          tmem_ld16(my_lane + TU + col, v);
          tmem_ld_wait();
          uint32_t hp[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            hp[i] = pack_f16(v[2 * i], v[2 * i + 1]);
            range_ok &= f16_ok(v[2 * i]) & f16_ok(v[2 * i + 1]);
          }
          tmem_st8(my_lane + TU16 + (col >> 1), hp);
        }
        const float* dec = misc + M_DECAY;
#pragma unroll 1
        for (int col = 0; col < kD; col += 16) {
          float v[16];
          tmem_ld16(my_lane + TS32 + col, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] *= dec[col + i];
          tmem_st16(my_lane + TS32 + col, v);
        }
        tmem_st_wait();
      }
      sync_tc();

      // ---------------- K: O^T += U^T P^T;  S^T += U^T Khat ----------------
      if (tid == 0) {
        const uint32_t bp = smem_u32(sm + G_P), bk = smem_u32(sm + OFF_KH);
        const uint32_t id_o = make_idesc_f16(128, kC, false, false);
        const uint32_t id_s = make_idesc_f16(128, kD, false, false);
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk) {
          const uint32_t au = tmem + TU16 + kk * 8;
          mma_ts(tmem + TO, au, make_sdesc(bp + kk * 32, 0, 1024, kSwizzle128), id_o, true);
          mma_ts(tmem + TS32, au, make_sdesc(bk + kk * 32, 0, 1024, kSwizzle128), id_s, true);
        }
        mma_commit(bar_mma);
      }
      ok = wait_bar(bar_mma, ph_mma, P.spin_cycles);
      ph_mma ^= 1;
      if (__syncthreads_or(!ok)) { aborted = true; break; }
      tc_fence_after();

      // ---------------- L: write O; S^T -> fp16 for the next chunk ----------------
      {
        __nv_bfloat16* ocol = P.out + ((size_t)t0 * H + h) * kD + tid;
#pragma unroll
        for (int col = 0; col < kC; col += 16) {
          float v[16];
          tmem_ld16(my_lane + TO + col, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (col + i < len) ocol[(size_t)(col + i) * H * kD] = __float2bfloat16_rn(v[i]);
        }
#pragma unroll 1
        for (int c0 = 0; c0 < kD; c0 += 16) {
          float v[16];
          tmem_ld16(my_lane + TS32 + c0, v);
          tmem_ld_wait();
          uint32_t hp[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            hp[i] = pack_f16(v[2 * i], v[2 * i + 1]);
            range_ok &= f16_ok(v[2 * i]) & f16_ok(v[2 * i + 1]);
          }
          tmem_st8(my_lane + TS16 + (c0 >> 1), hp);
        }
        tmem_st_wait();
      }
      sync_tc();
    }
    if (aborted) break;

    // ---- final state: lane n holds column n ----
    if (P.final_state) {
      float* dst = P.final_state + ((size_t)seq * H + h) * kD * kD + tid;
#pragma unroll 1
      for (int c0 = 0; c0 < kD; c0 += 16) {
        float v[16];
        tmem_ld16(my_lane + TS32 + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) dst[(size_t)(c0 + i) * kD] = v[i];
      }
    }
    sync_tc();
  }

  if (!range_ok) report_error(P.err, kErrDeviceCheck);
  if (aborted) {
    if (tid == 0) {
      report_error(P.err, kErrTimeout);
      // let copies already in flight land before the shared memory goes away
      if (pend_qkz) wait_bar(bar_qkz, ph_qkz, P.spin_cycles);
      if (pend_v) wait_bar(bar_v, ph_v, P.spin_cycles);
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

}  // namespace tcp

bool chunk_tc_supported(const Problem& p, const Args& a) {
  if (!p.io_bf16 || p.dk != 128 || p.dv != 128) return false;
  auto al = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
  return al(a.q) && al(a.k) && al(a.v) && al(a.z) && al(a.out) &&
         (!a.initial_state || al(a.initial_state)) && (!a.final_state || al(a.final_state));
}

cudaError_t launch_chunk_tc(const Problem& p, const Args& a, const int32_t* cu_host,
                            cudaStream_t st) {
  using namespace tcp;
  if (p.num_seqs == 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return attr_err;

  CUtensorMap mq, mk, mv, mz;
  const int T = std::max(p.total_tokens, 1);
  if (!make_map(&mq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.num_heads, T, 64,
                CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.num_heads, T, 64,
                CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&mv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.num_heads, T, 64,
                CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&mz, a.z, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.num_heads, T, 128,
                CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;

  static thread_local Params prm;  // large: keep off the stack
  prm.beta = a.beta;
  prm.initial_state = a.initial_state;
  prm.cu = a.cu_seqlens;
  prm.out = static_cast<__nv_bfloat16*>(a.out);
  prm.final_state = a.final_state;
  prm.err = a.err;
  prm.H = p.num_heads;
  prm.total = p.total_tokens;
  prm.num_seqs = p.num_seqs;
  prm.num_units = p.num_seqs * p.num_heads;
  prm.spin_cycles = 4000000000LL;  // ~2 s at 2 GHz
  prm.use_order = 0;
  if (cu_host && p.num_seqs <= kMaxOrder) {
    std::vector<int> idx(p.num_seqs);
    std::iota(idx.begin(), idx.end(), 0);
    std::stable_sort(idx.begin(), idx.end(), [&](int x, int y) {
      return cu_host[x + 1] - cu_host[x] > cu_host[y + 1] - cu_host[y];
    });
    for (int i = 0; i < p.num_seqs; ++i) prm.order[i] = idx[i];
    prm.use_order = 1;
  }
  const int grid = std::min(prm.num_units, sms);
  chunk_tc_kernel<<<grid, kNT, SMEM_BYTES, st>>>(mq, mk, mv, mz, prm);
  return cudaGetLastError();
}

}  // namespace kda
