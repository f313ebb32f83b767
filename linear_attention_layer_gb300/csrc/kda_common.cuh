// kda_common.cuh -- small device helpers shared by the libkda kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

// Lower bound of the log-decay: log alpha = kGateMin * sigmoid(z)
// (blog.higcp.com "猜想：K3 可能是最适合 TPU 的 MoE 架构", section "下界衰减").
constexpr float kGateMin = -5.0f;
// L2-normalisation epsilon: x / sqrt(sum x^2 + kNormEps).
constexpr float kNormEps = 1e-6f;

// Device error word codes (same values as kda_status_t).
constexpr int kErrTimeout = 4;
constexpr int kErrDeviceCheck = 5;

__device__ __forceinline__ void report_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

template <typename T>
struct IO;
template <>
struct IO<float> {
  static __device__ __forceinline__ float ld(const float* p) { return __ldg(p); }
  static __device__ __forceinline__ void st(float* p, float x) { *p = x; }
};
template <>
struct IO<__nv_bfloat16> {
  static __device__ __forceinline__ float ld(const __nv_bfloat16* p) {
    return __bfloat162float(__ldg(p));
  }
  static __device__ __forceinline__ void st(__nv_bfloat16* p, float x) {
    *p = __float2bfloat16_rn(x);
  }
};

// log-decay g = kGateMin * sigmoid(z).
__device__ __forceinline__ float log_decay(float z) {
  return __fdividef(kGateMin, 1.0f + __expf(-z));
}

// e^{A_h}, the scale applied to z before the gate (1 when no A is given).
__device__ __forceinline__ float gate_scale(const float* a_log, int h) {
  return a_log ? expf(__ldg(a_log + h)) : 1.f;
}

// 2^x by the hardware's approximate base-2 exponential (ex2.approx.ftz).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The gate with the head's scale folded into one coefficient (e^x = 2^{x log2 e}):
// g = kGateMin sigmoid(s z) = kGateMin / (1 + 2^{c z}), c = -s log2(e).
__device__ __forceinline__ float gate_coef(float zscale) { return -zscale * 1.4426950408889634f; }
__device__ __forceinline__ float log_decay_c(float z, float c) {
  return __fdividef(kGateMin, 1.0f + ex2_approx(c * z));
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Streaming (evict-first) 128-bit global load / store.
__device__ __forceinline__ float4 ld_stream(const float4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(float4* p, float4 v) { __stcs(p, v); }

// Checked [bos, eos) of sequence n; false (and the error word set) when the
// device copy of cu_seqlens is out of range or decreasing.
__device__ __forceinline__ bool seq_range(const int32_t* cu, int n, int total, int* err,
                                          int& bos, int& eos) {
  bos = cu[n];
  eos = cu[n + 1];
  if (bos < 0 || eos < bos || eos > total) {
    report_error(err, kErrDeviceCheck);
    return false;
  }
  return true;
}

}  // namespace kda
