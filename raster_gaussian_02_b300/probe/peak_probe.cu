// Throughput probes for the roofline's FP32 and SFU peaks (include/gs2d_probe.h).
// Each thread keeps 8 independent dependency chains, so that the issue
// slots, not the latency of one chain, limit the rate.
#include <cuda_runtime.h>

#include "gs2d_probe.h"

namespace {

constexpr int kThreads = 256;
constexpr int kChains = 8;

__global__ void __launch_bounds__(kThreads) k_probe_fma(float* __restrict__ out, int iters, float m,
                                                        float c) {
  float a[kChains];
#pragma unroll
  for (int j = 0; j < kChains; ++j) a[j] = float(threadIdx.x + j) * 1e-3f;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < kChains; ++j) a[j] = fmaf(a[j], m, c);
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kChains; ++j) s += a[j];
  out[size_t(blockIdx.x) * kThreads + threadIdx.x] = s;
}

__device__ __forceinline__ float ex2_neg(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(-x));
  return y;
}

__global__ void __launch_bounds__(kThreads) k_probe_ex2(float* __restrict__ out, int iters) {
  float a[kChains];
#pragma unroll
  for (int j = 0; j < kChains; ++j) a[j] = float(threadIdx.x + j) * 1e-3f;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < kChains; ++j) a[j] = ex2_neg(a[j]);
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kChains; ++j) s += a[j];
  out[size_t(blockIdx.x) * kThreads + threadIdx.x] = s;
}

bool args_ok(const float* out, int blocks, int iters) {
  return out && blocks >= 1 && blocks <= 65535 && iters >= 1 && iters <= (1 << 20);
}

}  // namespace

extern "C" {

int gs2d_probe_fp32_fma(float* out, int32_t blocks, int32_t iters, float m, float c,
                        gs2d_probe_stream_t stream) {
  if (!args_ok(out, blocks, iters)) return 1;
  k_probe_fma<<<blocks, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(out, iters, m, c);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

int gs2d_probe_ex2(float* out, int32_t blocks, int32_t iters, gs2d_probe_stream_t stream) {
  if (!args_ok(out, blocks, iters)) return 1;
  k_probe_ex2<<<blocks, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(out, iters);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // extern "C"
