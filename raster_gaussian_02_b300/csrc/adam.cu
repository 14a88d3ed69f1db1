// Selective Adam step on row-aligned parameters (DrawingWithGaussians README,
// MLX-specific notes: the COLMAP trainer keeps row-aligned optimizer state
// for its selective Adam; the update is Adam's, moments with bias
// correction).  One thread per element of a [n, width] array; with a pair
// count per row the step skips the rows whose Gaussian touched no tile
// (their parameters and both moments stay as they are).  Memory-bound:
// 16 bytes read and 12 written per updated element.
#include <cmath>

#include "gs2d_internal.cuh"

namespace gs2d {

namespace {

constexpr int kAdamThreads = 256;

__global__ void __launch_bounds__(kAdamThreads)
k_adam(long long total, int width, float* __restrict__ param, const float* __restrict__ grad,
       float* __restrict__ m, float* __restrict__ v, const int* __restrict__ count, float beta1,
       float beta2, float eps, float step_size, float sqrt_bc2) {
  pdl_enter();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    if (count && count[i / width] == 0) continue;
    const float g = grad[i];
    const float mi = fmaf(beta1, m[i], (1.0f - beta1) * g);
    const float vi = fmaf(beta2, v[i], (1.0f - beta2) * g * g);
    m[i] = mi;
    v[i] = vi;
    // p -= (lr / bc1) * m / (sqrt(v) / sqrt(bc2) + eps)
    param[i] -= step_size * (mi / (sqrtf(vi) / sqrt_bc2 + eps));
  }
}

}  // namespace

cudaError_t launch_adam(int n, int width, float* param, const float* grad, float* m, float* v,
                        const int* count, float lr, float beta1, float beta2, float eps, int step,
                        cudaStream_t s) {
  const long long total = (long long)n * width;
  if (total == 0) return cudaSuccess;
  // bias corrections in double, then rounded once
  const double bc1 = 1.0 - pow(double(beta1), double(step));
  const double bc2 = 1.0 - pow(double(beta2), double(step));
  const float step_size = float(double(lr) / bc1);
  const float sqrt_bc2 = float(sqrt(bc2));
  long long blocks = (total + kAdamThreads - 1) / kAdamThreads;
  const long long cap = 8ll * sm_count();  // grid-stride beyond 8 blocks per SM
  if (blocks > cap) blocks = cap;
  GS2D_TRY(launch(k_adam, dim3(unsigned(blocks)), dim3(kAdamThreads), 0, s, total, width, param, grad, m, v,
                  count, beta1, beta2, eps, step_size, sqrt_bc2));
  return cudaGetLastError();
}

}  // namespace gs2d
