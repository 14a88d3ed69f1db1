// L2 image loss (FlashImgs README, Configuration: l2_loss_ratio, the L2/MSE
// weight):  loss = (1/(3HW)) sum (C - target)^2,  dL/dC = 2 (C - target)/(3HW).
// Two kernels, no atomics: every block writes the partial sum of a fixed
// grid-stride set of elements, then one block adds the partials in order,
// so the loss is bit-reproducible.
#include <atomic>
#include <mutex>

#include "gs2d_internal.cuh"

namespace gs2d {

namespace {

constexpr int kLossThreads = 256;

__device__ __forceinline__ float block_sum_256(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.f;
  if (threadIdx.x == 0)
    for (int w = 0; w < kLossThreads / 32; ++w) s += red[w];
  return s;
}

template <bool kVec>
__global__ void __launch_bounds__(kLossThreads)
k_loss_partial(long long m, const float* __restrict__ image, const float* __restrict__ target,
               float scale, float* __restrict__ d_image, float* __restrict__ partials) {
  pdl_enter();
  __shared__ float red[kLossThreads / 32];
  float acc = 0.f;
  const long long stride = (long long)gridDim.x * blockDim.x;
  if (kVec) {
    const float4* a = reinterpret_cast<const float4*>(image);
    const float4* b = reinterpret_cast<const float4*>(target);
    float4* d = reinterpret_cast<float4*>(d_image);
    for (long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x; k < m / 4; k += stride) {
      const float4 x = a[k], y = b[k];
      const float4 e = make_float4(x.x - y.x, x.y - y.y, x.z - y.z, x.w - y.w);
      d[k] = make_float4(e.x * scale, e.y * scale, e.z * scale, e.w * scale);
      acc = fmaf(e.x, e.x, acc);
      acc = fmaf(e.y, e.y, acc);
      acc = fmaf(e.z, e.z, acc);
      acc = fmaf(e.w, e.w, acc);
    }
  } else {
    for (long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x; k < m; k += stride) {
      const float e = image[k] - target[k];
      d_image[k] = e * scale;
      acc = fmaf(e, e, acc);
    }
  }
  const float s = block_sum_256(acc, red);
  if (threadIdx.x == 0) partials[blockIdx.x] = s;
}

__global__ void __launch_bounds__(kLossThreads)
k_loss_final(int nb, const float* __restrict__ partials, float m, float* __restrict__ loss) {
  pdl_enter();
  __shared__ float red[kLossThreads / 32];
  float acc = 0.f;
  for (int k = threadIdx.x; k < nb; k += blockDim.x) acc += partials[k];
  const float s = block_sum_256(acc, red);
  if (threadIdx.x == 0) *loss = s / m;
}

}  // namespace

namespace {

// The loss's two kernels with the block partial sums in `partials`
// (kLossMaxBlocks floats): shared by the workspace and the fixed-array
// entry points, so that both give the same loss bit for bit.
cudaError_t launch_loss_l2_into(int h, int w, const float* image, const float* target, float* loss,
                                float* d_image, float* partials, cudaStream_t s) {
  const long long m = 3ll * h * w;
  const bool vec = (m % 4 == 0) && ((reinterpret_cast<uintptr_t>(image) |
                                     reinterpret_cast<uintptr_t>(target) |
                                     reinterpret_cast<uintptr_t>(d_image)) & 15) == 0;
  const long long work = vec ? m / 4 : m;
  long long blocks = (work + kLossThreads * 4 - 1) / (kLossThreads * 4);
  if (blocks < 1) blocks = 1;
  if (blocks > kLossMaxBlocks) blocks = kLossMaxBlocks;
  const float scale = float(2.0 / double(m));
  if (vec)
    GS2D_TRY(launch(k_loss_partial<true>, dim3(int(blocks)), dim3(kLossThreads), 0, s, m, image, target, scale, d_image, partials));
  else
    GS2D_TRY(launch(k_loss_partial<false>, dim3(int(blocks)), dim3(kLossThreads), 0, s, m, image, target, scale, d_image, partials));
  GS2D_TRY(launch(k_loss_final, dim3(1), dim3(kLossThreads), 0, s, int(blocks), partials, float(m), loss));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_loss_l2(int h, int w, const float* image, const float* target, float* loss,
                           float* d_image, unsigned char* ws, cudaStream_t s) {
  return launch_loss_l2_into(h, w, image, target, loss, d_image,
                             reinterpret_cast<float*>(ws + kOffLoss), s);
}

}  // namespace gs2d

// ---------------------------------------------------------------------------
// L2 loss without a caller-supplied workspace.
//
// Some callers cannot hand the library any device memory beyond the image,
// target and outputs: code that receives its buffers from another framework
// and has no allocator of its own to call, or a loop that must not call
// cudaMalloc because it implicitly synchronises the device or is not allowed
// while a stream capture is in progress.  For them the block partial sums
// of the loss live in this fixed device array instead of the workspace.
// The array is 4 KiB (kLossMaxBlocks floats); every GPU that loads the
// library holds one copy until the process exits.  The reduction never uses
// more than kLossMaxBlocks blocks, so every image within the library's
// 32768 x 32768 limit fits; larger ones are rejected.
static __device__ __align__(256) float g_loss_scratch[gs2d::kLossMaxBlocks];

namespace gs2d {

namespace {

constexpr int kMaxDevices = 256;

// The array's address is looked up once per device and CUDA context: a
// device reset (cudaDeviceReset) ends the context that holds the array, and
// the new context may hold it elsewhere, so a context change triggers a new
// lookup.  The current context is read with the driver's cuCtxGetCurrent,
// reached through the runtime (no link against the driver library); that
// query is allowed during a stream capture, the lookup itself is not.
struct ScratchSlot {
  std::atomic<void*> ctx{nullptr};   // the context the address belongs to
  std::atomic<float*> addr{nullptr};
};
ScratchSlot g_loss_scratch_slot[kMaxDevices];
std::mutex g_loss_scratch_mu;

using CtxGetCurrent = int (*)(void**);  // cuCtxGetCurrent(CUcontext*), CUresult 0 = success

CtxGetCurrent ctx_get_current() {
  static const CtxGetCurrent fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return CtxGetCurrent(nullptr);
    return reinterpret_cast<CtxGetCurrent>(p);
  }();
  return fn;
}

// The device address of g_loss_scratch in the current device's current context.
cudaError_t loss_scratch_address(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const CtxGetCurrent get = ctx_get_current();
  void* ctx = nullptr;
  if (!get || get(&ctx) != 0) return cudaErrorDeviceUninitialized;
  if (!ctx) {  // no context current yet (a first call, never inside a capture): make one
    e = cudaFree(nullptr);
    if (e != cudaSuccess) return e;
    if (get(&ctx) != 0 || !ctx) return cudaErrorDeviceUninitialized;
  }
  ScratchSlot& slot = g_loss_scratch_slot[dev];
  if (slot.ctx.load(std::memory_order_acquire) != ctx) {
    std::lock_guard<std::mutex> lock(g_loss_scratch_mu);
    if (slot.ctx.load(std::memory_order_acquire) != ctx) {
      void* addr = nullptr;
      e = cudaGetSymbolAddress(&addr, g_loss_scratch);
      if (e != cudaSuccess) return e;
      slot.addr.store(static_cast<float*>(addr), std::memory_order_relaxed);
      slot.ctx.store(ctx, std::memory_order_release);  // publishes addr
    }
  }
  *out = slot.addr.load(std::memory_order_relaxed);
  return cudaSuccess;
}

}  // namespace

}  // namespace gs2d

extern "C" gs2d_status gs2d_loss_l2_noalloc(int32_t height, int32_t width, const float* image,
                                            const float* target, float* loss, float* d_image,
                                            gs2d_stream_t stream) {
  using namespace gs2d;
  if (height < 1 || width < 1 || height > 32768 || width > 32768) return GS2D_ERR_INVALID_ARG;
  if (!image || !target || !loss || !d_image) return GS2D_ERR_INVALID_ARG;
  const uintptr_t bits = reinterpret_cast<uintptr_t>(image) | reinterpret_cast<uintptr_t>(target) |
                         reinterpret_cast<uintptr_t>(loss) | reinterpret_cast<uintptr_t>(d_image);
  if (bits & 3) return GS2D_ERR_INVALID_ARG;
  float* partials = nullptr;
  if (loss_scratch_address(&partials) != cudaSuccess) return GS2D_ERR_CUDA;
  // The same two kernels as gs2d_loss_l2, with the partials in the fixed array.
  return launch_loss_l2_into(height, width, image, target, loss, d_image, partials,
                             reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GS2D_OK
             : GS2D_ERR_CUDA;
}
