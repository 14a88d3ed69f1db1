// Projection (shape parameters -> inverse covariance, 3-sigma pixel box,
// tile rectangle) and its backward (per-pair partial gradients summed per
// Gaussian, then the chain rule from the inverse covariance to the shape).
//
// Sigma = L L^T with L = [[a, 0], [b, c]] (DrawingWithGaussians README,
// MLX-specific notes: lower-triangular L), or Sigma = R diag(s_x^2, s_y^2) R^T
// (FlashImgs README, Python API: project_gaussians_2d_scale_rot; GaussianImage
// project page, the "rs" scripts); the 8 parameters per Gaussian are
// position, covariance and colour (GaussianImage project page, Overview).
#include "project_body.cuh"

namespace gs2d {

namespace {

__global__ void __launch_bounds__(256)
k_project(gs2d_config c, int n, const float* __restrict__ xy, const float* __restrict__ chol,
          const float* __restrict__ rgb, const float* __restrict__ depth,
          const float* __restrict__ opacity, float4* __restrict__ rec, int4* __restrict__ rect,
          int* __restrict__ count) {
  pdl_enter();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) project_one(c, i, xy, chol, rgb, depth, opacity, rec, rect, count);
}

// Per Gaussian: sum its per-pair partials (one per tile of its rectangle, in
// emission order) and apply the chain rule to the shape parameters
// (sum_pair_partials, write_gaussian_grads).
// kAbs: also the pairs' absgrad sums (third float4 of the slot, .y and .z).
// One extra block, the last, sums no Gaussian: it adds, in a fixed order, the
// per-tile background partials (composite, d_bg non-null) and the fused
// pass's per-block loss partials (loss non-null; the total is divided by m,
// the number of image values).
constexpr int kWarpSlots = 32;

template <bool kComposite, bool kAbs>
__global__ void __launch_bounds__(256)
k_gather(int n, const float* __restrict__ chol, const float4* __restrict__ rec,
         const int4* __restrict__ rect, const int* __restrict__ offsets,
         const float4* __restrict__ partials, const Header* __restrict__ hdr,
         float* __restrict__ d_xy, float* __restrict__ d_chol, float* __restrict__ d_rgb,
         float* __restrict__ d_opacity, int T, const float4* __restrict__ tile_partials,
         float* __restrict__ d_bg, const float* __restrict__ loss_partials, int loss_blocks,
         float* __restrict__ loss, float m, int param, float sc, float* __restrict__ d_xy_abs) {
  pdl_enter();
  constexpr int kStride = (kComposite || kAbs) ? 3 : 2;  // float4 per pair slot
  const bool extra = blockIdx.x == gridDim.x - 1;
  const int i = extra ? n : blockIdx.x * blockDim.x + threadIdx.x;
  const int lane = threadIdx.x & 31;
  const bool bad = (hdr->flags & (GS2D_FLAG_CAPACITY | GS2D_FLAG_OVERFLOW | GS2D_FLAG_TIMEOUT)) != 0;
  // every per-Gaussian load is issued up front, so one round trip precedes
  // the partial slots' reads
  int4 rc = make_int4(0, 0, -1, -1);
  int off = 0;
  float A = 0.f;
  float3 shp = make_float3(0.f, 0.f, 0.f);
  if (i < n) {
    rc = rect[i];
    off = offsets[i];
    A = rec[3 * size_t(i)].z;
    shp = make_float3(chol[3 * i], chol[3 * i + 1], chol[3 * i + 2]);
  }
  const int cnt = (rc.z >= rc.x) ? (rc.z - rc.x + 1) * (rc.w - rc.y + 1) : 0;
  float s[9] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float ax = 0.f, ay = 0.f;
  const bool ok = i < n && !bad && cnt > 0 &&
                  check_ok(off >= 0 && off + (long long)cnt <= hdr->pairs, kCheckPartial);
  // A Gaussian with more than kWarpSlots slots (a large one, over many tiles)
  // is summed by its whole warp: lane l adds slots l, l + 32, ... in order,
  // then the lanes' sums are added in a fixed butterfly.  Alone, one thread's
  // chain through a few hundred slots set the kernel's length.
  const bool big = ok && cnt > kWarpSlots;
  if (ok && !big) sum_pair_partials<kStride, kComposite, kAbs>(partials + size_t(off) * kStride, cnt, s, ax, ay);
  for (unsigned int todo = __ballot_sync(0xffffffffu, big); todo; todo &= todo - 1) {
    const int src = __ffs(todo) - 1;
    const int boff = __shfl_sync(0xffffffffu, off, src), bcnt = __shfl_sync(0xffffffffu, cnt, src);
    float t[9] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float tx = 0.f, ty = 0.f;
    for (int k0 = lane; k0 < bcnt; k0 += 4 * 32) {
      float4 q[4][kStride];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (k0 + 32 * j < bcnt)
#pragma unroll
          for (int u = 0; u < kStride; ++u) q[j][u] = partials[size_t(boff + k0 + 32 * j) * kStride + u];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (k0 + 32 * j >= bcnt) break;
        t[0] += q[j][0].x; t[1] += q[j][0].y; t[2] += q[j][0].z; t[3] += q[j][0].w;
        t[4] += q[j][1].x; t[5] += q[j][1].y; t[6] += q[j][1].z; t[7] += q[j][1].w;
        if constexpr (kComposite || kAbs) {
          if (kComposite) t[8] += q[j][kStride - 1].x;
          if (kAbs) {
            tx += q[j][kStride - 1].y;
            ty += q[j][kStride - 1].z;
          }
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
      for (int u = 0; u < 9; ++u) t[u] += __shfl_xor_sync(0xffffffffu, t[u], o);
      tx += __shfl_xor_sync(0xffffffffu, tx, o);
      ty += __shfl_xor_sync(0xffffffffu, ty, o);
    }
    if (lane == src) {
#pragma unroll
      for (int u = 0; u < 9; ++u) s[u] = t[u];
      ax = tx;
      ay = ty;
    }
  }
  if (i < n)
    write_gaussian_grads(i, ok, s, ax, ay, A, shp, param, sc, d_xy, d_chol, d_rgb,
                         kComposite ? d_opacity : nullptr, kAbs ? d_xy_abs : nullptr);
  if ((d_bg || loss) && extra) {  // beside the others (done by block 0 after its own sums: 768x512 step 63.6 -> 62.1 us)
    // fixed-order reduction of the per-tile partials
    // Each thread adds entries tid, tid + 256, ... in that order; the loads of
    // kBatch entries are issued before their adds, so one round trip serves
    // kBatch of them.
    constexpr int kBatch = 8;
    __shared__ float red[4][256];
    float x = 0.f, y = 0.f, z = 0.f, l = 0.f;
    if (d_bg)
      for (int t0 = threadIdx.x; t0 < T; t0 += kBatch * blockDim.x) {
        float4 v[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const int t = t0 + j * blockDim.x;
          if (t < T) v[j] = tile_partials[t];
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
          if (t0 + j * int(blockDim.x) < T) {
            x += v[j].x; y += v[j].y; z += v[j].z;
          }
      }
    if (loss)
      for (int t0 = threadIdx.x; t0 < loss_blocks; t0 += kBatch * blockDim.x) {
        float v[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const int t = t0 + j * blockDim.x;
          if (t < loss_blocks) v[j] = loss_partials[t];
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
          if (t0 + j * int(blockDim.x) < loss_blocks) l += v[j];
      }
    red[0][threadIdx.x] = x;
    red[1][threadIdx.x] = y;
    red[2][threadIdx.x] = z;
    red[3][threadIdx.x] = l;
    __syncthreads();
    for (int h = blockDim.x / 2; h > 0; h >>= 1) {
      if (threadIdx.x < h)
        for (int q = 0; q < 4; ++q) red[q][threadIdx.x] += red[q][threadIdx.x + h];
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      if (d_bg) {
        d_bg[0] = bad ? 0.f : red[0][0];
        d_bg[1] = bad ? 0.f : red[1][0];
        d_bg[2] = bad ? 0.f : red[2][0];
      }
      if (loss) *loss = red[3][0] / m;
    }
  }
}

}  // namespace

cudaError_t launch_project(const gs2d_config& c, int n, const float* xy, const float* chol,
                           const float* rgb, const float* depth, const float* opacity,
                           gs2d_record* rec, int* rect, int* count, cudaStream_t s) {
  if (n > 0)
    GS2D_TRY(launch(k_project, dim3((n + 255) / 256), dim3(256), 0, s, c, n, xy, chol, rgb, depth, opacity,
                                              reinterpret_cast<float4*>(rec),
                                              reinterpret_cast<int4*>(rect), count));
  return cudaGetLastError();
}

cudaError_t launch_gather(const gs2d_config& c, int n, const float* chol, const gs2d_record* rec,
                          const int* rect, const unsigned char* ws, float* d_xy, float* d_chol,
                          float* d_rgb, float* d_opacity, float* d_bg, float* d_xy_abs,
                          float* loss, int loss_blocks, cudaStream_t s) {
  const Layout L = layout_of(c, n, 0);
  const int T = num_tiles(c);
  const int blocks = n > 0 ? (n + 255) / 256 : 1;
  const Header* hdr = reinterpret_cast<const Header*>(ws);
  const float m = float(3.0 * double(c.width) * double(c.height));
  const float4* tp = reinterpret_cast<const float4*>(ws + L.tile_partials);
  const float* lp = reinterpret_cast<const float*>(ws + L.loss_partials);
  const int* offsets = reinterpret_cast<const int*>(ws + L.offsets);
  const float4* partials = reinterpret_cast<const float4*>(ws + L.partials);
  const float4* r = reinterpret_cast<const float4*>(rec);
  const int4* rc = reinterpret_cast<const int4*>(rect);
  const int param = int(c.param);
  const bool comp = c.mode == GS2D_MODE_COMPOSITE;
  float* d_op = comp ? d_opacity : nullptr;
  float* d_b = comp ? d_bg : nullptr;
  auto go = [&](auto kern) {
    return launch(kern, dim3(blocks + 1), dim3(256), 0, s, n, chol, r, rc, offsets, partials, hdr, d_xy,
                  d_chol, d_rgb, d_op, T, tp, d_b, lp, loss_blocks, loss, m, param, render_scale(c),
                  d_xy_abs);
  };
  if (comp)
    GS2D_TRY(d_xy_abs ? go(k_gather<true, true>) : go(k_gather<true, false>));
  else
    GS2D_TRY(d_xy_abs ? go(k_gather<false, true>) : go(k_gather<false, false>));
  return cudaGetLastError();
}

GS2D_CHECK_WORD_READER(project)

}  // namespace gs2d
