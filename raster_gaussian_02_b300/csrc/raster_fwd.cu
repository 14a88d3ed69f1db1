// Forward raster: one block per 16x16 tile (or a half tile), one pixel per
// thread; the per-tile bodies live in tile_bodies.cuh.
//
// Sum (GaussianImage project page, Overview: accumulated-sum rendering;
// FlashImgs README: additive RGB, gate folded into the colour):
//     C(p) += rgb_i * exp(-q/2)            for every touching Gaussian i.
// Composite (DrawingWithGaussians README, Overview: alpha compositing over a
// trainable background), front to back in list (depth) order:
//     while T >= t_min: alpha = o_i exp(-q/2); C += rgb_i alpha T; T *= 1 - alpha
//     C += T * background.
#include "tile_bodies.cuh"

namespace gs2d {

namespace {

// A block of kWarps warps renders 8/kWarps of a tile (kWarps 8: the whole
// tile; 4: a 16x8 half).  Smaller blocks stage the tile's records more than
// once but let the scheduler spread the heavy tiles (Gaussians crowd along
// image edges) over more SMs.
// kLoss (the fused training pass): also forms the L2 loss at each pixel,
// writing dL/dC = scale (C - target) to d_image and the block's sum of
// (C - target)^2 (warps in order) to loss_partials[blockIdx.x]; the image
// is then optional (NULL: not written).
template <int kWarps, bool kLoss>
__global__ void __launch_bounds__(kWarps * 32, kWarps == 8 ? 8 : 10)
k_render_fwd_sum(gs2d_config c, int tiles_x, int n, const float4* __restrict__ rec,
                 const int2* __restrict__ ranges, const int* __restrict__ sorted_gid,
                 float* __restrict__ image, const float* __restrict__ target, float scale,
                 float* __restrict__ d_image, float* __restrict__ loss_partials,
                 const int4* __restrict__ order) {
  constexpr int kParts = 8 / kWarps;
  pdl_enter();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SumSmem<kWarps>& sm = *reinterpret_cast<SumSmem<kWarps>*>(smem_raw);
  int2 rg;
  const int tile = tile_of_slot(order, int(blockIdx.x / kParts), ranges, tiles_x * ((c.height + kTile - 1) / kTile), &rg);
  if (!check_ok(tile >= 0 && tile < tiles_x * ((c.height + kTile - 1) / kTile), kCheckTile) || tile < 0) return;
  const int tx = tile % tiles_x, ty = tile / tiles_x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = (blockIdx.x % kParts) * kWarps + warp;  // 8x4 sub-block 0..7 of the tile
  const int bx0 = tx * kTile + (sub & 1) * 8;
  const int by0 = ty * kTile + (sub >> 1) * 4;
  const int px = bx0 + (lane & 7), py = by0 + (lane >> 3);
  const float kk = __fmul_rn(c.cutoff_sigma, c.cutoff_sigma);
  if (!check_ok(rg.x >= 0 && rg.x <= rg.y, kCheckRange)) rg = make_int2(0, 0);
  const float3 a = sum_tile_forward<kWarps>(sm, rg, bx0, by0, float(px) + 0.5f, float(py) + 0.5f, kk,
                                            n, rec, sorted_gid);
  const bool inside = px < c.width && py < c.height;
  const size_t HW = size_t(c.width) * c.height;
  const size_t p = size_t(py) * c.width + px;
  if (inside && (!kLoss || image)) {
    image[p] = a.x;
    image[HW + p] = a.y;
    image[2 * HW + p] = a.z;
  }
  if constexpr (kLoss) {
    float er = 0.f, eg = 0.f, eb = 0.f;
    if (inside) {
      er = a.x - target[p];
      eg = a.y - target[HW + p];
      eb = a.z - target[2 * HW + p];
      d_image[p] = er * scale;
      d_image[HW + p] = eg * scale;
      d_image[2 * HW + p] = eb * scale;
    }
    const float l = block_sum_ordered<kWarps>(fmaf(eb, eb, fmaf(eg, eg, er * er)), sm.red);
    // indexed by tile (not by block) so that the launch order cannot change the sum
    if (threadIdx.x == 0) loss_partials[tile * kParts + int(blockIdx.x % kParts)] = l;
  }
}

__global__ void __launch_bounds__(256)
k_render_fwd_comp(gs2d_config c, int tiles_x, int n, const float4* __restrict__ rec,
                  const int2* __restrict__ ranges, const int* __restrict__ sorted_gid,
                  const float* __restrict__ bg, float* __restrict__ image,
                  float* __restrict__ t_final, int* __restrict__ last, const int4* __restrict__ order) {
  pdl_enter();
  __shared__ CompSmem sm;
  int2 rg;
  const int tile = tile_of_slot(order, int(blockIdx.x), ranges, tiles_x * ((c.height + kTile - 1) / kTile), &rg);  // longest lists first when known
  if (!check_ok(tile >= 0 && tile < tiles_x * ((c.height + kTile - 1) / kTile), kCheckTile) || tile < 0) return;
  const int tx = tile % tiles_x, ty = tile / tiles_x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bx0 = tx * kTile + (warp & 1) * 8;
  const int by0 = ty * kTile + (warp >> 1) * 4;
  const int px = bx0 + (lane & 7), py = by0 + (lane >> 3);
  const bool inside = px < c.width && py < c.height;
  const float kk = __fmul_rn(c.cutoff_sigma, c.cutoff_sigma);
  if (!check_ok(rg.x >= 0 && rg.x <= rg.y, kCheckRange)) rg = make_int2(0, 0);
  const CompFwdOut o = comp_tile_forward(sm, c, rg, bx0, by0, float(px) + 0.5f, float(py) + 0.5f,
                                         inside, kk, n, rec, sorted_gid);
  if (inside) {
    const size_t HW = size_t(c.width) * c.height;
    const size_t p = size_t(py) * c.width + px;
    float ar = o.r, ag = o.g, ab = o.b;
    if (bg) {
      ar = fmaf(o.T, bg[0], ar);
      ag = fmaf(o.T, bg[1], ag);
      ab = fmaf(o.T, bg[2], ab);
    }
    if (t_final) t_final[p] = o.T;
    if (last) last[p] = o.last;
    image[p] = ar;
    image[HW + p] = ag;
    image[2 * HW + p] = ab;
  }
}

template <int kWarps, bool kLoss>
cudaError_t launch_fwd_sum(const gs2d_config& c, int n, const float4* r, const int2* rg, const int* sorted_gid,
                           float* image, const float* target, float scale, float* d_image,
                           float* loss_partials, const int4* order, cudaStream_t s) {
  const size_t smem = sizeof(SumSmem<kWarps>);
  auto kern = k_render_fwd_sum<kWarps, kLoss>;
  GS2D_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
  GS2D_TRY(launch(kern, dim3(num_tiles(c) * (8 / kWarps)), dim3(kWarps * 32), smem, s, c, tiles_x(c), n,
                  r, rg, sorted_gid, image, target, scale, d_image, loss_partials, order));
  return cudaSuccess;
}

// Half-tile blocks when the whole-tile blocks would fill at most two waves
// of the GPU (8 resident per SM): the heavy tiles then spread over more SMs.
// With more tiles than that, staging each tile's records twice costs more
// than the balance gains (measured on a B300: 768x512 29.3 -> 27.2 us;
// 2048x2048 156 -> 168 us).
bool half_tile_blocks(int T) { return T <= 2 * 8 * sm_count(); }

}  // namespace

cudaError_t launch_render_fwd(const gs2d_config& c, int n, const gs2d_record* rec, const int* ranges,
                              const int* sorted_gid, const float* bg, float* image, float* t_final,
                              int* last, const unsigned char* ws, cudaStream_t s) {
  const int T = num_tiles(c);
  const float4* r = reinterpret_cast<const float4*>(rec);
  const int2* rg = reinterpret_cast<const int2*>(ranges);
  // the binning's launch order (counting sort only), when its workspace is given
  const int4* order = nullptr;
  if (ws) {
    const Layout L = layout_of(c, n, 0);
    if (L.count_sort) order = reinterpret_cast<const int4*>(ws + L.tile_order);
  }
  if (c.mode == GS2D_MODE_COMPOSITE) {
    GS2D_TRY(launch(k_render_fwd_comp, dim3(T), dim3(256), 0, s, c, tiles_x(c), n, r, rg, sorted_gid, bg, image,
                    t_final, last, order));
  } else {
    if (half_tile_blocks(T))
      GS2D_TRY((launch_fwd_sum<4, false>(c, n, r, rg, sorted_gid, image, nullptr, 0.f, nullptr, nullptr,
                                         order, s)));
    else
      GS2D_TRY((launch_fwd_sum<8, false>(c, n, r, rg, sorted_gid, image, nullptr, 0.f, nullptr, nullptr,
                                         order, s)));
  }
  return cudaGetLastError();
}

cudaError_t launch_render_fwd_loss(const gs2d_config& c, int n, const gs2d_record* rec, const int* ranges,
                                   const int* sorted_gid, const float* target, float scale,
                                   float* image, float* d_image, float* loss_partials, int* blocks,
                                   const int4* order, cudaStream_t s) {
  const int T = num_tiles(c);
  const float4* r = reinterpret_cast<const float4*>(rec);
  const int2* rg = reinterpret_cast<const int2*>(ranges);
  if (half_tile_blocks(T)) {
    *blocks = 2 * T;
    GS2D_TRY((launch_fwd_sum<4, true>(c, n, r, rg, sorted_gid, image, target, scale, d_image, loss_partials,
                                      order, s)));
  } else {
    *blocks = T;
    GS2D_TRY((launch_fwd_sum<8, true>(c, n, r, rg, sorted_gid, image, target, scale, d_image, loss_partials,
                                      order, s)));
  }
  return cudaGetLastError();
}

GS2D_CHECK_WORD_READER(raster_fwd)

}  // namespace gs2d
