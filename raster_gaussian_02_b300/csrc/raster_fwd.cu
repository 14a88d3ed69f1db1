// Forward raster: one block per 16x16 tile, one pixel per thread.
//
// Warps own 8x4-pixel sub-blocks of the tile.  The tile's Gaussian list is
// staged through shared memory (one coalesced record gather per thread);
// each warp then culls a window of 64 staged entries with one lane per
// entry, keeping, in list order, those whose pixel box meets its sub-block
// together with a 32-bit mask of the warp's lanes inside the box, so that
// the per-pixel box test is a single bit test.
//
// Sum (GaussianImage project page, Overview: accumulated-sum rendering;
// FlashImgs README: additive RGB, gate folded into the colour):
//     C(p) += rgb_i * exp(-q/2)            for every touching Gaussian i.
// Composite (DrawingWithGaussians README, Overview: alpha compositing over a
// trainable background), front to back in list (depth) order:
//     while T >= t_min: alpha = o_i exp(-q/2); C += rgb_i alpha T; T *= 1 - alpha
//     C += T * background.
#include "gs2d_internal.cuh"

namespace gs2d {

namespace {

constexpr int kWindow = 64;  // entries culled per warp at a time

struct Staged {
  float4 mc;  // mean_x, mean_y, A, 2B
  float4 cr;  // C, r, g, b
};

template <int kWarps>
struct SumSmem {
  Staged g[256];
  uint2 box[256];
  uint2 list[kWarps][kWindow];  // (staged index, lane mask)
};

// A block of kWarps warps renders 8/kWarps of a tile (kWarps 8: the whole
// tile; 4: a 16x8 half; 2: a 16x4 quarter).  Each warp owns an 8x4 pixel
// sub-block.  Smaller blocks stage the tile's records more than once but let
// the scheduler spread the heavy tiles (Gaussians crowd along image edges)
// over more SMs.
template <int kWarps>
__global__ void __launch_bounds__(kWarps * 32, kWarps == 8 ? 8 : (kWarps == 4 ? 10 : 20))
k_render_fwd_sum(gs2d_config c, int tiles_x, const float4* __restrict__ rec,
                 const int2* __restrict__ ranges, const int* __restrict__ sorted_gid,
                 float* __restrict__ image) {
  constexpr int kParts = 8 / kWarps;
  constexpr int kThreads = kWarps * 32;
  pdl_enter();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SumSmem<kWarps>& sm = *reinterpret_cast<SumSmem<kWarps>*>(smem_raw);
  const int tile = blockIdx.x / kParts;
  const int tx = tile % tiles_x, ty = tile / tiles_x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sub = (blockIdx.x % kParts) * kWarps + warp;  // 8x4 sub-block 0..7 of the tile
  const int bx0 = tx * kTile + (sub & 1) * 8;
  const int by0 = ty * kTile + (sub >> 1) * 4;
  const int px = bx0 + (lane & 7), py = by0 + (lane >> 3);
  const float pxf = float(px) + 0.5f, pyf = float(py) + 0.5f;
  const float kk = __fmul_rn(c.cutoff_sigma, c.cutoff_sigma);
  const unsigned int lt = (1u << lane) - 1u, bit = 1u << lane;
  const int2 rg = ranges[tile];
  uint2* list = sm.list[warp];

  float ar = 0.f, ag = 0.f, ab = 0.f;
  for (int rb = rg.x; rb < rg.y; rb += 256) {
    const int cnt = min(256, rg.y - rb);
    for (int k = tid; k < cnt; k += kThreads) {
      const float4* r = rec + 3 * size_t(sorted_gid[rb + k]);
      const float4 p0 = r[0], p1 = r[1], p2 = r[2];
      sm.g[k].mc = make_float4(p0.x, p0.y, p0.z, 2.0f * p0.w);
      sm.g[k].cr = p1;
      sm.box[k] = make_uint2(__float_as_uint(p2.x), __float_as_uint(p2.y));
    }
    __syncthreads();
    for (int wb = 0; wb < cnt; wb += kWindow) {
      const int wend = min(wb + kWindow, cnt);
      int nl = 0;
#pragma unroll
      for (int j0 = 0; j0 < kWindow; j0 += 32) {
        const int j = wb + j0 + lane;
        unsigned int m = 0;
        if (j < wend) m = box_lanes(sm.box[j], bx0, by0);
        const unsigned int hits = __ballot_sync(0xffffffffu, m != 0u);
        if (m) list[nl + __popc(hits & lt)] = make_uint2(unsigned(j), m);
        nl += __popc(hits);
      }
      __syncwarp();
      int e = 0;
      for (; e + 1 < nl; e += 2) {
        const uint2 u0 = list[e], u1 = list[e + 1];
        const Staged s0 = sm.g[u0.x], s1 = sm.g[u1.x];
        const float q0 = touch_q(__fsub_rn(pxf, s0.mc.x), __fsub_rn(pyf, s0.mc.y), s0.mc.z, s0.mc.w, s0.cr.x);
        const float q1 = touch_q(__fsub_rn(pxf, s1.mc.x), __fsub_rn(pyf, s1.mc.y), s1.mc.z, s1.mc.w, s1.cr.x);
        float w0 = ex2_approx(q0 * kNegHalfLog2e);
        float w1 = ex2_approx(q1 * kNegHalfLog2e);
        w0 = (q0 <= kk && (u0.y & bit)) ? w0 : 0.f;
        w1 = (q1 <= kk && (u1.y & bit)) ? w1 : 0.f;
        ar = fmaf(s0.cr.y, w0, ar);
        ag = fmaf(s0.cr.z, w0, ag);
        ab = fmaf(s0.cr.w, w0, ab);
        ar = fmaf(s1.cr.y, w1, ar);
        ag = fmaf(s1.cr.z, w1, ag);
        ab = fmaf(s1.cr.w, w1, ab);
      }
      if (e < nl) {
        const uint2 u0 = list[e];
        const Staged s0 = sm.g[u0.x];
        const float q0 = touch_q(__fsub_rn(pxf, s0.mc.x), __fsub_rn(pyf, s0.mc.y), s0.mc.z, s0.mc.w, s0.cr.x);
        float w0 = ex2_approx(q0 * kNegHalfLog2e);
        w0 = (q0 <= kk && (u0.y & bit)) ? w0 : 0.f;
        ar = fmaf(s0.cr.y, w0, ar);
        ag = fmaf(s0.cr.z, w0, ag);
        ab = fmaf(s0.cr.w, w0, ab);
      }
      __syncwarp();
    }
    __syncthreads();
  }
  if (px < c.width && py < c.height) {
    const size_t HW = size_t(c.width) * c.height;
    const size_t p = size_t(py) * c.width + px;
    image[p] = ar;
    image[HW + p] = ag;
    image[2 * HW + p] = ab;
  }
}

struct CompSmem {
  Staged g[256];
  uint2 box[256];
  float op[256];
  uint2 list[8][kWindow];
};

__global__ void __launch_bounds__(256)
k_render_fwd_comp(gs2d_config c, int tiles_x, const float4* __restrict__ rec,
                  const int2* __restrict__ ranges, const int* __restrict__ sorted_gid,
                  const float* __restrict__ bg, float* __restrict__ image,
                  float* __restrict__ t_final, int* __restrict__ last) {
  pdl_enter();
  __shared__ CompSmem sm;
  const int tile = blockIdx.x;
  const int tx = tile % tiles_x, ty = tile / tiles_x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bx0 = tx * kTile + (warp & 1) * 8;
  const int by0 = ty * kTile + (warp >> 1) * 4;
  const int px = bx0 + (lane & 7), py = by0 + (lane >> 3);
  const float pxf = float(px) + 0.5f, pyf = float(py) + 0.5f;
  const bool inside = px < c.width && py < c.height;
  const float kk = __fmul_rn(c.cutoff_sigma, c.cutoff_sigma);
  const unsigned int lt = (1u << lane) - 1u, bit = 1u << lane;
  const int2 rg = ranges[tile];
  uint2* list = sm.list[warp];

  float ar = 0.f, ag = 0.f, ab = 0.f, T = 1.f;
  int lst = 0;
  bool done = !inside;
  for (int rb = rg.x; rb < rg.y; rb += 256) {
    if (__syncthreads_and(done)) break;
    const int cnt = min(256, rg.y - rb);
    if (tid < cnt) {
      const float4* r = rec + 3 * size_t(sorted_gid[rb + tid]);
      const float4 p0 = r[0], p1 = r[1], p2 = r[2];
      sm.g[tid].mc = make_float4(p0.x, p0.y, p0.z, 2.0f * p0.w);
      sm.g[tid].cr = p1;
      sm.box[tid] = make_uint2(__float_as_uint(p2.x), __float_as_uint(p2.y));
      sm.op[tid] = p2.z;
    }
    __syncthreads();
    for (int wb = 0; wb < cnt; wb += kWindow) {
      if (__all_sync(0xffffffffu, done)) break;
      const int wend = min(wb + kWindow, cnt);
      int nl = 0;
#pragma unroll
      for (int j0 = 0; j0 < kWindow; j0 += 32) {
        const int j = wb + j0 + lane;
        unsigned int m = 0;
        if (j < wend) m = box_lanes(sm.box[j], bx0, by0);
        const unsigned int hits = __ballot_sync(0xffffffffu, m != 0u);
        if (m) list[nl + __popc(hits & lt)] = make_uint2(unsigned(j), m);
        nl += __popc(hits);
      }
      __syncwarp();
      for (int e = 0; e < nl; ++e) {
        const uint2 u = list[e];
        const Staged s = sm.g[u.x];
        const float q = touch_q(__fsub_rn(pxf, s.mc.x), __fsub_rn(pyf, s.mc.y), s.mc.z, s.mc.w, s.cr.x);
        if (q <= kk && (u.y & bit) && !done) {
          if (T < c.t_min) {
            done = true;
          } else {
            const float w = ex2_approx(q * kNegHalfLog2e);
            const float alpha = sm.op[u.x] * w;
            const float aT = alpha * T;
            ar = fmaf(s.cr.y, aT, ar);
            ag = fmaf(s.cr.z, aT, ag);
            ab = fmaf(s.cr.w, aT, ab);
            T = T * (1.0f - alpha);
            lst = rb - rg.x + int(u.x) + 1;
          }
        }
      }
      __syncwarp();
    }
    __syncthreads();
  }
  if (inside) {
    const size_t HW = size_t(c.width) * c.height;
    const size_t p = size_t(py) * c.width + px;
    if (bg) {
      ar = fmaf(T, bg[0], ar);
      ag = fmaf(T, bg[1], ag);
      ab = fmaf(T, bg[2], ab);
    }
    if (t_final) t_final[p] = T;
    if (last) last[p] = lst;
    image[p] = ar;
    image[HW + p] = ag;
    image[2 * HW + p] = ab;
  }
}

template <int kWarps>
cudaError_t launch_fwd_sum(const gs2d_config& c, const float4* r, const int2* rg, const int* sorted_gid,
                           float* image, cudaStream_t s) {
  const size_t smem = sizeof(SumSmem<kWarps>);
  auto kern = k_render_fwd_sum<kWarps>;
  GS2D_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
  GS2D_TRY(launch(kern, dim3(num_tiles(c) * (8 / kWarps)), dim3(kWarps * 32), smem, s, c, tiles_x(c), r,
                  rg, sorted_gid, image));
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_render_fwd(const gs2d_config& c, const gs2d_record* rec, const int* ranges,
                              const int* sorted_gid, const float* bg, float* image, float* t_final,
                              int* last, cudaStream_t s) {
  const int T = num_tiles(c);
  const float4* r = reinterpret_cast<const float4*>(rec);
  const int2* rg = reinterpret_cast<const int2*>(ranges);
  if (c.mode == GS2D_MODE_COMPOSITE) {
    GS2D_TRY(launch(k_render_fwd_comp, dim3(T), dim3(256), 0, s, c, tiles_x(c), r, rg, sorted_gid, bg, image, t_final, last));
  } else {
    // Half-tile blocks when the whole-tile blocks would fill at most two
    // waves of the GPU (8 resident per SM): the heavy tiles then spread over
    // more SMs.  With more tiles than that, staging each tile's records
    // twice costs more than the balance gains (measured on a B300: 768x512
    // 29.3 -> 27.2 us; 2048x2048 156 -> 168 us).
    if (T <= 2 * 8 * sm_count())
      GS2D_TRY(launch_fwd_sum<4>(c, r, rg, sorted_gid, image, s));
    else
      GS2D_TRY(launch_fwd_sum<8>(c, r, rg, sorted_gid, image, s));
  }
  return cudaGetLastError();
}

}  // namespace gs2d
