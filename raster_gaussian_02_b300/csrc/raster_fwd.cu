// Forward raster: one 256-thread block per 16x16 tile, one pixel per thread.
//
// The tile's Gaussian list is staged through shared memory in chunks of 256
// records (one coalesced gather per thread).  Each warp owns an 8x4 pixel
// sub-block and first compacts, with a ballot, the chunk entries whose pixel
// box meets its sub-block; it then evaluates only those, in list order.
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

constexpr int kFwdThreads = 256;
constexpr int kChunk = 256;

struct FwdStage {
  float4 mc[kChunk];  // mean_x, mean_y, A, 2B
  float4 cr[kChunk];  // C, r, g, b
  uint2 box[kChunk];  // packed pixel box
  float op[kChunk];   // opacity (composite)
  unsigned char list[8][kChunk];
};

template <bool kComposite>
__global__ void __launch_bounds__(kFwdThreads)
k_render_fwd(gs2d_config c, int tiles_x, const float4* __restrict__ rec,
             const int2* __restrict__ ranges, const int* __restrict__ sorted_gid,
             const float* __restrict__ bg, float* __restrict__ image, float* __restrict__ t_final,
             int* __restrict__ last) {
  __shared__ FwdStage sm;
  const int tile = blockIdx.x;
  const int tx = tile % tiles_x, ty = tile / tiles_x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bx0 = tx * kTile + (warp & 1) * 8;
  const int by0 = ty * kTile + (warp >> 1) * 4;
  const int px = bx0 + (lane & 7), py = by0 + (lane >> 3);
  const float pxf = float(px) + 0.5f, pyf = float(py) + 0.5f;
  const bool inside = px < c.width && py < c.height;
  const float kk = __fmul_rn(c.cutoff_sigma, c.cutoff_sigma);
  const unsigned int lt = (1u << lane) - 1u;
  const int2 rg = ranges[tile];
  const int start = rg.x, end = rg.y;

  float ar = 0.f, ag = 0.f, ab = 0.f, T = 1.f;
  int lst = 0;
  bool done = !inside;

  for (int cb = start; cb < end; cb += kChunk) {
    if (kComposite) {
      if (__syncthreads_and(done)) break;
    }
    const int k = cb + tid;
    if (k < end) {
      const float4* r = rec + 3 * size_t(sorted_gid[k]);
      const float4 p0 = r[0], p1 = r[1], p2 = r[2];
      sm.mc[tid] = make_float4(p0.x, p0.y, p0.z, 2.0f * p0.w);
      sm.cr[tid] = p1;
      sm.box[tid] = make_uint2(__float_as_uint(p2.x), __float_as_uint(p2.y));
      if (kComposite) sm.op[tid] = p2.z;
    }
    __syncthreads();
    const int cnt = min(kChunk, end - cb);
    bool skip = false;
    if (kComposite) skip = __all_sync(0xffffffffu, done);
    if (!skip) {
      int nl = 0;
      for (int j0 = 0; j0 < cnt; j0 += 32) {
        const int j = j0 + lane;
        bool hit = false;
        if (j < cnt) {
          const uint2 b = sm.box[j];
          hit = int(box_lo(b.x)) <= bx0 + 7 && int(box_hi(b.x)) >= bx0 &&
                int(box_lo(b.y)) <= by0 + 3 && int(box_hi(b.y)) >= by0;
        }
        const unsigned int m = __ballot_sync(0xffffffffu, hit);
        if (hit) sm.list[warp][nl + __popc(m & lt)] = (unsigned char)j;
        nl += __popc(m);
      }
      __syncwarp();
      for (int e = 0; e < nl; ++e) {
        const int j = sm.list[warp][e];
        const float4 mc = sm.mc[j];
        const float4 cr = sm.cr[j];
        const uint2 b = sm.box[j];
        const float dx = __fsub_rn(pxf, mc.x);
        const float dy = __fsub_rn(pyf, mc.y);
        const float q = touch_q(dx, dy, mc.z, mc.w, cr.x);
        const bool in = q <= kk &&
                        unsigned(px - int(box_lo(b.x))) <= unsigned(int(box_hi(b.x)) - int(box_lo(b.x))) &&
                        unsigned(py - int(box_lo(b.y))) <= unsigned(int(box_hi(b.y)) - int(box_lo(b.y)));
        if (kComposite) {
          if (in && !done) {
            if (T < c.t_min) {
              done = true;
            } else {
              const float w = ex2_approx(q * kNegHalfLog2e);
              const float alpha = sm.op[j] * w;
              const float aT = alpha * T;
              ar = fmaf(cr.y, aT, ar);
              ag = fmaf(cr.z, aT, ag);
              ab = fmaf(cr.w, aT, ab);
              T = T * (1.0f - alpha);
              lst = cb - start + j + 1;
            }
          }
        } else {
          if (in) {
            const float w = ex2_approx(q * kNegHalfLog2e);
            ar = fmaf(cr.y, w, ar);
            ag = fmaf(cr.z, w, ag);
            ab = fmaf(cr.w, w, ab);
          }
        }
      }
    }
    __syncthreads();
  }
  if (inside) {
    const size_t HW = size_t(c.width) * c.height;
    const size_t p = size_t(py) * c.width + px;
    if (kComposite) {
      if (bg) {
        ar = fmaf(T, bg[0], ar);
        ag = fmaf(T, bg[1], ag);
        ab = fmaf(T, bg[2], ab);
      }
      if (t_final) t_final[p] = T;
      if (last) last[p] = lst;
    }
    image[p] = ar;
    image[HW + p] = ag;
    image[2 * HW + p] = ab;
  }
}

}  // namespace

cudaError_t launch_render_fwd(const gs2d_config& c, const gs2d_record* rec, const int* ranges,
                              const int* sorted_gid, const float* bg, float* image, float* t_final,
                              int* last, cudaStream_t s) {
  const int T = num_tiles(c);
  const float4* r = reinterpret_cast<const float4*>(rec);
  const int2* rg = reinterpret_cast<const int2*>(ranges);
  if (c.mode == GS2D_MODE_COMPOSITE)
    k_render_fwd<true><<<T, kFwdThreads, 0, s>>>(c, tiles_x(c), r, rg, sorted_gid, bg, image,
                                                 t_final, last);
  else
    k_render_fwd<false><<<T, kFwdThreads, 0, s>>>(c, tiles_x(c), r, rg, sorted_gid, nullptr, image,
                                                  nullptr, nullptr);
  return cudaGetLastError();
}

}  // namespace gs2d
