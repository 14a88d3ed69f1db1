// Backward raster.  Gradients of the loss given dL/dC, with the touch and
// early-termination decisions held fixed.  Every (tile, Gaussian) pair
// writes its partial gradient to its own slot (the pair's emission slot:
// the Gaussian's pair offset plus the tile's position in its rectangle), so
// no atomics are needed and the per-Gaussian sums, taken later in a fixed
// order, are bit-reproducible.
//
// With q = A dx^2 + 2B dx dy + C dy^2 (dx = px - mu_x, dy = py - mu_y) and
// w = exp(-q/2), write t = w * dL/dw at a pixel.  Then dL/dq = -t/2 and
//     dL/dmu_x = sum t (A dx + B dy),   dL/dmu_y = sum t (B dx + C dy),
//     dL/dA = -1/2 sum t dx^2,  dL/dB = -sum t dx dy,  dL/dC = -1/2 sum t dy^2.
// Sum mode: dL/dw = sum_k g_k rgb_k and dL/drgb_k = sum g_k w (g = dL/dC).
// Composite: with alpha = o w, T the transmittance in front of the
// Gaussian and S the colour accumulated behind it (including T_final * bg),
//     dL/dalpha = sum_k g_k (rgb_k T - S_k / (1 - alpha)),
//     dL/do = w dL/dalpha,  dL/dw = o dL/dalpha,  dL/drgb_k = g_k alpha T,
//     dL/dbg_k = sum over pixels of T_final g_k.
#include "tile_bodies.cuh"

namespace gs2d {

namespace {

constexpr int kBwdThreads = 256;  // threads per block; pairs per block round: at most 256 / kSplit
// Tiles of dL/dC staged at a time (kStage): 8 with at most 2048 tiles, where
// a one-round chunk of up to 256 pairs spans several tiles (with 6, 768x512
// went 23.4 -> 35.6 us: chunks over more tiles skip the shape sort); 4 on
// larger images, where a 256-pair chunk spans 2-3 tiles and the smaller
// footprint leaves the L1 more room (2048x1360: 509.8 -> 500.5 us).
template <int kStage>
struct BwdSumSmem {
  float4 g[kStage][kTilePixels];  // dL/dC of the staged tiles (r, g, b, 0)
  float4 rec[kBwdThreads][3];          // the chunk's records
  int gid[kBwdThreads];
  int slot[kBwdThreads];               // index of the pair's tile among the chunk's tiles
  int tiles[kBwdThreads];              // the chunk's distinct tiles, in order
  int perm[kBwdThreads];               // processing order (similar boxes side by side)
  unsigned int bucket[256];
  unsigned int split_end[8];           // per warp: the largest bucket end within the split budget
  int ntiles;
};

__device__ __forceinline__ int block_inclusive_count_256(int flag, int* total, int* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned int b = __ballot_sync(0xffffffffu, flag != 0);
  const int in_warp = __popc(b & ((2u << lane) - 1u));
  if (lane == 31) warp_tot[warp] = __popc(b);
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const int v = warp_tot[w];
    if (w < warp) before += v;
    all += v;
  }
  __syncthreads();
  *total = all;
  return before + in_warp;
}

// One block's rounds of the sum backward (k_render_bwd_sum) over chunks of
// kChunkPairs consecutive (tile, Gaussian) pairs.  kSplit: threads per pair
// -- 1 (chunks of 256), 2 (chunks of 128), or kHybrid (one round, a chunk
// of 128 < kChunkPairs <= 256 pairs: up to 256 - kChunkPairs of its largest
// pairs get two threads each, the others one, so that few threads idle).
constexpr int kHybrid = 3;
template <bool kAbs, int kSplit, int kStageTiles>
__device__ __forceinline__ void bwd_sum_rounds(BwdSumSmem<kStageTiles>& sm, int* warp_tot, const gs2d_config& c,
                                               int tiles_x, int n_gauss, long long n,
                                               const Header* __restrict__ hdr,
                                               const unsigned char* __restrict__ ws,
                                               const float4* __restrict__ rec,
                                               const int4* __restrict__ rect,
                                               const int* __restrict__ sorted_gid,
                                               const int* __restrict__ offsets,
                                               const float* __restrict__ d_image,
                                               float4* __restrict__ partials, int kChunkPairs) {
  const int tid = threadIdx.x;
  const unsigned int* keys = reinterpret_cast<const unsigned int*>(ws + hdr->keys_final);
  for (long long k0 = (long long)blockIdx.x * kChunkPairs; k0 < n;
       k0 += (long long)gridDim.x * kChunkPairs) {
    const long long k = k0 + tid;
    const bool valid = tid < kChunkPairs && k < n;
    int tile = valid ? int(keys[k]) : -1;
    if (valid && !check_ok(tile >= 0 && tile < tiles_x * ((c.height + kTile - 1) / kTile), kCheckTile))
      tile = 0;
    const int prev = (valid && tid > 0) ? int(keys[k - 1]) : -2;
    // the pair's Gaussian index and record, loaded before the block-wide
    // count below so that their round trips overlap the key loads and the
    // count's barriers (768x512: 23.4 -> 21.3 us traced)
    int gid = 0;
    float4 p0 = make_float4(0.f, 0.f, 0.f, 0.f), p1 = p0, p2 = p0;
    if (valid) {
      gid = sorted_gid[k];
      if (!check_ok(gid >= 0 && gid < n_gauss, kCheckGaussian)) gid = 0;
      const float4* r = rec + 3 * size_t(gid);
      p0 = r[0];
      p1 = r[1];
      p2 = r[2];
    }
    int ntiles;
    const int slot = block_inclusive_count_256(valid && tile != prev, &ntiles, warp_tot) - 1;
    if (valid && tile != prev) sm.tiles[slot] = tile;
    int key = 255;  // sort key: boxes of the same shape (h, w) side by side, largest first
    if (valid) {
      sm.rec[tid][0] = p0;
      sm.rec[tid][1] = p1;
      sm.rec[tid][2] = p2;
      const int X0 = (tile % tiles_x) * kTile, Y0 = (tile / tiles_x) * kTile;
      const unsigned int bx = __float_as_uint(p2.x), by = __float_as_uint(p2.y);
      const int w = min(int(box_hi(bx)), X0 + kTile - 1) - max(int(box_lo(bx)), X0) + 1;
      const int h = min(int(box_hi(by)), Y0 + kTile - 1) - max(int(box_lo(by)), Y0) + 1;
      key = (kTile - h) * kTile + (kTile - w);
    }
    if (tid < kChunkPairs) {
      sm.gid[tid] = gid;
      sm.slot[tid] = slot;
    }
    sm.bucket[tid] = 0u;
    __syncthreads();
    // kHybrid: how many of the sorted pairs get two threads.  At most
    // 256 - chunk, and only whole shape buckets, so that the choice does not
    // depend on the (atomic) order of the pairs inside a bucket: results stay
    // bit-reproducible.
    int nsplit = kSplit == kHybrid ? kBwdThreads - kChunkPairs : 0;
    if (ntiles <= kStageTiles) {
      if (tid < kChunkPairs) atomicAdd(&sm.bucket[key], 1u);
      __syncthreads();
      // exclusive scan of the 256 bucket counts, one per thread
      const unsigned int cnt = sm.bucket[tid];
      unsigned int incl = cnt;
      const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) warp_tot[warp] = int(incl);
      __syncthreads();
      unsigned int before = 0;
#pragma unroll
      for (int w = 0; w < 8; ++w)
        if (w < warp) before += unsigned(warp_tot[w]);
      __syncthreads();
      sm.bucket[tid] = before + incl - cnt;
      if constexpr (kSplit == kHybrid) {
        const unsigned int end = before + incl;  // where bucket tid ends in sorted order
        unsigned int e = end <= unsigned(nsplit) ? end : 0u;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) e = max(e, __shfl_xor_sync(0xffffffffu, e, o));
        if (lane == 0) sm.split_end[warp] = e;
      }
      __syncthreads();
      if constexpr (kSplit == kHybrid) {
        unsigned int e = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) e = max(e, sm.split_end[w]);
        nsplit = int(e);
      }
      if (tid < kChunkPairs) {
        const unsigned int pos = atomicAdd(&sm.bucket[key], 1u);
        sm.perm[pos] = tid;
      }
    } else {
      if (tid < kChunkPairs) sm.perm[tid] = tid;
    }
    __syncthreads();

    const size_t HW = size_t(c.width) * c.height;
    const float kk = __fmul_rn(c.cutoff_sigma, c.cutoff_sigma);
    // the pair this thread walks (perm: the shape sort's order, largest
    // boxes first), which of its rows (half), and the row step
    int me = 0, half = 0, step = 1;
    bool in_chunk = true;
    if (kSplit == 1) {
      me = sm.perm[tid];
    } else if (kSplit == 2 || tid < 2 * nsplit) {
      me = sm.perm[tid >> 1];
      half = tid & 1;
      step = 2;
    } else {
      in_chunk = tid - nsplit < kChunkPairs;  // the threads left over idle
      me = in_chunk ? sm.perm[tid - nsplit] : 0;
    }
    const bool mine_valid = in_chunk && (k0 + me) < n;
    for (int t0 = 0; t0 < ntiles; t0 += kStageTiles) {
      const int nst = min(kStageTiles, ntiles - t0);
      for (int q = tid; q < nst * kTilePixels; q += kBwdThreads) {
        const int s = q >> 8, pp = q & 255;
        const int t = sm.tiles[t0 + s];
        const int x = (t % tiles_x) * kTile + (pp & 15), y = (t / tiles_x) * kTile + (pp >> 4);
        float4 g = make_float4(0.f, 0.f, 0.f, 0.f);
        if (x < c.width && y < c.height) {
          const size_t o = size_t(y) * c.width + x;
          g = make_float4(d_image[o], d_image[HW + o], d_image[2 * HW + o], 0.f);
        }
        sm.g[s][pp] = g;
      }
      __syncthreads();
      const int ms = sm.slot[me] - t0;
      const bool act = mine_valid && ms >= 0 && ms < nst;
      float sr = 0.f, sg = 0.f, sb = 0.f, Sx = 0.f, Sy = 0.f, Sxx = 0.f, Sxy = 0.f, Syy = 0.f;
      float ax = 0.f, ay = 0.f;
      int tx = 0, ty = 0;
      float A = 0.f, B = 0.f, C = 0.f;
      if (act) {
        const int t = sm.tiles[t0 + ms];
        tx = t % tiles_x; ty = t / tiles_x;
        const int X0 = tx * kTile, Y0 = ty * kTile;
        const float4 p0 = sm.rec[me][0], p1 = sm.rec[me][1], p2 = sm.rec[me][2];
        const float mx = p0.x, my = p0.y, B2 = 2.0f * p0.w;
        A = p0.z; B = p0.w; C = p1.x;
        const unsigned int bx = __float_as_uint(p2.x), by = __float_as_uint(p2.y);
        const int xa = max(int(box_lo(bx)), X0), xb = min(int(box_hi(bx)), X0 + kTile - 1);
        const int ya = max(int(box_lo(by)), Y0), yb = min(int(box_hi(by)), Y0 + kTile - 1);
        const float4* gt = sm.g[ms];
        for (int y = ya + half; y <= yb; y += (kSplit == kHybrid ? step : kSplit)) {
          const float dy = __fsub_rn(float(y) + 0.5f, my);
          const float b2dy = __fmul_rn(B2, dy);
          const float cdydy = __fmul_rn(__fmul_rn(C, dy), dy);
          const float bdy = B * dy, cdy = C * dy;
          float r0 = 0.f, rx = 0.f, rxx = 0.f;
          int gi = (y - Y0) * kTile + (xa - X0);
          float pxf = float(xa) + 0.5f;
  #pragma unroll 2
          for (int x = xa; x <= xb; ++x, ++gi, pxf += 1.0f) {
            const float dx = __fsub_rn(pxf, mx);
            const float q = __fmaf_rn(dx, __fmaf_rn(A, dx, b2dy), cdydy);
            float w = ex2_approx(q * kNegHalfLog2e);
            w = (q <= kk) ? w : 0.f;
            const float4 g = gt[gi];
            sr = fmaf(g.x, w, sr);
            sg = fmaf(g.y, w, sg);
            sb = fmaf(g.z, w, sb);
            const float t = w * fmaf(g.x, p1.y, fmaf(g.y, p1.z, g.z * p1.w));
            r0 += t;
            const float tdx = t * dx;
            rx += tdx;
            rxx = fmaf(tdx, dx, rxx);
            if constexpr (kAbs) {
              ax += fabsf(t * fmaf(A, dx, bdy));
              ay += fabsf(t * fmaf(B, dx, cdy));
            }
          }
          Sx += rx;
          Sy = fmaf(r0, dy, Sy);
          Sxx += rxx;
          Sxy = fmaf(rx, dy, Sxy);
          Syy = fmaf(r0 * dy, dy, Syy);
        }
      }
      if constexpr (kSplit != 1) {  // a split pair's two halves: even rows + odd rows
        float* vv[10] = {&sr, &sg, &sb, &Sx, &Sy, &Sxx, &Sxy, &Syy, &ax, &ay};
#pragma unroll
        for (int u = 0; u < (kAbs ? 10 : 8); ++u) {
          const float o = __shfl_xor_sync(0xffffffffu, *vv[u], 1);
          if (step == 2) *vv[u] += o;
        }
      }
      if (act && half == 0) {
        const int gid_me = sm.gid[me];
        const int4 rc = rect[gid_me];
        const int pslot = offsets[gid_me] + (ty - rc.y) * (rc.z - rc.x + 1) + (tx - rc.x);
        if (check_ok(pslot >= 0 && pslot < n, kCheckPartial)) {
          float4* out = partials + (kAbs ? 3 : 2) * size_t(pslot);
          out[0] = make_float4(fmaf(A, Sx, B * Sy), fmaf(B, Sx, C * Sy), -0.5f * Sxx, -Sxy);
          out[1] = make_float4(-0.5f * Syy, sr, sg, sb);
          if constexpr (kAbs) out[2] = make_float4(0.f, ax, ay, 0.f);
        }
      }
      __syncthreads();
    }
  }
}

// Sum mode: one thread per (tile, Gaussian) pair (or two, see below),
// walking exactly the pixels of the Gaussian's box inside the tile.  Blocks
// take fixed chunks of the sorted pair list, whatever the tile boundaries,
// so heavy tiles spread over many blocks; inside a block the pairs are
// reordered so that lanes of a warp walk boxes of the same shape.  The
// chunk length follows the pair count P and the grid G (4 blocks per SM):
//   P <= 128 G:  two adjacent threads share each pair, one taking its even
//                rows and one its odd rows, and add their sums with one
//                shuffle (fixed order); 128-pair chunks;
//   P <= 256 G:  chunks of ceil(P / G) pairs, so that every block has
//                exactly one round (measured on a B300 at 768x512 / 50K
//                Gaussians, 117K pairs: 25.4 -> 23.4 us against two threads
//                per pair in 1.55 rounds); up to 256 - chunk of the largest
//                pairs (whole shape buckets) get two threads each and the
//                rest one, so few threads idle (step 65.8 -> 64.1 us);
//   otherwise:   one thread per pair, 256-pair chunks.  kAbs: also the absgrad sums over the pair's
// pixels of |t (A dx + B dy)| and |t (B dx + C dy)| (each pixel's share of
// dL/dmu in absolute value), in a third float4 of the pair's slot.
template <bool kAbs, int kStage>
__global__ void __launch_bounds__(kBwdThreads, 4)  // 4 per SM: measured best (5 or 6 spill and lose)
k_render_bwd_sum(gs2d_config c, int tiles_x, int n_gauss, const Header* __restrict__ hdr,
                 const unsigned char* __restrict__ ws, const float4* __restrict__ rec,
                 const int4* __restrict__ rect, const int* __restrict__ sorted_gid,
                 const int* __restrict__ offsets, const float* __restrict__ d_image,
                 float4* __restrict__ partials) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  BwdSumSmem<kStage>& sm = *reinterpret_cast<BwdSumSmem<kStage>*>(smem_raw);
  __shared__ int warp_tot[8];
  const unsigned int f = hdr->flags;
  const long long n = (f & (GS2D_FLAG_CAPACITY | GS2D_FLAG_OVERFLOW | GS2D_FLAG_TIMEOUT)) ? 0
                      : hdr->pairs;
  const long long G = gridDim.x;
  if (n <= G * (kBwdThreads / 2))
    bwd_sum_rounds<kAbs, 2, kStage>(sm, warp_tot, c, tiles_x, n_gauss, n, hdr, ws, rec, rect, sorted_gid,
                            offsets, d_image, partials, kBwdThreads / 2);
  else if (n <= G * kBwdThreads)
    bwd_sum_rounds<kAbs, kHybrid, kStage>(sm, warp_tot, c, tiles_x, n_gauss, n, hdr, ws, rec, rect,
                                  sorted_gid, offsets, d_image, partials, int((n + G - 1) / G));
  else
    bwd_sum_rounds<kAbs, 1, kStage>(sm, warp_tot, c, tiles_x, n_gauss, n, hdr, ws, rec, rect, sorted_gid,
                            offsets, d_image, partials, kBwdThreads);
}

constexpr int kBwdCompThreads = 256;

// Composite: one block per tile, one pixel per thread (8x4 sub-block per
// warp as in the forward), walking the tile's list back to front from each
// pixel's last contributor (comp_tile_backward).
template <bool kAbs>
__global__ void __launch_bounds__(kBwdCompThreads)
k_render_bwd_comp(gs2d_config c, int tiles_x, int n, const Header* __restrict__ hdr,
                  const float4* __restrict__ rec,
                  const int4* __restrict__ rect, const int2* __restrict__ ranges,
                  const int* __restrict__ sorted_gid, const int* __restrict__ offsets,
                  const float* __restrict__ bg, const float* __restrict__ t_final,
                  const int* __restrict__ last, const float* __restrict__ d_image,
                  float4* __restrict__ partials, float4* __restrict__ tile_partials,
                  const int4* __restrict__ order) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  CompStage<kAbs>& sm = *reinterpret_cast<CompStage<kAbs>*>(smem_raw);
  int2 rg;
  const int tile = tile_of_slot(order, int(blockIdx.x), ranges, tiles_x * ((c.height + kTile - 1) / kTile), &rg);  // longest lists first when known
  if (!check_ok(tile >= 0 && tile < tiles_x * ((c.height + kTile - 1) / kTile), kCheckTile) || tile < 0) return;
  const long long pairs = hdr->pairs;
  if (!check_ok(rg.x >= 0 && rg.x <= rg.y && rg.y <= pairs, kCheckRange)) rg = make_int2(0, 0);
  const int tx = tile % tiles_x, ty = tile / tiles_x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bx0 = tx * kTile + (warp & 1) * 8;
  const int by0 = ty * kTile + (warp >> 1) * 4;
  const int px = bx0 + (lane & 7), py = by0 + (lane >> 3);
  const bool inside = px < c.width && py < c.height;
  const float kk = __fmul_rn(c.cutoff_sigma, c.cutoff_sigma);
  const size_t HW = size_t(c.width) * c.height;
  float T = 1.f, gr = 0.f, gg = 0.f, gb = 0.f;
  int lst = 0;
  if (inside) {
    const size_t p = size_t(py) * c.width + px;
    T = t_final[p];
    lst = last[p];
    gr = d_image[p];
    gg = d_image[HW + p];
    gb = d_image[2 * HW + p];
  }
  comp_tile_backward<kAbs>(sm, c, tile, tx, ty, rg, bx0, by0, float(px) + 0.5f, float(py) + 0.5f,
                           inside, kk, T, lst, gr, gg, gb, n, pairs, bg, rec, rect, sorted_gid,
                           offsets, partials, tile_partials);
}

}  // namespace

namespace {

template <bool kAbs>
cudaError_t launch_bwd_pairs(const gs2d_config& c, int n, const Layout& L, const float4* r, const int4* rc,
                             const int2* rg, const int* sorted_gid, const float* bg,
                             const float* t_final, const int* last, const float* d_image,
                             unsigned char* ws, cudaStream_t s) {
  const int T = num_tiles(c);
  const int* offsets = reinterpret_cast<const int*>(ws + L.offsets);
  float4* partials = reinterpret_cast<float4*>(ws + L.partials);
  if (c.mode == GS2D_MODE_COMPOSITE) {
    const size_t smem = sizeof(CompStage<kAbs>);
    auto kern = k_render_bwd_comp<kAbs>;
    GS2D_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
    GS2D_TRY(launch(kern, dim3(T), dim3(kBwdCompThreads), smem, s, c, tiles_x(c), n,
                    reinterpret_cast<const Header*>(ws), r, rc, rg, sorted_gid, offsets, bg, t_final, last, d_image, partials,
                    reinterpret_cast<float4*>(ws + L.tile_partials),
                    L.count_sort ? reinterpret_cast<const int4*>(ws + L.tile_order) : nullptr));
  } else {
    const bool wide = T > kCountSortMaxTiles;
    const size_t smem = wide ? sizeof(BwdSumSmem<4>) : sizeof(BwdSumSmem<8>);
    auto kern = wide ? k_render_bwd_sum<kAbs, 4> : k_render_bwd_sum<kAbs, 8>;
    GS2D_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
    GS2D_TRY(launch(kern, dim3(4 * sm_count()), dim3(kBwdThreads), smem, s, c, tiles_x(c), n,
                    reinterpret_cast<const Header*>(ws), static_cast<const unsigned char*>(ws), r, rc,
                    sorted_gid, offsets, d_image, partials));
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_render_bwd(const gs2d_config& c, int n, const float* chol,
                              const gs2d_record* rec, const int* rect, const int* ranges,
                              const int* sorted_gid, const float* bg, const float* t_final,
                              const int* last, const float* d_image, float* d_xy, float* d_chol,
                              float* d_rgb, float* d_opacity, float* d_bg, float* d_xy_abs,
                              unsigned char* ws, cudaStream_t s, float* loss, int loss_blocks) {
  const Layout L = layout_of(c, n, 0);
  const float4* r = reinterpret_cast<const float4*>(rec);
  const int4* rc = reinterpret_cast<const int4*>(rect);
  const int2* rg = reinterpret_cast<const int2*>(ranges);
  if (d_xy_abs)
    GS2D_TRY(launch_bwd_pairs<true>(c, n, L, r, rc, rg, sorted_gid, bg, t_final, last, d_image, ws, s));
  else
    GS2D_TRY(launch_bwd_pairs<false>(c, n, L, r, rc, rg, sorted_gid, bg, t_final, last, d_image, ws, s));
  return launch_gather(c, n, chol, rec, rect, ws, d_xy, d_chol, d_rgb, d_opacity, d_bg, d_xy_abs,
                       loss, loss_blocks, s);
}

GS2D_CHECK_WORD_READER(raster_bwd)

}  // namespace gs2d
