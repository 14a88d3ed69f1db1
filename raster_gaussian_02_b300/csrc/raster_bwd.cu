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
#include "gs2d_internal.cuh"

namespace gs2d {

namespace {

constexpr int kChunkPairs = 256;   // pairs per block, one per thread
constexpr int kStageTiles = 8;     // tiles of dL/dC staged at a time

struct BwdSumSmem {
  float4 g[kStageTiles][kTilePixels];  // dL/dC of the staged tiles (r, g, b, 0)
  float4 rec[kChunkPairs][3];          // the chunk's records
  int gid[kChunkPairs];
  int slot[kChunkPairs];               // index of the pair's tile among the chunk's tiles
  int tiles[kChunkPairs];              // the chunk's distinct tiles, in order
  int perm[kChunkPairs];               // processing order (similar boxes side by side)
  unsigned int bucket[256];
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

// Sum mode: one thread per (tile, Gaussian) pair, walking exactly the pixels
// of the Gaussian's box inside the tile.  Blocks take fixed chunks of the
// sorted pair list, whatever the tile boundaries, so heavy tiles spread over
// many blocks; inside a block the pairs are reordered so that lanes of a
// warp walk boxes of the same shape.
__global__ void __launch_bounds__(kChunkPairs)
k_render_bwd_sum(gs2d_config c, int tiles_x, const Header* __restrict__ hdr,
                 const unsigned char* __restrict__ ws, const float4* __restrict__ rec,
                 const int4* __restrict__ rect, const int* __restrict__ sorted_gid,
                 const int* __restrict__ offsets, const float* __restrict__ d_image,
                 float4* __restrict__ partials) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  BwdSumSmem& sm = *reinterpret_cast<BwdSumSmem*>(smem_raw);
  __shared__ int warp_tot[8];
  const int tid = threadIdx.x;
  const unsigned int f = hdr->flags;
  const long long n = (f & (GS2D_FLAG_CAPACITY | GS2D_FLAG_OVERFLOW | GS2D_FLAG_TIMEOUT)) ? 0
                      : hdr->pairs;
  const unsigned int* keys = reinterpret_cast<const unsigned int*>(ws + hdr->keys_final);
  for (long long k0 = (long long)blockIdx.x * kChunkPairs; k0 < n;
       k0 += (long long)gridDim.x * kChunkPairs) {
    const long long k = k0 + tid;
    const bool valid = k < n;
    const int tile = valid ? int(keys[k]) : -1;
    const int prev = (valid && tid > 0) ? int(keys[k - 1]) : -2;
    int ntiles;
    const int slot = block_inclusive_count_256(valid && tile != prev, &ntiles, warp_tot) - 1;
    if (valid && tile != prev) sm.tiles[slot] = tile;
    int gid = 0;
    int key = 255;  // sort key: boxes of the same shape (h, w) side by side, largest first
    if (valid) {
      gid = sorted_gid[k];
      const float4* r = rec + 3 * size_t(gid);
      const float4 p0 = r[0], p1 = r[1], p2 = r[2];
      sm.rec[tid][0] = p0;
      sm.rec[tid][1] = p1;
      sm.rec[tid][2] = p2;
      const int X0 = (tile % tiles_x) * kTile, Y0 = (tile / tiles_x) * kTile;
      const unsigned int bx = __float_as_uint(p2.x), by = __float_as_uint(p2.y);
      const int w = min(int(box_hi(bx)), X0 + kTile - 1) - max(int(box_lo(bx)), X0) + 1;
      const int h = min(int(box_hi(by)), Y0 + kTile - 1) - max(int(box_lo(by)), Y0) + 1;
      key = (kTile - h) * kTile + (kTile - w);
    }
    sm.gid[tid] = gid;
    sm.slot[tid] = slot;
    sm.bucket[tid] = 0u;
    __syncthreads();
    if (ntiles <= kStageTiles) {
      atomicAdd(&sm.bucket[key], 1u);
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
      __syncthreads();
      const unsigned int pos = atomicAdd(&sm.bucket[key], 1u);
      sm.perm[pos] = tid;
    } else {
      sm.perm[tid] = tid;
    }
    __syncthreads();

    const size_t HW = size_t(c.width) * c.height;
    const float kk = __fmul_rn(c.cutoff_sigma, c.cutoff_sigma);
    const int me = sm.perm[tid];
    const bool mine_valid = (k0 + me) < n;
    for (int t0 = 0; t0 < ntiles; t0 += kStageTiles) {
      const int nst = min(kStageTiles, ntiles - t0);
      for (int q = tid; q < nst * kTilePixels; q += kChunkPairs) {
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
      if (mine_valid && ms >= 0 && ms < nst) {
        const int t = sm.tiles[t0 + ms];
        const int tx = t % tiles_x, ty = t / tiles_x;
        const int X0 = tx * kTile, Y0 = ty * kTile;
        const float4 p0 = sm.rec[me][0], p1 = sm.rec[me][1], p2 = sm.rec[me][2];
        const float mx = p0.x, my = p0.y, A = p0.z, B = p0.w, B2 = 2.0f * p0.w, C = p1.x;
        const unsigned int bx = __float_as_uint(p2.x), by = __float_as_uint(p2.y);
        const int xa = max(int(box_lo(bx)), X0), xb = min(int(box_hi(bx)), X0 + kTile - 1);
        const int ya = max(int(box_lo(by)), Y0), yb = min(int(box_hi(by)), Y0 + kTile - 1);
        const float4* gt = sm.g[ms];
        float sr = 0.f, sg = 0.f, sb = 0.f, Sx = 0.f, Sy = 0.f, Sxx = 0.f, Sxy = 0.f, Syy = 0.f;
        for (int y = ya; y <= yb; ++y) {
          const float dy = __fsub_rn(float(y) + 0.5f, my);
          const float b2dy = __fmul_rn(B2, dy);
          const float cdydy = __fmul_rn(__fmul_rn(C, dy), dy);
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
          }
          Sx += rx;
          Sy = fmaf(r0, dy, Sy);
          Sxx += rxx;
          Sxy = fmaf(rx, dy, Sxy);
          Syy = fmaf(r0 * dy, dy, Syy);
        }
        const int gid_me = sm.gid[me];
        const int4 rc = rect[gid_me];
        const int pslot = offsets[gid_me] + (ty - rc.y) * (rc.z - rc.x + 1) + (tx - rc.x);
        float4* out = partials + 2 * size_t(pslot);
        out[0] = make_float4(fmaf(A, Sx, B * Sy), fmaf(B, Sx, C * Sy), -0.5f * Sxx, -Sxy);
        out[1] = make_float4(-0.5f * Syy, sr, sg, sb);
      }
      __syncthreads();
    }
  }
}

constexpr int kBwdCompThreads = 256;
constexpr int kCompChunk = 128;
constexpr int kCompVals = 9;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Butterfly reduce-scatter of eight per-lane values over the warp: returns,
// in every lane, the warp total of value ((lane >> 2) & 7) in the order
// v[0..7] (lane bit 4 picks values 4-7, bit 3 values +2, bit 2 values +1).
__device__ __forceinline__ float warp_reduce_scatter8(const float (&v)[8], int lane) {
  float a[4], b[2];
  const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = u16 ? v[i + 4] : v[i], send = u16 ? v[i] : v[i + 4];
    a[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = u8 ? a[i + 2] : a[i], send = u8 ? a[i] : a[i + 2];
    b[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  float c = (u4 ? b[1] : b[0]) + __shfl_xor_sync(0xffffffffu, u4 ? b[0] : b[1], 4);
  c += __shfl_xor_sync(0xffffffffu, c, 2);
  c += __shfl_xor_sync(0xffffffffu, c, 1);
  return c;
}

struct CompStage {
  float4 mc[kCompChunk];  // mean_x, mean_y, A, 2B
  float4 cr[kCompChunk];  // C, r, g, b
  uint2 box[kCompChunk];
  float op[kCompChunk];
  int gid[kCompChunk];
  uint2 list[8][kCompChunk];            // (chunk index, lane mask) per warp
  float acc[8][kCompChunk][kCompVals];  // per-warp partials, summed over warps in order
  float bgred[8][3];
};

// Composite: one block per tile, one pixel per thread (8x4 sub-block per
// warp as in the forward), walking the tile's list back to front from each
// pixel's last contributor.  Per (warp, Gaussian) the nine partial
// derivatives are reduced over the warp and kept in a per-warp slot; the
// slots are summed in warp order per chunk entry.
__global__ void __launch_bounds__(kBwdCompThreads)
k_render_bwd_comp(gs2d_config c, int tiles_x, const float4* __restrict__ rec,
                  const int4* __restrict__ rect, const int2* __restrict__ ranges,
                  const int* __restrict__ sorted_gid, const int* __restrict__ offsets,
                  const float* __restrict__ bg, const float* __restrict__ t_final,
                  const int* __restrict__ last, const float* __restrict__ d_image,
                  float4* __restrict__ partials, float4* __restrict__ bg_partials) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  CompStage& sm = *reinterpret_cast<CompStage*>(smem_raw);
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
  const size_t HW = size_t(c.width) * c.height;
  const float bgr = bg ? bg[0] : 0.f, bgg = bg ? bg[1] : 0.f, bgb = bg ? bg[2] : 0.f;
  uint2* list = sm.list[warp];

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
  // background gradient: T_final * g summed over the tile, fixed order
  {
    const float vr = warp_sum(inside ? T * gr : 0.f);
    const float vg = warp_sum(inside ? T * gg : 0.f);
    const float vb = warp_sum(inside ? T * gb : 0.f);
    if (lane == 0) {
      sm.bgred[warp][0] = vr;
      sm.bgred[warp][1] = vg;
      sm.bgred[warp][2] = vb;
    }
    __syncthreads();
    if (tid == 0) {
      float x = 0.f, y = 0.f, z = 0.f;
      for (int w = 0; w < 8; ++w) {
        x += sm.bgred[w][0];
        y += sm.bgred[w][1];
        z += sm.bgred[w][2];
      }
      bg_partials[tile] = make_float4(x, y, z, 0.f);
    }
  }
  float Sr = T * bgr, Sg = T * bgg, Sb = T * bgb;
  const int len = rg.y - rg.x;
  const int nchunks = (len + kCompChunk - 1) / kCompChunk;
  for (int ci = nchunks - 1; ci >= 0; --ci) {
    const int cb = rg.x + ci * kCompChunk;
    const int cnt = min(kCompChunk, rg.y - cb);
    if (tid < cnt) {
      const int gid = sorted_gid[cb + tid];
      const float4* r = rec + 3 * size_t(gid);
      const float4 p0 = r[0], p1 = r[1], p2 = r[2];
      sm.mc[tid] = make_float4(p0.x, p0.y, p0.z, 2.0f * p0.w);
      sm.cr[tid] = p1;
      sm.box[tid] = make_uint2(__float_as_uint(p2.x), __float_as_uint(p2.y));
      sm.op[tid] = p2.z;
      sm.gid[tid] = gid;
    }
    __syncthreads();
    int nl = 0;
    for (int j0 = 0; j0 < cnt; j0 += 32) {
      const int j = j0 + lane;
      unsigned int m = 0;
      if (j < cnt) {
        m = box_lanes(sm.box[j], bx0, by0);
        if (!m)
#pragma unroll
          for (int v = 0; v < kCompVals; ++v) sm.acc[warp][j][v] = 0.f;
      }
      const unsigned int hits = __ballot_sync(0xffffffffu, m != 0u);
      if (m) list[nl + __popc(hits & lt)] = make_uint2(unsigned(j), m);
      nl += __popc(hits);
    }
    __syncwarp();
    for (int e = nl - 1; e >= 0; --e) {
      const uint2 u = list[e];
      const int j = int(u.x);
      const int idx = cb - rg.x + j;  // position in the tile's list
      const float4 mc = sm.mc[j];
      const float4 cr = sm.cr[j];
      const float dx = __fsub_rn(pxf, mc.x);
      const float dy = __fsub_rn(pyf, mc.y);
      const float q = touch_q(dx, dy, mc.z, mc.w, cr.x);
      const bool act = inside && (u.y & bit) && idx < lst && q <= kk;
      float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      float v8 = 0.f;
      if (act) {
        const float o = sm.op[j];
        const float w = ex2_approx(q * kNegHalfLog2e);
        const float alpha = o * w;
        const float inv = 1.0f / (1.0f - alpha);
        const float Tb = T * inv;  // transmittance in front of this Gaussian
        const float aT = alpha * Tb;
        const float dal = gr * (cr.y * Tb - Sr * inv) + gg * (cr.z * Tb - Sg * inv) +
                          gb * (cr.w * Tb - Sb * inv);
        const float t = w * o * dal;
        v[0] = t * dx;
        v[1] = t * dy;
        v[2] = v[0] * dx;
        v[3] = v[0] * dy;
        v[4] = v[1] * dy;
        v[5] = gr * aT;
        v[6] = gg * aT;
        v[7] = gb * aT;
        v8 = dal * w;
        Sr = fmaf(cr.y, aT, Sr);
        Sg = fmaf(cr.z, aT, Sg);
        Sb = fmaf(cr.w, aT, Sb);
        T = Tb;
      }
      if (__any_sync(0xffffffffu, act)) {
        const float tot = warp_reduce_scatter8(v, lane);
        const float tot8 = warp_sum(v8);
        if ((lane & 3) == 0) sm.acc[warp][j][(lane >> 2) & 7] = tot;
        if (lane == 0) sm.acc[warp][j][8] = tot8;
      } else if (lane < kCompVals) {
        sm.acc[warp][j][lane] = 0.f;
      }
    }
    __syncthreads();
    if (tid < cnt) {
      float s[kCompVals];
#pragma unroll
      for (int u = 0; u < kCompVals; ++u) s[u] = 0.f;
      for (int w = 0; w < 8; ++w)
#pragma unroll
        for (int u = 0; u < kCompVals; ++u) s[u] += sm.acc[w][tid][u];
      const int gid = sm.gid[tid];
      const float A = sm.mc[tid].z, B = 0.5f * sm.mc[tid].w, C = sm.cr[tid].x;
      const int4 rc = rect[gid];
      const int slot = offsets[gid] + (ty - rc.y) * (rc.z - rc.x + 1) + (tx - rc.x);
      float4* out = partials + 3 * size_t(slot);
      out[0] = make_float4(fmaf(A, s[0], B * s[1]), fmaf(B, s[0], C * s[1]), -0.5f * s[2], -s[3]);
      out[1] = make_float4(-0.5f * s[4], s[5], s[6], s[7]);
      out[2] = make_float4(s[8], 0.f, 0.f, 0.f);
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_render_bwd(const gs2d_config& c, int n, const float* chol,
                              const gs2d_record* rec, const int* rect, const int* ranges,
                              const int* sorted_gid, const float* bg, const float* t_final,
                              const int* last, const float* d_image, float* d_xy, float* d_chol,
                              float* d_rgb, float* d_opacity, float* d_bg, unsigned char* ws,
                              cudaStream_t s) {
  const Layout L = layout_of(c, n, 0);
  const int T = num_tiles(c);
  const float4* r = reinterpret_cast<const float4*>(rec);
  const int4* rc = reinterpret_cast<const int4*>(rect);
  const int2* rg = reinterpret_cast<const int2*>(ranges);
  const int* offsets = reinterpret_cast<const int*>(ws + L.offsets);
  float4* partials = reinterpret_cast<float4*>(ws + L.partials);
  if (c.mode == GS2D_MODE_COMPOSITE) {
    const size_t smem = sizeof(CompStage);
    cudaError_t e = cudaFuncSetAttribute(k_render_bwd_comp, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    GS2D_TRY(launch(k_render_bwd_comp, dim3(T), dim3(kBwdCompThreads), smem, s, c, tiles_x(c), r, rc, rg, sorted_gid, offsets, bg, t_final, last, d_image, partials,
        reinterpret_cast<float4*>(ws + L.bg_partials)));
  } else {
    const size_t smem = sizeof(BwdSumSmem);
    cudaError_t e = cudaFuncSetAttribute(k_render_bwd_sum, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    GS2D_TRY(launch(k_render_bwd_sum, dim3(4 * sm_count()), dim3(kChunkPairs), smem, s, c, tiles_x(c), reinterpret_cast<const Header*>(ws), ws, r, rc, sorted_gid, offsets,
        d_image, partials));
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_gather(c, n, chol, rec, rect, ws, d_xy, d_chol, d_rgb, d_opacity, d_bg, s);
}

}  // namespace gs2d
