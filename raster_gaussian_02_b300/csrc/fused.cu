// Fused training pass: render, L2 loss and backward (FlashImgs README,
// Project Structure: training-time rasterization with fused forward/backward).
// dL/dC = 2 (C - target) / (3HW) is formed at each pixel as soon as the
// pixel's colour is known, so no separate loss pass reads the image back.
// Results equal the separate forward, loss and backward calls up to the
// order of floating-point additions; the per-pair partials go to the same
// emission slots and the same gather kernel sums them per Gaussian.
//
// Composite: one block per tile runs the forward and the backward bodies
// back to back, the pixel's transmittance, last contributor and dL/dC kept
// in registers; neither dL/dC nor (image NULL) the image touches memory.
// Sum: the forward also takes the loss and writes dL/dC to the workspace,
// then the pair-parallel backward runs.  (A per-tile sum backward, one warp
// per pair with dL/dC kept in shared memory, measured 1.4-1.8x slower on a
// B300: every pair ends in a serial shuffle reduction and a dependent
// load, and the tile's pairs cannot spread over other SMs.)
#include "tile_bodies.cuh"

namespace gs2d {

namespace {

template <bool kAbs>
struct FusedCompSmem {
  union {
    CompSmem f;
    CompStage<kAbs> b;
  } u;
  float red[8];
};

// A tile whose list is longer than kCompSegLen entries gets a second block.
// Both render the tile (the forward, and with it every touch and termination
// decision, is the same in each); then block 0 back-propagates the back
// half of the list and block 1 the front half, starting from the
// transmittance and colour its forward recorded at the midpoint.  The
// longest lists' serial chains, which set this kernel's length, lose half
// their backward part.  Each block writes the pair slots of its own half;
// block 0 also writes the image, the loss and the background partial.
// Measured on a B300 at 768x512 / 50K Gaussians (lists up to ~500 entries):
// 129.9 us unsplit; split above 96 / 128 / 192 / 256 / 320 / 384 entries:
// 121.7 / 119.6 / 113.5 / 109.4 / 111.4 / 125.8 us; three or four parts per
// long list were slower (the extra forwards cost more than the shorter
// backward chains save).  The code takes K = ceil(len / kCompSegLen) parts,
// at most kCompMaxParts.
constexpr int kCompSegLen = 256;
constexpr int kCompMaxParts = 2;

template <bool kAbs>
__global__ void __launch_bounds__(256)
k_fused_comp(gs2d_config c, int tiles_x, int n, const Header* __restrict__ hdr, float scale,
             const float4* __restrict__ rec,
             const int4* __restrict__ rect, const int2* __restrict__ ranges,
             const int* __restrict__ sorted_gid, const int* __restrict__ offsets,
             const float* __restrict__ bg, const float* __restrict__ target,
             float* __restrict__ image, float4* __restrict__ partials,
             float4* __restrict__ tile_partials, float* __restrict__ loss_partials,
             const int4* __restrict__ order) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  FusedCompSmem<kAbs>& sm = *reinterpret_cast<FusedCompSmem<kAbs>*>(smem_raw);
  // kCompMaxParts blocks per tile (its parts), longest lists first when known;
  // the parts of one tile have adjacent block indices
  const int part = int(blockIdx.x % kCompMaxParts);
  int2 rg;
  const int tile = tile_of_slot(order, int(blockIdx.x / kCompMaxParts), ranges, tiles_x * ((c.height + kTile - 1) / kTile), &rg);
  if (!check_ok(tile >= 0 && tile < tiles_x * ((c.height + kTile - 1) / kTile), kCheckTile) || tile < 0) return;
  const int tx = tile % tiles_x, ty = tile / tiles_x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bx0 = tx * kTile + (warp & 1) * 8;
  const int by0 = ty * kTile + (warp >> 1) * 4;
  const int px = bx0 + (lane & 7), py = by0 + (lane >> 3);
  const float pxf = float(px) + 0.5f, pyf = float(py) + 0.5f;
  const bool inside = px < c.width && py < c.height;
  const float kk = __fmul_rn(c.cutoff_sigma, c.cutoff_sigma);
  const long long pairs = hdr->pairs;
  if (!check_ok(rg.x >= 0 && rg.x <= rg.y && rg.y <= pairs, kCheckRange)) rg = make_int2(0, 0);
  const int len = rg.y - rg.x;
  const int parts = min(kCompMaxParts, max(1, (len + kCompSegLen - 1) / kCompSegLen));
  if (part >= parts) return;  // the whole block: no barrier reached yet
  // this block's segment [lo, hi) of the list, segments counted from the back
  const int lo = int((long long)(parts - 1 - part) * len / parts);
  const int hi = int((long long)(parts - part) * len / parts);
  // every thread has passed its last read of the forward's staging area when
  // comp_tile_forward returns (each round ends at a block barrier)
  const CompFwdOut o = comp_tile_forward<true>(sm.u.f, c, rg, bx0, by0, pxf, pyf, inside, kk, n, rec,
                                               sorted_gid, part > 0 ? hi : 0x7fffffff);
  float er = 0.f, eg = 0.f, eb = 0.f;
  if (inside) {
    const size_t HW = size_t(c.width) * c.height;
    const size_t p = size_t(py) * c.width + px;
    float ar = o.r, ag = o.g, ab = o.b;
    if (bg) {
      ar = fmaf(o.T, bg[0], ar);
      ag = fmaf(o.T, bg[1], ag);
      ab = fmaf(o.T, bg[2], ab);
    }
    if (image && part == 0) {
      image[p] = ar;
      image[HW + p] = ag;
      image[2 * HW + p] = ab;
    }
    er = ar - target[p];
    eg = ag - target[HW + p];
    eb = ab - target[2 * HW + p];
  }
  if (part == 0) {
    const float tl = block_sum_ordered<8>(fmaf(eb, eb, fmaf(eg, eg, er * er)), sm.red);
    if (threadIdx.x == 0) loss_partials[tile] = tl;
    // the whole list, or its back segment [lo, len)
    comp_tile_backward<kAbs>(sm.u.b, c, tile, tx, ty, rg, bx0, by0, pxf, pyf, inside, kk, o.T, o.last,
                             er * scale, eg * scale, eb * scale, n, pairs, bg, rec, rect, sorted_gid,
                             offsets, partials, tile_partials, lo);
  } else {
    // an earlier segment [lo, hi): behind it lie the transmittance the forward
    // recorded at hi and the colour the later segments and the background add
    float Sr = 0.f, Sg = 0.f, Sb = 0.f;
    if (inside) {
      const float fr = bg ? fmaf(o.T, bg[0], o.r) : o.r, fg = bg ? fmaf(o.T, bg[1], o.g) : o.g,
                  fb = bg ? fmaf(o.T, bg[2], o.b) : o.b;
      Sr = fr - o.mr;
      Sg = fg - o.mg;
      Sb = fb - o.mb;
    }
    comp_tile_backward<kAbs>(sm.u.b, c, tile, tx, ty, rg, bx0, by0, pxf, pyf, inside, kk, o.Tm, o.last,
                             er * scale, eg * scale, eb * scale, n, pairs, bg, rec, rect, sorted_gid,
                             offsets, partials, tile_partials, lo, hi, false, Sr, Sg, Sb);
  }
}

}  // namespace

cudaError_t launch_render_fused_l2(const gs2d_config& c, int n, const float* chol,
                                   const gs2d_record* rec, const int* rect, const int* ranges,
                                   const int* sorted_gid, const float* bg, const float* target,
                                   float* image, float* loss, float* d_xy, float* d_chol,
                                   float* d_rgb, float* d_opacity, float* d_bg, float* d_xy_abs,
                                   unsigned char* ws, cudaStream_t s) {
  const Layout L = layout_of(c, n, 0);
  const int T = num_tiles(c);
  const float4* r = reinterpret_cast<const float4*>(rec);
  const int4* rc = reinterpret_cast<const int4*>(rect);
  const int2* rg = reinterpret_cast<const int2*>(ranges);
  const int* offsets = reinterpret_cast<const int*>(ws + L.offsets);
  float4* tp = reinterpret_cast<float4*>(ws + L.tile_partials);
  // the same scale as the L2 loss kernel: 2 / (3HW)
  const float scale = float(2.0 / (3.0 * double(c.width) * double(c.height)));
  float* lp = reinterpret_cast<float*>(ws + L.loss_partials);
  if (c.mode == GS2D_MODE_COMPOSITE) {
    auto go = [&](auto kern, size_t smem) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
      if (e != cudaSuccess) return e;
      return launch(kern, dim3(kCompMaxParts * T), dim3(256), smem, s, c, tiles_x(c), n,
                    reinterpret_cast<const Header*>(ws), scale, r, rc, rg, sorted_gid,
                    offsets, bg, target, image, reinterpret_cast<float4*>(ws + L.partials), tp, lp,
                    L.count_sort ? reinterpret_cast<const int4*>(ws + L.tile_order) : nullptr);
    };
    if (d_xy_abs)
      GS2D_TRY(go(k_fused_comp<true>, sizeof(FusedCompSmem<true>)));
    else
      GS2D_TRY(go(k_fused_comp<false>, sizeof(FusedCompSmem<false>)));
    return launch_gather(c, n, chol, rec, rect, ws, d_xy, d_chol, d_rgb, d_opacity, d_bg, d_xy_abs,
                         loss, T, s);
  }
  float* d_image = reinterpret_cast<float*>(ws + L.dimage);
  int blocks = 0;
  // the counting sort leaves a longest-first launch order of the tiles
  const int4* order = L.count_sort ? reinterpret_cast<const int4*>(ws + L.tile_order) : nullptr;
  GS2D_TRY(launch_render_fwd_loss(c, n, rec, ranges, sorted_gid, target, scale, image, d_image, lp, &blocks,
                                  order, s));
  return launch_render_bwd(c, n, chol, rec, rect, ranges, sorted_gid, nullptr, nullptr, nullptr, d_image,
                           d_xy, d_chol, d_rgb, nullptr, nullptr, d_xy_abs, ws, s, loss, blocks);
}

GS2D_CHECK_WORD_READER(fused)

}  // namespace gs2d
