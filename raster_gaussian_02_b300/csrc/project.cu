// Projection (shape parameters -> inverse covariance, 3-sigma pixel box,
// tile rectangle) and its backward (per-pair partial gradients summed per
// Gaussian, then the chain rule from the inverse covariance to the shape).
//
// Sigma = L L^T with L = [[a, 0], [b, c]] (DrawingWithGaussians README,
// MLX-specific notes: lower-triangular L), or Sigma = R diag(s_x^2, s_y^2) R^T
// (FlashImgs README, Python API: project_gaussians_2d_scale_rot; GaussianImage
// project page, the "rs" scripts); the 8 parameters per Gaussian are
// position, covariance and colour (GaussianImage project page, Overview).
#include "gs2d_internal.cuh"

namespace gs2d {

namespace {

__global__ void __launch_bounds__(256)
k_project(gs2d_config c, int n, const float* __restrict__ xy, const float* __restrict__ chol,
          const float* __restrict__ rgb, const float* __restrict__ depth,
          const float* __restrict__ opacity, float4* __restrict__ rec, int4* __restrict__ rect,
          int* __restrict__ count) {
  pdl_enter();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  // Render scale s: the mean and the shape's lengths enter as the rounded
  // products s * x (the rotation angle unscaled); s = 1 changes nothing.
  const float sc = render_scale(c);
  const bool rot = c.param == GS2D_PARAM_SCALE_ROT;  // (a, b, cc) = (s_x, s_y, theta)
  const float mx = __fmul_rn(sc, xy[2 * i]), my = __fmul_rn(sc, xy[2 * i + 1]);
  const float a = __fmul_rn(sc, chol[3 * i]), b = __fmul_rn(sc, chol[3 * i + 1]);
  const float cc = rot ? chol[3 * i + 2] : __fmul_rn(sc, chol[3 * i + 2]);
  const float r = rgb[3 * i], g = rgb[3 * i + 1], bl = rgb[3 * i + 2];
  const bool comp = c.mode == GS2D_MODE_COMPOSITE;
  float o = 0.0f, d = 0.0f;
  if (comp) {
    o = opacity[i];
    d = depth[i];
  }
  bool ok = isfinite(mx) && isfinite(my) && isfinite(a) && isfinite(b) && isfinite(cc) &&
            isfinite(r) && isfinite(g) && isfinite(bl);
  ok = ok && (rot ? (a != 0.0f && b != 0.0f && fabsf(cc) <= 65536.0f) : (a != 0.0f && cc != 0.0f));
  if (comp) ok = ok && isfinite(d) && isfinite(o) && o >= 0.0f && o < 1.0f;

  // Sigma^-1 = [[A, B], [B, C]] and the box half widths k*sqrt(Sigma_xx),
  // k*sqrt(Sigma_yy), in these FP32 orders (IEEE division, explicit rounding):
  //   Cholesky: A = (b^2 + c^2)/(a^2 c^2), B = -b/(a c^2), C = 1/c^2;
  //     Sigma_xx = a^2, Sigma_yy = b^2 + c^2.
  //   scale-rotation: u = 1/s_x^2, v = 1/s_y^2, c = cos, s = sin:
  //     A = c^2 u + s^2 v, B = c s (u - v), C = s^2 u + c^2 v;
  //     Sigma_xx = c^2 s_x^2 + s^2 s_y^2, Sigma_yy = s^2 s_x^2 + c^2 s_y^2.
  float A = 0.0f, B = 0.0f, C = 0.0f, rx = 0.0f, ry = 0.0f;
  if (ok) {
    const float k = c.cutoff_sigma;
    if (rot) {
      float sn, cs;
      sincos_fp32(cc, &sn, &cs);
      const float isx = __fdiv_rn(1.0f, a), isy = __fdiv_rn(1.0f, b);
      const float u = __fmul_rn(isx, isx), v = __fmul_rn(isy, isy);
      const float c2 = __fmul_rn(cs, cs), s2 = __fmul_rn(sn, sn), csn = __fmul_rn(cs, sn);
      A = __fmaf_rn(c2, u, __fmul_rn(s2, v));
      B = __fmul_rn(csn, __fsub_rn(u, v));
      C = __fmaf_rn(s2, u, __fmul_rn(c2, v));
      const float sx2 = __fmul_rn(a, a), sy2 = __fmul_rn(b, b);
      rx = __fmul_rn(k, __fsqrt_rn(__fmaf_rn(c2, sx2, __fmul_rn(s2, sy2))));
      ry = __fmul_rn(k, __fsqrt_rn(__fmaf_rn(s2, sx2, __fmul_rn(c2, sy2))));
    } else {
      const float ia = __fdiv_rn(1.0f, a);
      const float ic = __fdiv_rn(1.0f, cc);
      C = __fmul_rn(ic, ic);
      const float t = __fmul_rn(b, ia);
      B = -__fmul_rn(t, C);
      A = __fmaf_rn(__fmul_rn(t, t), C, __fmul_rn(ia, ia));
      rx = __fmul_rn(k, fabsf(a));
      ry = __fmul_rn(k, __fsqrt_rn(__fmaf_rn(b, b, __fmul_rn(cc, cc))));
    }
    ok = isfinite(A) && isfinite(B) && isfinite(C);
  }
  // Tight box of the ellipse q <= k^2; column j is inside when its centre
  // j + 0.5 lies in [mu_x - r_x, mu_x + r_x].
  int x0 = 0, y0 = 0, x1 = -1, y1 = -1;
  if (ok) {
    const float fx0 = ceilf(__fsub_rn(__fsub_rn(mx, rx), 0.5f));
    const float fx1 = floorf(__fsub_rn(__fadd_rn(mx, rx), 0.5f));
    const float fy0 = ceilf(__fsub_rn(__fsub_rn(my, ry), 0.5f));
    const float fy1 = floorf(__fsub_rn(__fadd_rn(my, ry), 0.5f));
    const float wmax = float(c.width - 1), hmax = float(c.height - 1);
    ok = (fx0 <= fx1) && (fy0 <= fy1) && !(fx0 > wmax || fx1 < 0.0f || fy0 > hmax || fy1 < 0.0f);
    if (ok) {
      x0 = int(fmaxf(fx0, 0.0f));
      y0 = int(fmaxf(fy0, 0.0f));
      x1 = int(fminf(fx1, wmax));
      y1 = int(fminf(fy1, hmax));
    }
  }
  float4* out = rec + 3 * size_t(i);
  if (ok) {
    out[0] = make_float4(mx, my, A, B);
    out[1] = make_float4(C, r, g, bl);
    out[2] = make_float4(__uint_as_float(unsigned(x0) | (unsigned(x1) << 16)),
                         __uint_as_float(unsigned(y0) | (unsigned(y1) << 16)), o, d);
    const int4 rc = make_int4(x0 / kTile, y0 / kTile, x1 / kTile, y1 / kTile);
    rect[i] = rc;
    count[i] = (rc.z - rc.x + 1) * (rc.w - rc.y + 1);
  } else {
    out[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    out[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    out[2] = make_float4(__uint_as_float(0xFFFFu), __uint_as_float(0xFFFFu), 0.f, 0.f);
    rect[i] = make_int4(0, 0, -1, -1);
    count[i] = 0;
  }
}

// Per Gaussian: sum its per-pair partials (one per tile of its rectangle, in
// emission order) and apply the chain rule to the shape parameters.
// Cholesky:
//   dA/da = -2A/a,        dA/db = 2b/(a^2 c^2),  dA/dc = -2b^2/(a^2 c^3)
//   dB/da = b/(a^2 c^2),  dB/db = -1/(a c^2),    dB/dc = 2b/(a c^3)
//   dC/dc = -2/c^3.
// Scale-rotation (u = 1/s_x^2, v = 1/s_y^2, c = cos theta, s = sin theta):
//   d(A, B, C)/du = (c^2, c s, s^2),  d(A, B, C)/dv = (s^2, -c s, c^2),
//   du/ds_x = -2/s_x^3,  dv/ds_y = -2/s_y^3,
//   d(A, B, C)/dtheta = (-2B, (c^2 - s^2)(u - v), 2B).
// d(xy) = d(mean).
// kAbs: also the pairs' absgrad sums (third float4 of the slot, .y and .z).
// The last block also sums, in a fixed order, the per-tile background
// partials (composite, d_bg non-null) and the fused pass's per-block loss
// partials (loss non-null; the total is divided by m, the number of image
// values).
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
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const bool bad = (hdr->flags & (GS2D_FLAG_CAPACITY | GS2D_FLAG_OVERFLOW | GS2D_FLAG_TIMEOUT)) != 0;
  if (i < n) {
    const int4 rc = rect[i];
    const int cnt = (rc.z >= rc.x) ? (rc.z - rc.x + 1) * (rc.w - rc.y + 1) : 0;
    float s[9] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float ax = 0.f, ay = 0.f;
    const int off = (!bad && cnt > 0) ? offsets[i] : 0;
    if (!bad && cnt > 0 && check_ok(off >= 0 && off + (long long)cnt <= hdr->pairs, kCheckPartial)) {
      constexpr int kStride = (kComposite || kAbs) ? 3 : 2;
      const float4* p = partials + size_t(off) * kStride;
      for (int k = 0; k < cnt; ++k, p += kStride) {
        const float4 u = p[0], v = p[1];
        s[0] += u.x; s[1] += u.y; s[2] += u.z; s[3] += u.w;
        s[4] += v.x; s[5] += v.y; s[6] += v.z; s[7] += v.w;
        if constexpr (kComposite || kAbs) {
          const float4 x = p[2];
          if (kComposite) s[8] += x.x;
          if (kAbs) {
            ax += x.y;
            ay += x.z;
          }
        }
      }
    }
    float g0 = 0.f, g1 = 0.f, g2 = 0.f;
    if (cnt > 0 && !bad) {
      // derivatives at the scaled shape, then back to the unscaled one
      const bool rot = param == GS2D_PARAM_SCALE_ROT;
      const float a = sc * chol[3 * i], b = sc * chol[3 * i + 1];
      const float c = rot ? chol[3 * i + 2] : sc * chol[3 * i + 2];
      const float dA = s[2], dB = s[3], dC = s[4];
      if (rot) {
        float sn, cs;
        sincos_fp32(c, &sn, &cs);
        const float isx = 1.0f / a, isy = 1.0f / b;
        const float u = isx * isx, v = isy * isy;
        const float c2 = cs * cs, s2 = sn * sn, csn = cs * sn;
        const float Bv = csn * (u - v);
        g0 = (dA * c2 + dB * csn + dC * s2) * (-2.0f * u * isx);
        g1 = (dA * s2 - dB * csn + dC * c2) * (-2.0f * v * isy);
        g2 = 2.0f * Bv * (dC - dA) + dB * (c2 - s2) * (u - v);
      } else {
        const float A = rec[3 * size_t(i)].z;
        const float ia = 1.0f / a, ic = 1.0f / c;
        const float ia2ic2 = ia * ia * ic * ic;
        g0 = dA * (-2.0f * A * ia) + dB * (b * ia2ic2);
        g1 = dA * (2.0f * b * ia2ic2) + dB * (-ia * ic * ic);
        g2 = dA * (-2.0f * b * b * ia2ic2 * ic) + dB * (2.0f * b * ia * ic * ic * ic) +
             dC * (-2.0f * ic * ic * ic);
      }
      g0 *= sc;
      g1 *= sc;
      if (!rot) g2 *= sc;
      s[0] *= sc;
      s[1] *= sc;
      ax *= sc;
      ay *= sc;
    } else {
      for (int k = 0; k < 9; ++k) s[k] = 0.f;
    }
    d_xy[2 * i] = s[0];
    d_xy[2 * i + 1] = s[1];
    d_chol[3 * i] = g0;
    d_chol[3 * i + 1] = g1;
    d_chol[3 * i + 2] = g2;
    d_rgb[3 * i] = s[5];
    d_rgb[3 * i + 1] = s[6];
    d_rgb[3 * i + 2] = s[7];
    if (kComposite && d_opacity) d_opacity[i] = s[8];
    if constexpr (kAbs) {
      d_xy_abs[2 * i] = ax;
      d_xy_abs[2 * i + 1] = ay;
    }
  }
  if ((d_bg || loss) && blockIdx.x == gridDim.x - 1) {
    // fixed-order reduction of the per-tile partials
    __shared__ float red[4][256];
    float x = 0.f, y = 0.f, z = 0.f, l = 0.f;
    if (d_bg)
      for (int t = threadIdx.x; t < T; t += blockDim.x) {
        const float4 v = tile_partials[t];
        x += v.x; y += v.y; z += v.z;
      }
    if (loss)
      for (int t = threadIdx.x; t < loss_blocks; t += blockDim.x) l += loss_partials[t];
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
    return launch(kern, dim3(blocks), dim3(256), 0, s, n, chol, r, rc, offsets, partials, hdr, d_xy,
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
