// Projection of one Gaussian (shape parameters -> inverse covariance,
// 3-sigma pixel box, tile rectangle), shared by the projection kernel and
// the counting sort's fused projection + histogram kernel.
//
// Sigma = L L^T with L = [[a, 0], [b, c]] (DrawingWithGaussians README,
// MLX-specific notes: lower-triangular L), or Sigma = R diag(s_x^2, s_y^2) R^T
// (FlashImgs README, Python API: project_gaussians_2d_scale_rot; GaussianImage
// project page, the "rs" scripts); the 8 parameters per Gaussian are
// position, covariance and colour (GaussianImage project page, Overview).
#pragma once

#include "gs2d_internal.cuh"

namespace gs2d {

// Projects Gaussian i: writes its record, tile rectangle and tile count,
// and returns the rectangle ((0, 0, -1, -1) when culled).
__device__ __forceinline__ int4 project_one(const gs2d_config& c, int i, const float* __restrict__ xy,
                                           const float* __restrict__ chol,
                                           const float* __restrict__ rgb,
                                           const float* __restrict__ depth,
                                           const float* __restrict__ opacity,
                                           float4* __restrict__ rec, int4* __restrict__ rect,
                                           int* __restrict__ count) {
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
    return rc;
  }
  out[0] = make_float4(0.f, 0.f, 0.f, 0.f);
  out[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  out[2] = make_float4(__uint_as_float(0xFFFFu), __uint_as_float(0xFFFFu), 0.f, 0.f);
  rect[i] = make_int4(0, 0, -1, -1);
  count[i] = 0;
  return make_int4(0, 0, -1, -1);
}


}  // namespace gs2d
