/*
 * gs2d oracle: a plain, slow, single-threaded CPU statement of the tile-based
 * 2D Gaussian-splatting rasterizer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path calls, links or
 * loads this file; only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * helper with the CUDA library: the configuration struct below is declared
 * here on its own.
 *
 * What it computes, and where that comes from:
 *   - Each Gaussian has 8 parameters: position (2), covariance (3) and colour
 *     (3).  Images are rendered by an accumulated (order-independent) sum of
 *     the Gaussians' colours weighted by exp(-q/2)
 *     (GaussianImage project page, Overview).
 *   - The covariance is given by a lower-triangular Cholesky factor L,
 *     Sigma = L L^T (DrawingWithGaussians README, MLX-specific notes;
 *     GaussianImage project page, "Representation" scripts for the Cholesky
 *     variant), or by a scale and a rotation angle (FlashImgs README, Python
 *     API: project_gaussians_2d_scale_rot and the (xy, scale, rot, feat)
 *     parameters; GaussianImage project page, the "rs" scripts):
 *     Sigma = R(theta) diag(s_x^2, s_y^2) R(theta)^T.
 *   - In the sum form there is no opacity: the gate is folded into the colour,
 *     and colours add (FlashImgs README, Python API and Web viewer sections).
 *   - The optional variant alpha-composites depth-ordered Gaussians front to
 *     back over a trainable background (DrawingWithGaussians README,
 *     Overview, "2D fitting").
 *   - Gaussians are binned to 16x16 pixel tiles (fVDB radiance_fields API,
 *     GaussianSplatReconstructionConfig.tile_size).
 *   - The loss is the L2 (mean squared) image error (FlashImgs README,
 *     Configuration: l2_loss_ratio).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - pixel (row i, column j) has its centre at (j + 0.5, i + 0.5) in pixel
 *     units, x to the right and y down;
 *   - a Gaussian touches a pixel when the pixel lies inside its 3-sigma
 *     axis-aligned box AND q = d^T Sigma^-1 d <= k^2 at the pixel centre
 *     (k = cutoff_sigma, 3 by default).  That decision is an integer outcome
 *     taken from floating point, so it is taken here in the same FP32
 *     operation sequence as the GPU kernel (see ref_mask_data); every value
 *     (weights, colours, gradients) is computed in double;
 *   - sum-mode tile lists are in ascending Gaussian index; composite lists in
 *     ascending depth with ties broken by ascending index;
 *   - composite: a masked Gaussian contributes only while the transmittance
 *     before it is >= t_min; the background is added with weight T_final;
 *   - Gaussians with non-finite parameters, a zero diagonal entry of L (or
 *     a zero scale), a non-finite FP32 inverse covariance, an empty box, or
 *     (composite) an opacity outside [0, 1) are culled: they touch no pixel
 *     and get a zero gradient;
 *   - scale-rotation: R(theta) = [[cos, -sin], [sin, cos]] with theta in
 *     radians, scales in pixels; the FP32 mask data take cos and sin from
 *     the FP32 evaluation in ref_sincos_f32 (the kernel evaluates the same
 *     sequence), |theta| > 65536 is culled.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (oracle/build.py).
 * -ffp-contract=off keeps every FP32 product and sum separately rounded, so
 * that only the explicit fmaf calls fuse.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int32_t width;
  int32_t height;
  int32_t tile;          /* 16 */
  int32_t mode;          /* 0: accumulated sum, 1: alpha composite */
  float cutoff_sigma;    /* k: the mask is q <= k*k */
  float t_min;           /* composite early-termination threshold */
  int32_t param;         /* 0: Cholesky factor (l11, l21, l22); 1: scale-rotation (s_x, s_y, theta) */
  float scale;           /* output pixels per unit of xy and shape (any-resolution render); 0 means 1 */
} ref_cfg;

#define REF_MODE_SUM 0
#define REF_MODE_COMPOSITE 1
#define REF_PARAM_CHOLESKY 0
#define REF_PARAM_SCALE_ROT 1

static int32_t ref_tiles_x(const ref_cfg* cfg) { return (cfg->width + cfg->tile - 1) / cfg->tile; }
static int32_t ref_tiles_y(const ref_cfg* cfg) { return (cfg->height + cfg->tile - 1) / cfg->tile; }

int32_t gs2dref_num_tiles(const ref_cfg* cfg) { return ref_tiles_x(cfg) * ref_tiles_y(cfg); }

/*
 * Rendering at any resolution (FlashImgs README, Lifecycle / building-block
 * API: render at any height): the parameters live in the units of the image they were fitted
 * to, and the render scales them by s output pixels per unit.  The mean and
 * every length of the shape (the whole Cholesky factor, or both scales) are
 * multiplied by s, the rotation and the colour are unchanged, so Sigma is
 * multiplied by s^2 and the peak value stays the colour.  In FP32 the mask
 * data take the rounded products s * x as their inputs; s = 1 changes
 * nothing.
 */
static float ref_scale(const ref_cfg* cfg) { return cfg->scale == 0.0f ? 1.0f : cfg->scale; }

/* The scaled double-precision mean and shape of one Gaussian. */
static void ref_scaled(const ref_cfg* cfg, const double* xy, const double* P, double xs[2],
                       double Ps[3]) {
  const double s = (double)ref_scale(cfg);
  xs[0] = s * xy[0];
  xs[1] = s * xy[1];
  Ps[0] = s * P[0];
  Ps[1] = s * P[1];
  Ps[2] = (cfg->param == REF_PARAM_SCALE_ROT) ? P[2] : s * P[2];
}

/* ------------------------------------------------------------------------- */
/* Projection: validity, FP32 inverse covariance, pixel box, tile rectangle.  */
/* ------------------------------------------------------------------------- */

/*
 * Mask data of one Gaussian in FP32, the precision in which the kernel takes
 * the touch/no-touch decision.
 *
 * With L = [[a, 0], [b, c]], Sigma = L L^T = [[a^2, ab], [ab, b^2 + c^2]] and
 * Sigma^-1 = [[A, B], [B, C]] with A = (b^2 + c^2)/(a^2 c^2), B = -b/(a c^2),
 * C = 1/c^2.  The FP32 evaluation order is fixed (each product rounded, one
 * explicit fused multiply-add):
 *     ia = 1/a, ic = 1/c, C = ic*ic, t = b*ia, B = -(t*C), A = fma(t*t, C, ia*ia).
 * The box is the tight axis-aligned box of the ellipse q <= k^2, whose half
 * widths are k*sqrt(Sigma_xx) = k|a| and k*sqrt(Sigma_yy) = k*sqrt(b^2 + c^2),
 * clipped to the image; pixel column j is inside when its centre j + 0.5 lies
 * within [mu_x - r_x, mu_x + r_x].
 * Returns 1 and fills conic/aabb, or 0 when the Gaussian is culled.
 */
static int ref_mask_data(const ref_cfg* cfg, float mx, float my, float a, float b, float c,
                         float conic[3], int32_t aabb[4]) {
  if (a == 0.0f || c == 0.0f) return 0;
  const float ia = 1.0f / a;
  const float ic = 1.0f / c;
  const float C = ic * ic;
  const float t = b * ia;
  const float B = -(t * C);
  const float A = fmaf(t * t, C, ia * ia);
  if (!isfinite(A) || !isfinite(B) || !isfinite(C)) return 0;

  const float k = cfg->cutoff_sigma;
  const float rx = k * fabsf(a);
  const float ry = k * sqrtf(fmaf(b, b, c * c));
  const float fx0 = ceilf((mx - rx) - 0.5f);
  const float fx1 = floorf((mx + rx) - 0.5f);
  const float fy0 = ceilf((my - ry) - 0.5f);
  const float fy1 = floorf((my + ry) - 0.5f);
  const float wmax = (float)(cfg->width - 1);
  const float hmax = (float)(cfg->height - 1);
  if (!(fx0 <= fx1) || !(fy0 <= fy1)) return 0;
  if (fx0 > wmax || fx1 < 0.0f || fy0 > hmax || fy1 < 0.0f) return 0;
  conic[0] = A;
  conic[1] = B;
  conic[2] = C;
  aabb[0] = (int32_t)fmaxf(fx0, 0.0f);
  aabb[1] = (int32_t)fmaxf(fy0, 0.0f);
  aabb[2] = (int32_t)fminf(fx1, wmax);
  aabb[3] = (int32_t)fminf(fy1, hmax);
  return 1;
}

/*
 * sin and cos of theta in FP32, the sequence the kernel evaluates:
 * Cody and Waite's additive range reduction, theta = k (pi/2) + r with
 * k = rint(theta * 2/pi) and pi/2 split into three FP32 parts (each product
 * fused, so r carries no rounding of k * pi/2), |r| <= pi/4 (up to rounding);
 * the Taylor polynomials of sin r (to r^9) and cos r (to r^10) in Horner
 * form with the FP32 values of 1/n!; then the quadrant k mod 4 picks
 * (sin, cos) = (s, c), (c, -s), (-s, -c) or (-c, s).  For |theta| <= 65536,
 * k is an exact integer.
 */
static void ref_sincos_f32(float th, float* sn, float* cs) {
  const float k = rintf(th * 0.636619747f);
  float r = fmaf(-k, 1.57079637f, th);
  r = fmaf(-k, -4.37113883e-08f, r);
  r = fmaf(-k, -1.71512451e-15f, r);
  const float r2 = r * r;
  float p = fmaf(2.75573188e-06f, r2, -1.98412701e-04f);
  p = fmaf(p, r2, 8.33333377e-03f);
  p = fmaf(p, r2, -1.66666672e-01f);
  const float s = fmaf(p * r2, r, r);
  float q = fmaf(-2.75573200e-07f, r2, 2.48015876e-05f);
  q = fmaf(q, r2, -1.38888892e-03f);
  q = fmaf(q, r2, 4.16666679e-02f);
  q = fmaf(q, r2, -0.5f);
  const float c = fmaf(q, r2, 1.0f);
  const int quad = (int)(k - 4.0f * floorf(k * 0.25f));
  switch (quad) {
    case 0: *sn = s; *cs = c; break;
    case 1: *sn = c; *cs = -s; break;
    case 2: *sn = -s; *cs = -c; break;
    default: *sn = -c; *cs = s; break;
  }
}

/* Exported for the accuracy pin of the FP32 sin/cos. */
void gs2dref_sincos_f32(int32_t m, const float* th, float* sn, float* cs) {
  for (int32_t i = 0; i < m; ++i) ref_sincos_f32(th[i], sn + i, cs + i);
}

/*
 * Mask data from a scale and rotation: Sigma = R diag(s_x^2, s_y^2) R^T, so
 * Sigma^-1 = R diag(u, v) R^T with u = 1/s_x^2, v = 1/s_y^2:
 *     A = c^2 u + s^2 v,   B = c s (u - v),   C = s^2 u + c^2 v   (c = cos, s = sin),
 * and Sigma_xx = c^2 s_x^2 + s^2 s_y^2, Sigma_yy = s^2 s_x^2 + c^2 s_y^2.  FP32
 * order: cos and sin from ref_sincos_f32; isx = 1/s_x, u = isx*isx (and
 * v alike); A = fma(c*c, u, (s*s)*v), B = (c*s)*(u - v), C = fma(s*s, u, (c*c)*v);
 * r_x = k*sqrt(fma(c*c, s_x*s_x, (s*s)*(s_y*s_y))), r_y = k*sqrt(fma(s*s, s_x*s_x,
 * (c*c)*(s_y*s_y))).  The box rule is that of ref_mask_data.
 */
static int ref_mask_data_sr(const ref_cfg* cfg, float mx, float my, float sx, float sy,
                            float th, float conic[3], int32_t aabb[4]) {
  if (sx == 0.0f || sy == 0.0f || !(fabsf(th) <= 65536.0f)) return 0;
  float co, si;
  ref_sincos_f32(th, &si, &co);
  const float isx = 1.0f / sx;
  const float isy = 1.0f / sy;
  const float u = isx * isx;
  const float v = isy * isy;
  const float cc = co * co, ss = si * si, cs = co * si;
  const float A = fmaf(cc, u, ss * v);
  const float B = cs * (u - v);
  const float C = fmaf(ss, u, cc * v);
  if (!isfinite(A) || !isfinite(B) || !isfinite(C)) return 0;

  const float k = cfg->cutoff_sigma;
  const float sx2 = sx * sx, sy2 = sy * sy;
  const float rx = k * sqrtf(fmaf(cc, sx2, ss * sy2));
  const float ry = k * sqrtf(fmaf(ss, sx2, cc * sy2));
  const float fx0 = ceilf((mx - rx) - 0.5f);
  const float fx1 = floorf((mx + rx) - 0.5f);
  const float fy0 = ceilf((my - ry) - 0.5f);
  const float fy1 = floorf((my + ry) - 0.5f);
  const float wmax = (float)(cfg->width - 1);
  const float hmax = (float)(cfg->height - 1);
  if (!(fx0 <= fx1) || !(fy0 <= fy1)) return 0;
  if (fx0 > wmax || fx1 < 0.0f || fy0 > hmax || fy1 < 0.0f) return 0;
  conic[0] = A;
  conic[1] = B;
  conic[2] = C;
  aabb[0] = (int32_t)fmaxf(fx0, 0.0f);
  aabb[1] = (int32_t)fmaxf(fy0, 0.0f);
  aabb[2] = (int32_t)fminf(fx1, wmax);
  aabb[3] = (int32_t)fminf(fy1, hmax);
  return 1;
}

/*
 * Per-Gaussian projection for n Gaussians.
 *   conic[n,3]  FP32 (A, B, C) of Sigma^-1, zero when culled
 *   aabb[n,4]   pixel box (x0, y0, x1, y1) inclusive, (0, 0, -1, -1) when culled
 *   rect[n,4]   tile rectangle (tx0, ty0, tx1, ty1) inclusive, same when culled
 *   count[n]    number of tiles in rect, 0 when culled
 * depth/opacity are read only in composite mode (may be NULL in sum mode).
 * Returns the number of valid Gaussians.
 */
int32_t gs2dref_project(const ref_cfg* cfg, int32_t n, const float* xy, const float* chol,
                        const float* rgb, const float* depth, const float* opacity, float* conic,
                        int32_t* aabb, int32_t* rect, int32_t* count) {
  int32_t valid = 0;
  for (int32_t i = 0; i < n; ++i) {
    float* cn = conic + 3 * (int64_t)i;
    int32_t* bb = aabb + 4 * (int64_t)i;
    int32_t* rc = rect + 4 * (int64_t)i;
    cn[0] = cn[1] = cn[2] = 0.0f;
    bb[0] = bb[1] = 0;
    bb[2] = bb[3] = -1;
    rc[0] = rc[1] = 0;
    rc[2] = rc[3] = -1;
    count[i] = 0;

    int ok = 1;
    for (int d = 0; d < 2; ++d) ok &= isfinite(xy[2 * (int64_t)i + d]) != 0;
    for (int d = 0; d < 3; ++d) ok &= isfinite(chol[3 * (int64_t)i + d]) != 0;
    for (int d = 0; d < 3; ++d) ok &= isfinite(rgb[3 * (int64_t)i + d]) != 0;
    if (cfg->mode == REF_MODE_COMPOSITE) {
      ok &= isfinite(depth[i]) != 0;
      ok &= isfinite(opacity[i]) != 0;
      ok &= (opacity[i] >= 0.0f && opacity[i] < 1.0f);
    }
    if (!ok) continue;

    float cf[3];
    int32_t b4[4];
    const float* sh = chol + 3 * (int64_t)i;  /* shape parameters, per cfg->param */
    const float sc = ref_scale(cfg);
    const float mx = sc * xy[2 * (int64_t)i], my = sc * xy[2 * (int64_t)i + 1];
    const int kept = (cfg->param == REF_PARAM_SCALE_ROT)
                         ? ref_mask_data_sr(cfg, mx, my, sc * sh[0], sc * sh[1], sh[2], cf, b4)
                         : ref_mask_data(cfg, mx, my, sc * sh[0], sc * sh[1], sc * sh[2], cf, b4);
    if (!kept) continue;
    memcpy(cn, cf, sizeof cf);
    memcpy(bb, b4, sizeof b4);
    rc[0] = b4[0] / cfg->tile;
    rc[1] = b4[1] / cfg->tile;
    rc[2] = b4[2] / cfg->tile;
    rc[3] = b4[3] / cfg->tile;
    count[i] = (rc[2] - rc[0] + 1) * (rc[3] - rc[1] + 1);
    ++valid;
  }
  return valid;
}

/* ------------------------------------------------------------------------- */
/* Tile lists.                                                                */
/* ------------------------------------------------------------------------- */

static const float* g_sort_depth; /* qsort has no context argument */

static int ref_cmp_depth_gid(const void* pa, const void* pb) {
  const int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
  const float da = g_sort_depth[a], db = g_sort_depth[b];
  if (da < db) return -1;
  if (db < da) return 1;
  return (a > b) - (a < b);
}

/*
 * The list of tile t holds every Gaussian whose tile rectangle contains t:
 * in ascending index (sum) or ascending (depth, index) (composite).
 *   ranges[T,2]     [start, end) of tile t in sorted_gid (may be NULL)
 *   sorted_gid[P]   concatenated lists, tiles in row-major order (may be NULL)
 * Returns P, the total number of (tile, Gaussian) pairs.
 */
int64_t gs2dref_bin(const ref_cfg* cfg, int32_t n, const int32_t* rect, const int32_t* count,
                    const float* depth, int32_t* ranges, int32_t* sorted_gid) {
  const int32_t tx = ref_tiles_x(cfg), T = gs2dref_num_tiles(cfg);
  int64_t P = 0;
  for (int32_t i = 0; i < n; ++i) P += count[i];
  if (!ranges && !sorted_gid) return P;

  int64_t* start = (int64_t*)calloc((size_t)T + 1, sizeof(int64_t));
  for (int32_t i = 0; i < n; ++i) {
    if (count[i] == 0) continue;
    const int32_t* r = rect + 4 * (int64_t)i;
    for (int32_t y = r[1]; y <= r[3]; ++y)
      for (int32_t x = r[0]; x <= r[2]; ++x) start[(int64_t)y * tx + x + 1] += 1;
  }
  for (int32_t t = 0; t < T; ++t) start[t + 1] += start[t];
  if (ranges)
    for (int32_t t = 0; t < T; ++t) {
      ranges[2 * (int64_t)t] = (int32_t)start[t];
      ranges[2 * (int64_t)t + 1] = (int32_t)start[t + 1];
    }
  if (sorted_gid) {
    int64_t* fill = (int64_t*)malloc(sizeof(int64_t) * (size_t)T);
    memcpy(fill, start, sizeof(int64_t) * (size_t)T);
    for (int32_t i = 0; i < n; ++i) { /* ascending i: each list comes out ascending */
      if (count[i] == 0) continue;
      const int32_t* r = rect + 4 * (int64_t)i;
      for (int32_t y = r[1]; y <= r[3]; ++y)
        for (int32_t x = r[0]; x <= r[2]; ++x) sorted_gid[fill[(int64_t)y * tx + x]++] = i;
    }
    if (cfg->mode == REF_MODE_COMPOSITE) {
      g_sort_depth = depth;
      for (int32_t t = 0; t < T; ++t)
        qsort(sorted_gid + start[t], (size_t)(start[t + 1] - start[t]), sizeof(int32_t),
              ref_cmp_depth_gid);
    }
    free(fill);
  }
  free(start);
  return P;
}

/* ------------------------------------------------------------------------- */
/* Per-pair evaluation.                                                       */
/* ------------------------------------------------------------------------- */

/* The touch decision for pixel (row i, column j), FP32 as in the kernel:
 * the pixel lies in the box and q <= k^2 with
 * q = fma(dx, fma(A, dx, (2B)*dy), (C*dy)*dy),  dx = (j+0.5) - mu_x, dy = (i+0.5) - mu_y. */
static int ref_touches(const ref_cfg* cfg, const float* xy, const float* conic, const int32_t* bb,
                       int32_t i, int32_t j) {
  if (j < bb[0] || j > bb[2] || i < bb[1] || i > bb[3]) return 0;
  const float kk = cfg->cutoff_sigma * cfg->cutoff_sigma;
  const float sc = ref_scale(cfg);
  const float dx = ((float)j + 0.5f) - sc * xy[0];
  const float dy = ((float)i + 0.5f) - sc * xy[1];
  const float q = fmaf(dx, fmaf(conic[0], dx, (2.0f * conic[1]) * dy), (conic[2] * dy) * dy);
  return q <= kk;
}

/*
 * Sigma^-1 = [[A, B], [B, C]] in double from the shape parameters P.
 * Cholesky, L = [[a,0],[b,c]]: adj(Sigma)/det(Sigma) of Sigma = L L^T.
 * Scale-rotation (s_x, s_y, theta): R diag(1/s_x^2, 1/s_y^2) R^T.
 */
static void ref_inverse_cov(const ref_cfg* cfg, const double* P, double* A, double* B,
                            double* C) {
  if (cfg->param == REF_PARAM_SCALE_ROT) {
    const double c = cos(P[2]), s = sin(P[2]);
    const double u = 1.0 / (P[0] * P[0]), v = 1.0 / (P[1] * P[1]);
    *A = c * c * u + s * s * v;
    *B = c * s * (u - v);
    *C = s * s * u + c * c * v;
    return;
  }
  const double a = P[0], b = P[1], c = P[2];
  const double sxx = a * a, sxy = a * b, syy = b * b + c * c;
  const double det = sxx * syy - sxy * sxy;
  *A = syy / det;
  *B = -sxy / det;
  *C = sxx / det;
}

/* One Gaussian at one pixel centre, in double: w = exp(-q/2), plus dx, dy. */
static double ref_weight(const ref_cfg* cfg, const double* xy0, const double* L0, int32_t i,
                         int32_t j, double* dx, double* dy) {
  double xy[2], L[3], A, B, C;
  ref_scaled(cfg, xy0, L0, xy, L);
  ref_inverse_cov(cfg, L, &A, &B, &C);
  *dx = ((double)j + 0.5) - xy[0];
  *dy = ((double)i + 0.5) - xy[1];
  const double q = A * (*dx) * (*dx) + 2.0 * B * (*dx) * (*dy) + C * (*dy) * (*dy);
  return exp(-0.5 * q);
}

/* Double-precision parameters, FP32 mask data and tile lists, bundled. */
typedef struct {
  const ref_cfg* cfg;
  const double* xy;
  const double* chol;
  const double* rgb;
  const double* opacity; /* composite only */
  const double* bg;      /* composite only, [3] */
  const float* xy_f;     /* FP32 positions for the mask decision */
  const float* conic_f;
  const int32_t* aabb;
  const int32_t* ranges;
  const int32_t* sorted_gid;
} ref_scene;

typedef struct {
  int32_t gid;
  double w, alpha, T; /* T is the transmittance in front of this Gaussian */
  double dx, dy;
} ref_contrib;

/*
 * Forward at pixel (i, j) over a list of Gaussian indices.  Fills out[3];
 * for composite also *tfin, *last (1 + list position of the last Gaussian
 * that contributed, 0 if none) and *margin = min over the termination checks
 * of |ln(T / t_min)|, the distance of the early-termination decision from its
 * threshold (HUGE_VAL when no check was made).  When contrib is non-NULL the
 * contributing Gaussians are recorded in order and *ncontrib set.
 */
static void ref_pixel_fwd(const ref_scene* s, const int32_t* list, int64_t len, int32_t i,
                          int32_t j, double out[3], double* tfin, int32_t* last, double* margin,
                          int64_t* masked, ref_contrib* contrib, int64_t* ncontrib) {
  const ref_cfg* cfg = s->cfg;
  double C[3] = {0.0, 0.0, 0.0};
  double T = 1.0, mg = HUGE_VAL;
  int32_t lst = 0;
  int64_t nm = 0, nc = 0;
  for (int64_t k = 0; k < len; ++k) {
    const int32_t g = list[k];
    if (!ref_touches(cfg, s->xy_f + 2 * (int64_t)g, s->conic_f + 3 * (int64_t)g,
                     s->aabb + 4 * (int64_t)g, i, j))
      continue;
    ++nm;
    double dx, dy;
    const double w =
        ref_weight(cfg, s->xy + 2 * (int64_t)g, s->chol + 3 * (int64_t)g, i, j, &dx, &dy);
    const double* c = s->rgb + 3 * (int64_t)g;
    if (cfg->mode == REF_MODE_SUM) {
      for (int d = 0; d < 3; ++d) C[d] += c[d] * w;
      if (contrib) contrib[nc] = (ref_contrib){g, w, 0.0, 1.0, dx, dy};
      ++nc;
    } else {
      const double m = fabs(log(T / (double)cfg->t_min));
      if (m < mg) mg = m;
      if (T < (double)cfg->t_min) break;
      const double alpha = s->opacity[g] * w;
      for (int d = 0; d < 3; ++d) C[d] += c[d] * alpha * T;
      if (contrib) contrib[nc] = (ref_contrib){g, w, alpha, T, dx, dy};
      ++nc;
      T *= (1.0 - alpha);
      lst = (int32_t)(k + 1);
    }
  }
  if (cfg->mode == REF_MODE_COMPOSITE)
    for (int d = 0; d < 3; ++d) C[d] += T * s->bg[d];
  for (int d = 0; d < 3; ++d) out[d] = C[d];
  if (tfin) *tfin = (cfg->mode == REF_MODE_COMPOSITE) ? T : 1.0;
  if (last) *last = lst;
  if (margin) *margin = mg;
  if (masked) *masked += nm;
  if (ncontrib) *ncontrib = nc;
}

static void ref_scene_init(ref_scene* s, const ref_cfg* cfg, const double* xy, const double* chol,
                           const double* rgb, const double* opacity, const double* bg,
                           const float* xy_f, const float* conic_f, const int32_t* aabb,
                           const int32_t* ranges, const int32_t* sorted_gid) {
  s->cfg = cfg;
  s->xy = xy;
  s->chol = chol;
  s->rgb = rgb;
  s->opacity = opacity;
  s->bg = bg;
  s->xy_f = xy_f;
  s->conic_f = conic_f;
  s->aabb = aabb;
  s->ranges = ranges;
  s->sorted_gid = sorted_gid;
}

/*
 * Full-image forward, pixel by pixel over the pixel's tile list.
 *   image[3,H,W] (planar), t_final[H,W], last[H,W], margin[H,W]: outputs,
 *   the last three may be NULL.  Returns the number of (pixel, Gaussian)
 *   pairs that pass the touch test.
 */
int64_t gs2dref_render_fwd(const ref_cfg* cfg, const double* xy, const double* chol,
                           const double* rgb, const double* opacity, const double* bg,
                           const float* xy_f, const float* conic_f, const int32_t* aabb,
                           const int32_t* ranges, const int32_t* sorted_gid, double* image,
                           double* t_final, int32_t* last, double* margin) {
  ref_scene s;
  ref_scene_init(&s, cfg, xy, chol, rgb, opacity, bg, xy_f, conic_f, aabb, ranges, sorted_gid);
  const int64_t H = cfg->height, W = cfg->width, HW = H * W;
  const int32_t tx = ref_tiles_x(cfg);
  int64_t masked = 0;
  for (int32_t i = 0; i < cfg->height; ++i)
    for (int32_t j = 0; j < cfg->width; ++j) {
      const int64_t t = (int64_t)(i / cfg->tile) * tx + j / cfg->tile;
      const int32_t* list = sorted_gid + ranges[2 * t];
      const int64_t len = ranges[2 * t + 1] - ranges[2 * t];
      double out[3], tf, mg;
      int32_t ls;
      ref_pixel_fwd(&s, list, len, i, j, out, &tf, &ls, &mg, &masked, NULL, NULL);
      const int64_t p = (int64_t)i * W + j;
      for (int d = 0; d < 3; ++d) image[d * HW + p] = out[d];
      if (t_final) t_final[p] = tf;
      if (last) last[p] = ls;
      if (margin) margin[p] = mg;
    }
  return masked;
}

/* Forward at m sampled pixels (linear index i*W + j); out[m,3]. */
void gs2dref_render_pixels(const ref_cfg* cfg, const double* xy, const double* chol,
                           const double* rgb, const double* opacity, const double* bg,
                           const float* xy_f, const float* conic_f, const int32_t* aabb,
                           const int32_t* ranges, const int32_t* sorted_gid, const int64_t* pix,
                           int64_t m, double* out, double* t_final, int32_t* last,
                           double* margin) {
  ref_scene s;
  ref_scene_init(&s, cfg, xy, chol, rgb, opacity, bg, xy_f, conic_f, aabb, ranges, sorted_gid);
  const int32_t tx = ref_tiles_x(cfg);
  for (int64_t k = 0; k < m; ++k) {
    const int32_t i = (int32_t)(pix[k] / cfg->width), j = (int32_t)(pix[k] % cfg->width);
    const int64_t t = (int64_t)(i / cfg->tile) * tx + j / cfg->tile;
    double tf, mg;
    int32_t ls;
    ref_pixel_fwd(&s, sorted_gid + ranges[2 * t], ranges[2 * t + 1] - ranges[2 * t], i, j,
                  out + 3 * k, &tf, &ls, &mg, NULL, NULL, NULL);
    if (t_final) t_final[k] = tf;
    if (last) last[k] = ls;
    if (margin) margin[k] = mg;
  }
}

/*
 * Brute force: every pixel against every valid Gaussian, no tiles.  Sum mode
 * visits Gaussians in index order; composite in (depth, index) order.
 * valid[n] is the projection's count > 0.
 */
void gs2dref_render_brute(const ref_cfg* cfg, int32_t n, const double* xy, const double* chol,
                          const double* rgb, const double* opacity, const double* bg,
                          const float* xy_f, const float* conic_f, const int32_t* aabb,
                          const int32_t* count, const float* depth, double* image,
                          double* t_final) {
  ref_scene s;
  ref_scene_init(&s, cfg, xy, chol, rgb, opacity, bg, xy_f, conic_f, aabb, NULL, NULL);
  int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
  int64_t len = 0;
  for (int32_t g = 0; g < n; ++g)
    if (count[g] > 0) order[len++] = g;
  if (cfg->mode == REF_MODE_COMPOSITE) {
    g_sort_depth = depth;
    qsort(order, (size_t)len, sizeof(int32_t), ref_cmp_depth_gid);
  }
  const int64_t HW = (int64_t)cfg->height * cfg->width;
  for (int32_t i = 0; i < cfg->height; ++i)
    for (int32_t j = 0; j < cfg->width; ++j) {
      double out[3], tf;
      ref_pixel_fwd(&s, order, len, i, j, out, &tf, NULL, NULL, NULL, NULL, NULL);
      const int64_t p = (int64_t)i * cfg->width + j;
      for (int d = 0; d < 3; ++d) image[d * HW + p] = out[d];
      if (t_final) t_final[p] = tf;
    }
  free(order);
}

/* ------------------------------------------------------------------------- */
/* L2 loss.                                                                   */
/* ------------------------------------------------------------------------- */

/* loss = (1/(3HW)) sum (C - target)^2 and d_image = 2 (C - target) / (3HW). */
double gs2dref_loss_l2(int32_t h, int32_t w, const double* image, const double* target,
                       double* d_image) {
  const int64_t m = 3 * (int64_t)h * w;
  double acc = 0.0;
  for (int64_t k = 0; k < m; ++k) {
    const double e = image[k] - target[k];
    acc += e * e;
    if (d_image) d_image[k] = 2.0 * e / (double)m;
  }
  return m > 0 ? acc / (double)m : 0.0;
}

/* ------------------------------------------------------------------------- */
/* Backward.                                                                  */
/* ------------------------------------------------------------------------- */

/*
 * Gradient accumulators of one Gaussian, in the variables the image depends
 * on directly: mean, inverse-covariance entries (A, B, C), colour, opacity.
 */
typedef struct {
  double dmu[2], dconic[3], drgb[3], dopac;
  double dmu_abs[2]; /* absgrad: sum over pixels of |the pixel's share of dmu| */
} ref_grad;

/*
 * Chain rule through one touching pair, given dL/dw (how the loss moves with
 * the weight w of this Gaussian at this pixel).  The pair's share of the mean
 * gradient is also added in absolute value (absgrad: DrawingWithGaussians
 * README, Fit 3D Gaussians and export to SuperSplat: gsplat-style absgrad,
 * per-pixel absolute mean-gradient contributions; the three colour channels
 * are summed before the absolute value, since dL/dw already holds all
 * three).  With
 * q = A dx^2 + 2B dx dy + C dy^2, dx = px - mu_x, dy = py - mu_y and
 * w = exp(-q/2):  dw/dq = -w/2,  dq/dmu_x = -2(A dx + B dy),
 * dq/dmu_y = -2(B dx + C dy),  dq/dA = dx^2, dq/dB = 2 dx dy, dq/dC = dy^2.
 */
static void ref_accumulate_w(const ref_cfg* cfg, ref_grad* g, const double* L0, double w,
                             double dLdw, double dx, double dy) {
  double xy_unused[2], L[3], A, B, C;
  const double zero[2] = {0.0, 0.0};
  ref_scaled(cfg, zero, L0, xy_unused, L);
  ref_inverse_cov(cfg, L, &A, &B, &C);
  const double dq = dLdw * (-0.5 * w);
  const double gx = dq * (-2.0) * (A * dx + B * dy);
  const double gy = dq * (-2.0) * (B * dx + C * dy);
  g->dmu[0] += gx;
  g->dmu[1] += gy;
  g->dmu_abs[0] += fabs(gx);
  g->dmu_abs[1] += fabs(gy);
  g->dconic[0] += dq * dx * dx;
  g->dconic[1] += dq * 2.0 * dx * dy;
  g->dconic[2] += dq * dy * dy;
}

/*
 * Backward at pixel (i, j): adds this pixel's share of dL/d(params) to
 * grads[] (indexed by Gaussian) or, when only_gid >= 0, only to grads[0] for
 * that Gaussian.  dimg3 is dL/dC at the pixel; dbg (composite, may be NULL)
 * receives T_final * dL/dC.
 *   sum:        C = sum_i c_i w_i;  dC/dc_i = w_i,  dC/dw_i = c_i.
 *   composite:  C = sum_i c_i a_i T_i + T_N bg, a_i = o_i w_i,
 *               T_i = prod_{l<i} (1 - a_l);
 *               dC/dc_i = a_i T_i,
 *               dC/da_i = c_i T_i - S_i / (1 - a_i),
 *               S_i = sum_{j>i} c_j a_j T_j + T_N bg,
 *               da_i/do_i = w_i, da_i/dw_i = o_i, dC/dbg = T_N.
 * The touch decision and the early-termination decision are held fixed (the
 * mask is piecewise constant, its derivative is zero almost everywhere).
 */
static void ref_pixel_bwd(const ref_scene* s, const int32_t* list, int64_t len, int32_t i,
                          int32_t j, const double dimg3[3], ref_grad* grads, int32_t only_gid,
                          double* dbg, ref_contrib* scratch) {
  const ref_cfg* cfg = s->cfg;
  double out[3], T;
  int64_t nc = 0;
  ref_pixel_fwd(s, list, len, i, j, out, &T, NULL, NULL, NULL, scratch, &nc);
  if (cfg->mode == REF_MODE_SUM) {
    for (int64_t k = 0; k < nc; ++k) {
      const ref_contrib* e = &scratch[k];
      if (only_gid >= 0 && e->gid != only_gid) continue;
      ref_grad* g = only_gid >= 0 ? &grads[0] : &grads[e->gid];
      const double* c = s->rgb + 3 * (int64_t)e->gid;
      double dLdw = 0.0;
      for (int d = 0; d < 3; ++d) {
        g->drgb[d] += dimg3[d] * e->w;
        dLdw += dimg3[d] * c[d];
      }
      ref_accumulate_w(cfg, g, s->chol + 3 * (int64_t)e->gid, e->w, dLdw, e->dx, e->dy);
    }
    return;
  }
  /* composite: suffix sums S_i walked from the back */
  double S[3];
  for (int d = 0; d < 3; ++d) S[d] = T * s->bg[d];
  if (dbg)
    for (int d = 0; d < 3; ++d) dbg[d] += T * dimg3[d];
  for (int64_t k = nc - 1; k >= 0; --k) {
    const ref_contrib* e = &scratch[k];
    const double* c = s->rgb + 3 * (int64_t)e->gid;
    if (!(only_gid >= 0 && e->gid != only_gid)) {
      ref_grad* g = only_gid >= 0 ? &grads[0] : &grads[e->gid];
      double dLda = 0.0;
      for (int d = 0; d < 3; ++d) {
        g->drgb[d] += dimg3[d] * e->alpha * e->T;
        dLda += dimg3[d] * (c[d] * e->T - S[d] / (1.0 - e->alpha));
      }
      const double o = s->opacity[e->gid];
      g->dopac += dLda * e->w;
      ref_accumulate_w(cfg, g, s->chol + 3 * (int64_t)e->gid, e->w, dLda * o, e->dx, e->dy);
    }
    for (int d = 0; d < 3; ++d) S[d] += c[d] * e->alpha * e->T;
  }
}

/*
 * From the inverse-covariance gradient to the shape parameters.
 * Cholesky, with A = b^2/(a^2 c^2) + 1/a^2, B = -b/(a c^2), C = 1/c^2:
 *   dA/da = -2A/a,            dA/db = 2b/(a^2 c^2),  dA/dc = -2b^2/(a^2 c^3),
 *   dB/da = b/(a^2 c^2),      dB/db = -1/(a c^2),    dB/dc = 2b/(a c^3),
 *   dC/dc = -2/c^3.
 * Scale-rotation, with u = 1/s_x^2, v = 1/s_y^2, c = cos theta, s = sin theta
 * and A = c^2 u + s^2 v, B = c s (u - v), C = s^2 u + c^2 v:
 *   d/du = (c^2, c s, s^2), d/dv = (s^2, -c s, c^2) on (A, B, C),
 *   du/ds_x = -2/s_x^3, dv/ds_y = -2/s_y^3,
 *   dA/dtheta = -2B, dB/dtheta = (c^2 - s^2)(u - v), dC/dtheta = 2B.
 * These are taken at the scaled parameters; with a render scale s the
 * gradients with respect to the unscaled ones are s times the mean, absgrad
 * and length gradients (the rotation's is unchanged).
 * The position gradient is the mean gradient (xy is the mean).
 */
static void ref_finish(const ref_cfg* cfg, const double* L0, const ref_grad* g, double* dxy,
                       double* dchol, double* drgb, double* dopac, double* dxy_abs) {
  double xy_unused[2], L[3], A, B, C;
  const double zero[2] = {0.0, 0.0};
  ref_scaled(cfg, zero, L0, xy_unused, L);
  ref_inverse_cov(cfg, L, &A, &B, &C);
  const double dA = g->dconic[0], dB = g->dconic[1], dC = g->dconic[2];
  if (cfg->param == REF_PARAM_SCALE_ROT) {
    const double sx = L[0], sy = L[1], c = cos(L[2]), s = sin(L[2]);
    const double u = 1.0 / (sx * sx), v = 1.0 / (sy * sy);
    dchol[0] = (dA * c * c + dB * c * s + dC * s * s) * (-2.0 / (sx * sx * sx));
    dchol[1] = (dA * s * s - dB * c * s + dC * c * c) * (-2.0 / (sy * sy * sy));
    dchol[2] = dA * (-2.0 * B) + dB * (c * c - s * s) * (u - v) + dC * (2.0 * B);
  } else {
    const double a = L[0], b = L[1], c = L[2];
    dchol[0] = dA * (-2.0 * A / a) + dB * (b / (a * a * c * c));
    dchol[1] = dA * (2.0 * b / (a * a * c * c)) + dB * (-1.0 / (a * c * c));
    dchol[2] = dA * (-2.0 * b * b / (a * a * c * c * c)) + dB * (2.0 * b / (a * c * c * c)) +
               dC * (-2.0 / (c * c * c));
  }
  const double sc = (double)ref_scale(cfg);
  dchol[0] *= sc;
  dchol[1] *= sc;
  if (cfg->param != REF_PARAM_SCALE_ROT) dchol[2] *= sc;
  dxy[0] = sc * g->dmu[0];
  dxy[1] = sc * g->dmu[1];
  if (dxy_abs) {
    dxy_abs[0] = sc * g->dmu_abs[0];
    dxy_abs[1] = sc * g->dmu_abs[1];
  }
  for (int d = 0; d < 3; ++d) drgb[d] = g->drgb[d];
  if (dopac) *dopac = g->dopac;
}

static int64_t ref_max_list(const ref_cfg* cfg, const int32_t* ranges) {
  int64_t mx = 1;
  for (int64_t t = 0; t < gs2dref_num_tiles(cfg); ++t)
    if (ranges[2 * t + 1] - ranges[2 * t] > mx) mx = ranges[2 * t + 1] - ranges[2 * t];
  return mx;
}

/*
 * Full backward: gradients of the loss for all n Gaussians, given
 * d_image[3,H,W] = dL/dC.  Outputs d_xy[n,2], d_chol[n,3], d_rgb[n,3],
 * d_opacity[n] (composite, may be NULL), d_bg[3] (composite, may be NULL),
 * d_conic[n,3] (may be NULL), d_xy_abs[n,2] (absgrad, may be NULL).
 * count[n] marks valid Gaussians.
 */
void gs2dref_render_bwd(const ref_cfg* cfg, int32_t n, const double* xy, const double* chol,
                        const double* rgb, const double* opacity, const double* bg,
                        const float* xy_f, const float* conic_f, const int32_t* aabb,
                        const int32_t* count, const int32_t* ranges, const int32_t* sorted_gid,
                        const double* d_image, double* d_xy, double* d_chol, double* d_rgb,
                        double* d_opacity, double* d_bg, double* d_conic, double* d_xy_abs) {
  ref_scene s;
  ref_scene_init(&s, cfg, xy, chol, rgb, opacity, bg, xy_f, conic_f, aabb, ranges, sorted_gid);
  ref_grad* grads = (ref_grad*)calloc((size_t)(n > 0 ? n : 1), sizeof(ref_grad));
  ref_contrib* scratch = (ref_contrib*)malloc(sizeof(ref_contrib) * (size_t)ref_max_list(cfg, ranges));
  double dbg[3] = {0.0, 0.0, 0.0};
  const int64_t HW = (int64_t)cfg->height * cfg->width;
  const int32_t tx = ref_tiles_x(cfg);
  for (int32_t i = 0; i < cfg->height; ++i)
    for (int32_t j = 0; j < cfg->width; ++j) {
      const int64_t p = (int64_t)i * cfg->width + j;
      const int64_t t = (int64_t)(i / cfg->tile) * tx + j / cfg->tile;
      const double g3[3] = {d_image[p], d_image[HW + p], d_image[2 * HW + p]};
      ref_pixel_bwd(&s, sorted_gid + ranges[2 * t], ranges[2 * t + 1] - ranges[2 * t], i, j, g3,
                    grads, -1, dbg, scratch);
    }
  for (int32_t g = 0; g < n; ++g) {
    double dummy = 0.0;
    if (count[g] == 0) {
      memset(d_xy + 2 * (int64_t)g, 0, 2 * sizeof(double));
      memset(d_chol + 3 * (int64_t)g, 0, 3 * sizeof(double));
      memset(d_rgb + 3 * (int64_t)g, 0, 3 * sizeof(double));
      if (d_opacity) d_opacity[g] = 0.0;
      if (d_conic) memset(d_conic + 3 * (int64_t)g, 0, 3 * sizeof(double));
      if (d_xy_abs) memset(d_xy_abs + 2 * (int64_t)g, 0, 2 * sizeof(double));
      continue;
    }
    ref_finish(cfg, chol + 3 * (int64_t)g, &grads[g], d_xy + 2 * (int64_t)g, d_chol + 3 * (int64_t)g,
               d_rgb + 3 * (int64_t)g, d_opacity ? d_opacity + g : &dummy,
               d_xy_abs ? d_xy_abs + 2 * (int64_t)g : NULL);
    if (d_conic)
      for (int d = 0; d < 3; ++d) d_conic[3 * (int64_t)g + d] = grads[g].dconic[d];
  }
  if (d_bg)
    for (int d = 0; d < 3; ++d) d_bg[d] = (cfg->mode == REF_MODE_COMPOSITE) ? dbg[d] : 0.0;
  free(scratch);
  free(grads);
}

/*
 * Backward for m sampled Gaussians, visiting each one's own pixel box (a
 * different traversal from gs2dref_render_bwd, which walks pixels).  For
 * every pixel of the box it replays that pixel's tile list, so composite
 * gradients see the Gaussians in front and behind.  Outputs are [m, ...].
 */
void gs2dref_render_bwd_gaussians(const ref_cfg* cfg, int32_t n, const double* xy,
                                  const double* chol, const double* rgb, const double* opacity,
                                  const double* bg, const float* xy_f, const float* conic_f,
                                  const int32_t* aabb, const int32_t* count,
                                  const int32_t* ranges, const int32_t* sorted_gid,
                                  const double* d_image, const int32_t* gids, int32_t m,
                                  double* d_xy, double* d_chol, double* d_rgb,
                                  double* d_opacity, double* d_xy_abs) {
  (void)n;
  ref_scene s;
  ref_scene_init(&s, cfg, xy, chol, rgb, opacity, bg, xy_f, conic_f, aabb, ranges, sorted_gid);
  ref_contrib* scratch = (ref_contrib*)malloc(sizeof(ref_contrib) * (size_t)ref_max_list(cfg, ranges));
  const int64_t HW = (int64_t)cfg->height * cfg->width;
  const int32_t tx = ref_tiles_x(cfg);
  for (int32_t k = 0; k < m; ++k) {
    const int32_t g = gids[k];
    ref_grad acc;
    memset(&acc, 0, sizeof acc);
    double dummy = 0.0;
    if (count[g] > 0) {
      const int32_t* bb = aabb + 4 * (int64_t)g;
      for (int32_t i = bb[1]; i <= bb[3]; ++i)
        for (int32_t j = bb[0]; j <= bb[2]; ++j) {
          if (!ref_touches(cfg, xy_f + 2 * (int64_t)g, conic_f + 3 * (int64_t)g, bb, i, j))
            continue;
          const int64_t p = (int64_t)i * cfg->width + j;
          const int64_t t = (int64_t)(i / cfg->tile) * tx + j / cfg->tile;
          const double g3[3] = {d_image[p], d_image[HW + p], d_image[2 * HW + p]};
          ref_pixel_bwd(&s, sorted_gid + ranges[2 * t], ranges[2 * t + 1] - ranges[2 * t], i, j,
                        g3, &acc, g, NULL, scratch);
        }
      ref_finish(cfg, chol + 3 * (int64_t)g, &acc, d_xy + 2 * (int64_t)k, d_chol + 3 * (int64_t)k,
                 d_rgb + 3 * (int64_t)k, d_opacity ? d_opacity + k : &dummy,
                 d_xy_abs ? d_xy_abs + 2 * (int64_t)k : NULL);
    } else {
      if (d_xy_abs) memset(d_xy_abs + 2 * (int64_t)k, 0, 2 * sizeof(double));
      memset(d_xy + 2 * (int64_t)k, 0, 2 * sizeof(double));
      memset(d_chol + 3 * (int64_t)k, 0, 3 * sizeof(double));
      memset(d_rgb + 3 * (int64_t)k, 0, 3 * sizeof(double));
      if (d_opacity) d_opacity[k] = 0.0;
    }
  }
  free(scratch);
}

/* ------------------------------------------------------------------------- */
/* Moment-matching merge (sum mode).                                          */
/* ------------------------------------------------------------------------- */

/*
 * FlashImgs merges an overcomplete fit down to a target count "via
 * moment-matching", merging similar Gaussians (FlashImgs README, merge --
 * Best quality pipeline; the CUDA library's merge_gaussians).  The pages do
 * not say which Gaussians count as similar or how the moments are weighted;
 * the readings here:
 *   - Sigma of a Gaussian: Cholesky [[a^2, ab], [ab, b^2 + c^2]];
 *     scale-rotation R diag(s_x^2, s_y^2) R^T with cos and sin from
 *     ref_sincos_f32;
 *   - cost(i, j) = d^T M^-1 d, d = mu_i - mu_j, M = (Sigma_i + Sigma_j) / 2
 *     (the Mahalanobis distance of the means under the average covariance),
 *     taken in FP32 in the order of ref_merge_cost (a decision: the kernel
 *     evaluates the same sequence), +inf when det M <= 0, the quadratic form
 *     clamped at 0;
 *   - candidates of i: the other valid Gaussians in the tile list of the tile
 *     holding i's rendered mean (clamped to the image); nn(i) = the candidate
 *     of least cost, ties to the smaller index;
 *   - i < j = nn(i) with nn(j) = i form a pair ("mutual nearest neighbours");
 *   - at most max_merges pairs merge: ordered by the top 16 bits of the FP32
 *     cost (sign, exponent, 7 mantissa bits), ties by index, the first ones;
 *   - weights w = sqrt(det Sigma) (|r| + |g| + |b|) (the Gaussian's mass,
 *     channels summed; 2 pi cancels), equal weights if both are 0; the merged
 *     mean and covariance are the w-weighted first and second moments, and
 *     each colour channel keeps its mass: c = (c_i sqrt(det Sigma_i) +
 *     c_j sqrt(det Sigma_j)) / sqrt(det Sigma);
 *   - the merged shape: Cholesky a = sqrt(Sxx), b = Sxy / a,
 *     c = sqrt(Syy - b^2); scale-rotation theta = atan2(2 Sxy, Sxx - Syy) / 2,
 *     s_x^2, s_y^2 the eigenvalues along theta and across it;
 *   - output: the Gaussians in index order, a merged pair in the slot of its
 *     lower index and its upper index dropped; culled Gaussians pass through.
 * The merged values are computed in double.
 */
static void ref_sigma_d(const ref_cfg* cfg, const float* P, double S[3]) {
  if (cfg->param == REF_PARAM_SCALE_ROT) {
    float sn, cs;
    ref_sincos_f32(P[2], &sn, &cs);
    const double c = (double)cs, s = (double)sn;
    const double x2 = (double)P[0] * (double)P[0], y2 = (double)P[1] * (double)P[1];
    S[0] = c * c * x2 + s * s * y2;
    S[1] = c * s * (x2 - y2);
    S[2] = s * s * x2 + c * c * y2;
  } else {
    const double a = P[0], b = P[1], c = P[2];
    S[0] = a * a;
    S[1] = a * b;
    S[2] = b * b + c * c;
  }
}

/* Sigma in FP32 for the pairing decision: the same products as
 * ref_sigma_d, each rounded to FP32. */
static void ref_sigma_f(const ref_cfg* cfg, const float* P, float S[3]) {
  if (cfg->param == REF_PARAM_SCALE_ROT) {
    float sn, cs;
    ref_sincos_f32(P[2], &sn, &cs);
    const float x2 = P[0] * P[0], y2 = P[1] * P[1];
    S[0] = (cs * cs) * x2 + (sn * sn) * y2;
    S[1] = (cs * sn) * (x2 - y2);
    S[2] = (sn * sn) * x2 + (cs * cs) * y2;
  } else {
    S[0] = P[0] * P[0];
    S[1] = P[0] * P[1];
    S[2] = P[1] * P[1] + P[2] * P[2];
  }
}

static float ref_merge_cost(const float* xi, const float* Si, const float* xj, const float* Sj) {
  const float m0 = 0.5f * (Si[0] + Sj[0]), m1 = 0.5f * (Si[1] + Sj[1]), m2 = 0.5f * (Si[2] + Sj[2]);
  const float dx = xi[0] - xj[0], dy = xi[1] - xj[1];
  const float det = m0 * m2 - m1 * m1;
  if (!(det > 0.0f)) return HUGE_VALF;
  const float num = ((m2 * dx) * dx - ((2.0f * m1) * dx) * dy) + (m0 * dy) * dy;
  return (num > 0.0f ? num : 0.0f) / det; /* -0 and NaN clamp to +0 */
}

/*
 * The pairing cost of m pairs, the k-th of (xa, sha) against the k-th of
 * (xb, shb), each Sigma from its shape parameters as the merge forms it
 * (FP32 products): out[k] = cost in the sequence of ref_merge_cost.  The
 * merge itself calls the same function; this entry point exposes it so that
 * its values can be pinned.
 */
void gs2dref_merge_cost(const ref_cfg* cfg, int32_t m, const float* xa, const float* sha,
                        const float* xb, const float* shb, float* out) {
  for (int32_t k = 0; k < m; ++k) {
    float Sa[3], Sb[3];
    ref_sigma_f(cfg, sha + 3 * (int64_t)k, Sa);
    ref_sigma_f(cfg, shb + 3 * (int64_t)k, Sb);
    out[k] = ref_merge_cost(xa + 2 * (int64_t)k, Sa, xb + 2 * (int64_t)k, Sb);
  }
}

static int ref_cmp_u64(const void* pa, const void* pb) {
  const uint64_t a = *(const uint64_t*)pa, b = *(const uint64_t*)pb;
  return (a > b) - (a < b);
}

int32_t gs2dref_merge(const ref_cfg* cfg, int32_t n, const float* xy, const float* shape,
                      const float* rgb, const int32_t* count, const int32_t* ranges,
                      const int32_t* sorted_gid, int32_t max_merges, float* out_xy,
                      float* out_shape, float* out_rgb, int32_t* partner) {
  const int32_t tx = ref_tiles_x(cfg);
  const float sc = ref_scale(cfg);
  double* S = (double*)malloc(sizeof(double) * 3 * (size_t)(n > 0 ? n : 1));
  float* Sf = (float*)malloc(sizeof(float) * 3 * (size_t)(n > 0 ? n : 1));
  int32_t* nn = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
  float* cost = (float*)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
  for (int32_t i = 0; i < n; ++i) {
    ref_sigma_d(cfg, shape + 3 * (int64_t)i, S + 3 * (int64_t)i);
    ref_sigma_f(cfg, shape + 3 * (int64_t)i, Sf + 3 * (int64_t)i);
  }
  for (int32_t i = 0; i < n; ++i) {
    nn[i] = -1;
    cost[i] = HUGE_VALF;
    if (count[i] == 0) continue;
    const float px = floorf(sc * xy[2 * (int64_t)i]), py = floorf(sc * xy[2 * (int64_t)i + 1]);
    const int32_t col = px < 0.0f ? 0 : (px > (float)(cfg->width - 1) ? cfg->width - 1 : (int32_t)px);
    const int32_t row = py < 0.0f ? 0 : (py > (float)(cfg->height - 1) ? cfg->height - 1 : (int32_t)py);
    const int64_t t = (int64_t)(row / cfg->tile) * tx + col / cfg->tile;
    for (int32_t k = ranges[2 * t]; k < ranges[2 * t + 1]; ++k) {
      const int32_t j = sorted_gid[k];
      if (j == i) continue;
      const float c = ref_merge_cost(xy + 2 * (int64_t)i, Sf + 3 * (int64_t)i, xy + 2 * (int64_t)j,
                                     Sf + 3 * (int64_t)j);
      if (c < cost[i] || (c == cost[i] && j < nn[i])) {
        cost[i] = c;
        nn[i] = j;
      }
    }
  }
  /* mutual pairs (lower index), ordered by the top 16 bits of the FP32 cost, then index */
  int32_t* pairs = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
  uint32_t* key = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)(n > 0 ? n : 1));
  int32_t np = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t j = nn[i];
    if (j > i && nn[j] == i) {
      uint32_t u;
      memcpy(&u, &cost[i], sizeof u);
      key[np] = u >> 16;
      pairs[np++] = i;
    }
  }
  /* the first max_merges pairs in (key, index) order */
  uint64_t* order = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)(np > 0 ? np : 1));
  for (int32_t q = 0; q < np; ++q) order[q] = ((uint64_t)key[q] << 32) | (uint32_t)pairs[q];
  qsort(order, (size_t)np, sizeof(uint64_t), ref_cmp_u64);
  char* take = (char*)calloc((size_t)(n > 0 ? n : 1), 1);
  int32_t merges = 0;
  for (int32_t q = 0; q < np && merges < max_merges; ++q, ++merges)
    take[(int32_t)(order[q] & 0xFFFFFFFFu)] = 1;
  free(order);
  /* write the merged set */
  char* dropped = (char*)calloc((size_t)(n > 0 ? n : 1), 1);
  for (int32_t i = 0; i < n; ++i)
    if (take[i]) dropped[nn[i]] = 1;
  if (partner) /* for the tests: the merged partner of each lower index, else -1 */
    for (int32_t i = 0; i < n; ++i) partner[i] = take[i] ? nn[i] : -1;
  int32_t o = 0;
  for (int32_t i = 0; i < n; ++i) {
    if (dropped[i]) continue;
    float* X = out_xy + 2 * (int64_t)o;
    float* P = out_shape + 3 * (int64_t)o;
    float* Cc = out_rgb + 3 * (int64_t)o;
    if (!take[i]) {
      memcpy(X, xy + 2 * (int64_t)i, 2 * sizeof(float));
      memcpy(P, shape + 3 * (int64_t)i, 3 * sizeof(float));
      memcpy(Cc, rgb + 3 * (int64_t)i, 3 * sizeof(float));
      ++o;
      continue;
    }
    const int32_t j = nn[i];
    const double* Si = S + 3 * (int64_t)i;
    const double* Sj = S + 3 * (int64_t)j;
    const double ri = sqrt(Si[0] * Si[2] - Si[1] * Si[1]);
    const double rj = sqrt(Sj[0] * Sj[2] - Sj[1] * Sj[1]);
    const float* ci = rgb + 3 * (int64_t)i;
    const float* cj = rgb + 3 * (int64_t)j;
    double wi = ri * (fabs((double)ci[0]) + fabs((double)ci[1]) + fabs((double)ci[2]));
    double wj = rj * (fabs((double)cj[0]) + fabs((double)cj[1]) + fabs((double)cj[2]));
    if (wi + wj == 0.0) wi = wj = 1.0;
    const double W = wi + wj;
    const double xi0 = xy[2 * (int64_t)i], xi1 = xy[2 * (int64_t)i + 1];
    const double xj0 = xy[2 * (int64_t)j], xj1 = xy[2 * (int64_t)j + 1];
    const double m0 = (wi * xi0 + wj * xj0) / W, m1 = (wi * xi1 + wj * xj1) / W;
    const double di0 = xi0 - m0, di1 = xi1 - m1, dj0 = xj0 - m0, dj1 = xj1 - m1;
    const double sxx = (wi * (Si[0] + di0 * di0) + wj * (Sj[0] + dj0 * dj0)) / W;
    const double sxy = (wi * (Si[1] + di0 * di1) + wj * (Sj[1] + dj0 * dj1)) / W;
    const double syy = (wi * (Si[2] + di1 * di1) + wj * (Sj[2] + dj1 * dj1)) / W;
    const double r = sqrt(sxx * syy - sxy * sxy);
    X[0] = (float)m0;
    X[1] = (float)m1;
    for (int d = 0; d < 3; ++d) Cc[d] = (float)(((double)ci[d] * ri + (double)cj[d] * rj) / r);
    if (cfg->param == REF_PARAM_SCALE_ROT) {
      const double th = 0.5 * atan2(2.0 * sxy, sxx - syy);
      const double c = cos(th), s = sin(th);
      /* eigenvalue along theta: the quadratic form of (cos, sin); the other
         is the trace minus it */
      const double l1 = c * c * sxx + 2.0 * c * s * sxy + s * s * syy;
      const double l2 = (sxx + syy) - l1;
      P[0] = (float)sqrt(l1);
      P[1] = (float)sqrt(l2 > 0.0 ? l2 : 0.0);
      P[2] = (float)th;
    } else {
      const double a = sqrt(sxx), b = sxy / a;
      P[0] = (float)a;
      P[1] = (float)b;
      P[2] = (float)sqrt(syy - b * b);
    }
    ++o;
  }
  free(S);
  free(Sf);
  free(nn);
  free(cost);
  free(pairs);
  free(key);
  free(take);
  free(dropped);
  return merges;
}
