/*
 * Multi-threaded timing driver of the CPU oracle -- TEST INFRASTRUCTURE, not
 * product code: only the test suite and the benchmark's CPU-baseline leg use
 * it.  It shares nothing with the CUDA library.
 *
 * The oracle's definition is evaluated per pixel over the pixel's tile list
 * (gs2d_oracle.c).  This file compiles that same source (included below, so
 * the per-pixel functions are the very same code) and adds the one thing a
 * parallel run needs: the image is split into rows of 16x16 tiles handed to
 * OpenMP threads round-robin (schedule(static, 1), so each thread's rows
 * are fixed by the thread count), every thread accumulates gradients into
 * its own per-Gaussian buffer, and the buffers are summed in thread order.
 * The forward writes disjoint pixels and needs no reduction.  No arithmetic
 * of the method is restated here.
 */
#include "gs2d_oracle.c"

#include <omp.h>

/* Sets the thread count the calls below use (0 or less: back to OpenMP's
 * default, as first seen) and returns it. */
int32_t gs2dref_omp_threads(int32_t want) {
  static int dflt = -1;
  if (dflt < 0) dflt = omp_get_max_threads();
  omp_set_num_threads(want > 0 ? want : dflt);
  return (int32_t)omp_get_max_threads();
}

/* gs2dref_render_fwd with tile rows spread over the threads; same arguments and results. */
int64_t gs2dref_omp_render_fwd(const ref_cfg* cfg, const double* xy, const double* chol,
                               const double* rgb, const double* opacity, const double* bg,
                               const float* xy_f, const float* conic_f, const int32_t* aabb,
                               const int32_t* ranges, const int32_t* sorted_gid, double* image,
                               double* t_final, int32_t* last, double* margin) {
  ref_scene s;
  ref_scene_init(&s, cfg, xy, chol, rgb, opacity, bg, xy_f, conic_f, aabb, ranges, sorted_gid);
  const int64_t H = cfg->height, W = cfg->width, HW = H * W;
  const int32_t tx = ref_tiles_x(cfg), ty_n = ref_tiles_y(cfg);
  int64_t masked = 0;
#pragma omp parallel for schedule(static, 1) reduction(+ : masked)
  for (int32_t ty = 0; ty < ty_n; ++ty) {
    const int32_t i1 = (ty + 1) * cfg->tile < cfg->height ? (ty + 1) * cfg->tile : cfg->height;
    for (int32_t i = ty * cfg->tile; i < i1; ++i)
      for (int32_t j = 0; j < cfg->width; ++j) {
        const int64_t t = (int64_t)ty * tx + j / cfg->tile;
        double out[3], tf, mg;
        int32_t ls;
        ref_pixel_fwd(&s, sorted_gid + ranges[2 * t], ranges[2 * t + 1] - ranges[2 * t], i, j,
                      out, &tf, &ls, &mg, &masked, NULL, NULL);
        const int64_t p = (int64_t)i * W + j;
        for (int d = 0; d < 3; ++d) image[d * HW + p] = out[d];
        if (t_final) t_final[p] = tf;
        if (last) last[p] = ls;
        if (margin) margin[p] = mg;
      }
  }
  return masked;
}

/*
 * gs2dref_render_bwd with tile rows spread over the threads; same arguments
 * and results (up to the order of the double additions).  Each thread's
 * per-Gaussian accumulators take n * 88 bytes, so the thread count is capped
 * to keep them within `max_bytes` (0: 4 GiB).
 */
void gs2dref_omp_render_bwd(const ref_cfg* cfg, int32_t n, const double* xy, const double* chol,
                            const double* rgb, const double* opacity, const double* bg,
                            const float* xy_f, const float* conic_f, const int32_t* aabb,
                            const int32_t* count, const int32_t* ranges, const int32_t* sorted_gid,
                            const double* d_image, double* d_xy, double* d_chol, double* d_rgb,
                            double* d_opacity, double* d_bg, double* d_conic, double* d_xy_abs,
                            int64_t max_bytes) {
  ref_scene s;
  ref_scene_init(&s, cfg, xy, chol, rgb, opacity, bg, xy_f, conic_f, aabb, ranges, sorted_gid);
  const size_t per = sizeof(ref_grad) * (size_t)(n > 0 ? n : 1);
  const size_t cap = max_bytes > 0 ? (size_t)max_bytes : ((size_t)4 << 30);
  int nt = omp_get_max_threads();
  if ((size_t)nt * per > cap) nt = (int)(cap / per) > 0 ? (int)(cap / per) : 1;
  ref_grad* grads = (ref_grad*)calloc((size_t)nt, per);
  double* dbg = (double*)calloc((size_t)nt * 3, sizeof(double));
  const int64_t maxl = ref_max_list(cfg, ranges);
  const int64_t HW = (int64_t)cfg->height * cfg->width;
  const int32_t tx = ref_tiles_x(cfg), ty_n = ref_tiles_y(cfg);
#pragma omp parallel num_threads(nt)
  {
    const int me = omp_get_thread_num();
    ref_grad* mine = grads + (size_t)me * (size_t)(n > 0 ? n : 1);
    ref_contrib* scratch = (ref_contrib*)malloc(sizeof(ref_contrib) * (size_t)maxl);
#pragma omp for schedule(static, 1)
    for (int32_t ty = 0; ty < ty_n; ++ty) {
      const int32_t i1 = (ty + 1) * cfg->tile < cfg->height ? (ty + 1) * cfg->tile : cfg->height;
      for (int32_t i = ty * cfg->tile; i < i1; ++i)
        for (int32_t j = 0; j < cfg->width; ++j) {
          const int64_t p = (int64_t)i * cfg->width + j;
          const int64_t t = (int64_t)ty * tx + j / cfg->tile;
          const double g3[3] = {d_image[p], d_image[HW + p], d_image[2 * HW + p]};
          ref_pixel_bwd(&s, sorted_gid + ranges[2 * t], ranges[2 * t + 1] - ranges[2 * t], i, j,
                        g3, mine, -1, dbg + 3 * me, scratch);
        }
    }
    free(scratch);
  }
  /* thread order: buffer 0 collects the others */
  for (int k = 1; k < nt; ++k) {
    const ref_grad* o = grads + (size_t)k * (size_t)(n > 0 ? n : 1);
    for (int32_t g = 0; g < n; ++g) {
      ref_grad* a = &grads[g];
      for (int d = 0; d < 2; ++d) a->dmu[d] += o[g].dmu[d];
      for (int d = 0; d < 3; ++d) a->dconic[d] += o[g].dconic[d];
      for (int d = 0; d < 3; ++d) a->drgb[d] += o[g].drgb[d];
      a->dopac += o[g].dopac;
      for (int d = 0; d < 2; ++d) a->dmu_abs[d] += o[g].dmu_abs[d];
    }
    for (int d = 0; d < 3; ++d) dbg[d] += dbg[3 * k + d];
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
  free(dbg);
  free(grads);
}
