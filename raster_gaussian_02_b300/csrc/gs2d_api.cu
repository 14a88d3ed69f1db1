// The C ABI (include/gs2d.h): host-side argument checks, workspace sizing,
// and the launches of each call on the caller's stream.  Every check runs
// before anything is enqueued; no call aborts, throws or traps.
#include <cstddef>
#include <math.h>
#include <stdint.h>

#include "gs2d_internal.cuh"

using namespace gs2d;

namespace {

constexpr int kMaxSide = 32768;
constexpr long long kMaxCapacity = (1ll << 30) - 1;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool config_ok(const gs2d_config* c) {
  if (!c) return false;
  if (c->width < 1 || c->width > kMaxSide || c->height < 1 || c->height > kMaxSide) return false;
  if (c->tile != kTile) return false;
  if (c->mode != GS2D_MODE_SUM && c->mode != GS2D_MODE_COMPOSITE) return false;
  if (c->param != GS2D_PARAM_CHOLESKY && c->param != GS2D_PARAM_SCALE_ROT) return false;
  if (!isfinite(c->scale) || c->scale < 0.0f) return false;
  if (!isfinite(c->cutoff_sigma) || !(c->cutoff_sigma > 0.0f)) return false;
  if (!isfinite(c->cutoff_sigma * c->cutoff_sigma)) return false;
  if (c->mode == GS2D_MODE_COMPOSITE && !(c->t_min >= 0.0f && c->t_min <= 1.0f)) return false;
  return true;
}

gs2d_status from_cuda(cudaError_t e) { return e == cudaSuccess ? GS2D_OK : GS2D_ERR_CUDA; }

gs2d_status from_flags(unsigned int f) {
  if (f & GS2D_FLAG_TIMEOUT) return GS2D_ERR_TIMEOUT;
  if (f & GS2D_FLAG_OVERFLOW) return GS2D_ERR_OVERFLOW;
  if (f & GS2D_FLAG_CAPACITY) return GS2D_ERR_CAPACITY;
  return GS2D_OK;
}

}  // namespace

extern "C" {

size_t gs2d_workspace_size(const gs2d_config* cfg, int32_t n, int64_t pair_capacity) {
  if (!config_ok(cfg) || n < 0 || pair_capacity < 0 || pair_capacity > kMaxCapacity) return 0;
  return layout_of(*cfg, n, pair_capacity).total;
}

gs2d_status gs2d_project(const gs2d_config* cfg, int32_t n, const float* xy, const float* shape,
                         const float* rgb, const float* depth, const float* opacity,
                         gs2d_record* rec, int32_t* rect, int32_t* count, gs2d_stream_t stream) {
  if (!config_ok(cfg) || n < 0) return GS2D_ERR_INVALID_ARG;
  if (n == 0) return GS2D_OK;
  if (!xy || !shape || !rgb || !rec || !rect || !count) return GS2D_ERR_INVALID_ARG;
  if (cfg->mode == GS2D_MODE_COMPOSITE && (!depth || !opacity)) return GS2D_ERR_INVALID_ARG;
  if (!aligned(rec, 16) || !aligned(rect, 16) || !aligned(xy, 4) || !aligned(shape, 4) ||
      !aligned(rgb, 4) || !aligned(count, 4) || (depth && !aligned(depth, 4)) ||
      (opacity && !aligned(opacity, 4)))
    return GS2D_ERR_INVALID_ARG;
  return from_cuda(launch_project(*cfg, n, xy, shape, rgb, depth, opacity, rec, rect, count,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

gs2d_status gs2d_bin_and_sort(const gs2d_config* cfg, int32_t n, const gs2d_record* rec,
                              const int32_t* rect, const int32_t* count, int64_t pair_capacity,
                              int64_t* pairs_out, int32_t* tile_ranges, int32_t* sorted_gid,
                              void* workspace, gs2d_stream_t stream) {
  if (!config_ok(cfg) || n < 0) return GS2D_ERR_INVALID_ARG;
  if (pair_capacity < 0 || pair_capacity > kMaxCapacity) return GS2D_ERR_INVALID_ARG;
  if (!tile_ranges || !workspace || !aligned(tile_ranges, 16) || !aligned(workspace, 16))
    return GS2D_ERR_INVALID_ARG;
  if (pair_capacity > 0 && (!sorted_gid || !aligned(sorted_gid, 4))) return GS2D_ERR_INVALID_ARG;
  if (n > 0 && (!rec || !rect || !count || !aligned(rec, 16) || !aligned(rect, 16) ||
                !aligned(count, 4)))
    return GS2D_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_binning(*cfg, n, rec, rect, count, pair_capacity, tile_ranges, sorted_gid,
                                 static_cast<unsigned char*>(workspace), s);
  if (e != cudaSuccess) return GS2D_ERR_CUDA;
  if (!pairs_out) return GS2D_OK;
  uint32_t flags = 0;
  const gs2d_status st = gs2d_read_status(workspace, pairs_out, &flags, stream);
  return st;
}

gs2d_status gs2d_project_bin_and_sort(const gs2d_config* cfg, int32_t n, const float* xy,
                                      const float* shape, const float* rgb, const float* depth,
                                      const float* opacity, gs2d_record* rec, int32_t* rect,
                                      int32_t* count, int64_t pair_capacity, int64_t* pairs_out,
                                      int32_t* tile_ranges, int32_t* sorted_gid, void* workspace,
                                      gs2d_stream_t stream) {
  if (!config_ok(cfg) || n < 0) return GS2D_ERR_INVALID_ARG;
  if (pair_capacity < 0 || pair_capacity > kMaxCapacity) return GS2D_ERR_INVALID_ARG;
  if (!tile_ranges || !workspace || !aligned(tile_ranges, 16) || !aligned(workspace, 16))
    return GS2D_ERR_INVALID_ARG;
  if (pair_capacity > 0 && (!sorted_gid || !aligned(sorted_gid, 4))) return GS2D_ERR_INVALID_ARG;
  if (n > 0) {
    if (!xy || !shape || !rgb || !rec || !rect || !count) return GS2D_ERR_INVALID_ARG;
    if (cfg->mode == GS2D_MODE_COMPOSITE && (!depth || !opacity)) return GS2D_ERR_INVALID_ARG;
    if (!aligned(rec, 16) || !aligned(rect, 16) || !aligned(xy, 4) || !aligned(shape, 4) ||
        !aligned(rgb, 4) || !aligned(count, 4) || (depth && !aligned(depth, 4)) ||
        (opacity && !aligned(opacity, 4)))
      return GS2D_ERR_INVALID_ARG;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const ProjectIn in{xy, shape, rgb, depth, opacity};
  cudaError_t e = launch_project_binning(*cfg, n, in, rec, rect, count, pair_capacity, tile_ranges,
                                         sorted_gid, static_cast<unsigned char*>(workspace), s);
  if (e != cudaSuccess) return GS2D_ERR_CUDA;
  if (!pairs_out) return GS2D_OK;
  uint32_t flags = 0;
  return gs2d_read_status(workspace, pairs_out, &flags, stream);
}

gs2d_status gs2d_render_fwd(const gs2d_config* cfg, int32_t n, const gs2d_record* rec,
                            const int32_t* tile_ranges, const int32_t* sorted_gid,
                            const float* background, float* image, float* t_final, int32_t* last,
                            const void* workspace, gs2d_stream_t stream) {
  if (!config_ok(cfg) || n < 0) return GS2D_ERR_INVALID_ARG;
  if (workspace && !aligned(workspace, 16)) return GS2D_ERR_INVALID_ARG;
  if (!tile_ranges || !image || !aligned(tile_ranges, 16) || !aligned(image, 4))
    return GS2D_ERR_INVALID_ARG;
  if (n > 0 && (!rec || !sorted_gid || !aligned(rec, 16) || !aligned(sorted_gid, 4)))
    return GS2D_ERR_INVALID_ARG;
  if ((t_final && !aligned(t_final, 4)) || (last && !aligned(last, 4)) ||
      (background && !aligned(background, 4)))
    return GS2D_ERR_INVALID_ARG;
  return from_cuda(launch_render_fwd(*cfg, n, rec, tile_ranges, sorted_gid, background, image, t_final,
                                     last, static_cast<const unsigned char*>(workspace),
                                     reinterpret_cast<cudaStream_t>(stream)));
}

gs2d_status gs2d_loss_l2(int32_t height, int32_t width, const float* image, const float* target,
                         float* loss, float* d_image, void* workspace, gs2d_stream_t stream) {
  if (height < 1 || width < 1 || height > kMaxSide || width > kMaxSide) return GS2D_ERR_INVALID_ARG;
  if (!image || !target || !loss || !d_image || !workspace) return GS2D_ERR_INVALID_ARG;
  if (!aligned(image, 4) || !aligned(target, 4) || !aligned(loss, 4) || !aligned(d_image, 4) ||
      !aligned(workspace, 16))
    return GS2D_ERR_INVALID_ARG;
  return from_cuda(launch_loss_l2(height, width, image, target, loss, d_image,
                                  static_cast<unsigned char*>(workspace),
                                  reinterpret_cast<cudaStream_t>(stream)));
}

gs2d_status gs2d_render_bwd(const gs2d_config* cfg, int32_t n, const float* shape,
                            const gs2d_record* rec, const int32_t* rect,
                            const int32_t* tile_ranges, const int32_t* sorted_gid,
                            const float* background, const float* t_final, const int32_t* last,
                            const float* d_image, float* d_xy, float* d_shape, float* d_rgb,
                            float* d_opacity, float* d_background, float* d_xy_abs,
                            void* workspace, gs2d_stream_t stream) {
  if (!config_ok(cfg) || n < 0) return GS2D_ERR_INVALID_ARG;
  const bool comp = cfg->mode == GS2D_MODE_COMPOSITE;
  if (!tile_ranges || !d_image || !workspace || !aligned(tile_ranges, 16) ||
      !aligned(d_image, 4) || !aligned(workspace, 16))
    return GS2D_ERR_INVALID_ARG;
  if (n > 0 && (!shape || !rec || !rect || !sorted_gid || !d_xy || !d_shape || !d_rgb ||
                !aligned(rec, 16) || !aligned(rect, 16) || !aligned(shape, 4) ||
                !aligned(sorted_gid, 4) || !aligned(d_xy, 4) || !aligned(d_shape, 4) ||
                !aligned(d_rgb, 4)))
    return GS2D_ERR_INVALID_ARG;
  if (comp && (!t_final || !last || !aligned(t_final, 4) || !aligned(last, 4)))
    return GS2D_ERR_INVALID_ARG;
  if ((d_opacity && !aligned(d_opacity, 4)) || (d_background && !aligned(d_background, 4)) ||
      (background && !aligned(background, 4)) || (d_xy_abs && !aligned(d_xy_abs, 4)))
    return GS2D_ERR_INVALID_ARG;
  return from_cuda(launch_render_bwd(*cfg, n, shape, rec, rect, tile_ranges, sorted_gid,
                                     comp ? background : nullptr, t_final, last, d_image, d_xy,
                                     d_shape, d_rgb, comp ? d_opacity : nullptr,
                                     comp ? d_background : nullptr, n > 0 ? d_xy_abs : nullptr,
                                     static_cast<unsigned char*>(workspace),
                                     reinterpret_cast<cudaStream_t>(stream)));
}

gs2d_status gs2d_render_fwd_bwd_l2(const gs2d_config* cfg, int32_t n, const float* shape,
                                   const gs2d_record* rec, const int32_t* rect,
                                   const int32_t* tile_ranges, const int32_t* sorted_gid,
                                   const float* background, const float* target, float* image,
                                   float* loss, float* d_xy, float* d_shape, float* d_rgb,
                                   float* d_opacity, float* d_background, float* d_xy_abs,
                                   void* workspace, gs2d_stream_t stream) {
  if (!config_ok(cfg) || n < 0) return GS2D_ERR_INVALID_ARG;
  const bool comp = cfg->mode == GS2D_MODE_COMPOSITE;
  if (!tile_ranges || !target || !loss || !workspace || !aligned(tile_ranges, 16) ||
      !aligned(target, 4) || !aligned(loss, 4) || !aligned(workspace, 16))
    return GS2D_ERR_INVALID_ARG;
  if (n > 0 && (!shape || !rec || !rect || !sorted_gid || !d_xy || !d_shape || !d_rgb ||
                !aligned(rec, 16) || !aligned(rect, 16) || !aligned(shape, 4) ||
                !aligned(sorted_gid, 4) || !aligned(d_xy, 4) || !aligned(d_shape, 4) ||
                !aligned(d_rgb, 4)))
    return GS2D_ERR_INVALID_ARG;
  if ((image && !aligned(image, 4)) || (d_opacity && !aligned(d_opacity, 4)) ||
      (d_background && !aligned(d_background, 4)) || (background && !aligned(background, 4)) ||
      (d_xy_abs && !aligned(d_xy_abs, 4)))
    return GS2D_ERR_INVALID_ARG;
  return from_cuda(launch_render_fused_l2(*cfg, n, shape, rec, rect, tile_ranges, sorted_gid,
                                          comp ? background : nullptr, target, image, loss, d_xy,
                                          d_shape, d_rgb, comp ? d_opacity : nullptr,
                                          comp ? d_background : nullptr, n > 0 ? d_xy_abs : nullptr,
                                          static_cast<unsigned char*>(workspace),
                                          reinterpret_cast<cudaStream_t>(stream)));
}

size_t gs2d_merge_workspace_size(int32_t n) {
  if (n < 0) return 0;
  return merge_workspace_size(n);
}

gs2d_status gs2d_adam_step(const gs2d_adam* opt, int32_t n, int32_t width, float* param,
                           const float* grad, float* exp_avg, float* exp_avg_sq, const int32_t* count,
                           gs2d_stream_t stream) {
  if (!opt || n < 0 || width < 1 || width > 16) return GS2D_ERR_INVALID_ARG;
  if (!param || !grad || !exp_avg || !exp_avg_sq) return GS2D_ERR_INVALID_ARG;
  if (!aligned(param, 4) || !aligned(grad, 4) || !aligned(exp_avg, 4) || !aligned(exp_avg_sq, 4) ||
      (count && !aligned(count, 4)))
    return GS2D_ERR_INVALID_ARG;
  if (opt->step < 1 || !isfinite(opt->lr) || opt->lr < 0.0f) return GS2D_ERR_INVALID_ARG;
  if (!(opt->beta1 >= 0.0f && opt->beta1 < 1.0f) || !(opt->beta2 >= 0.0f && opt->beta2 < 1.0f))
    return GS2D_ERR_INVALID_ARG;
  if (!isfinite(opt->eps) || !(opt->eps > 0.0f)) return GS2D_ERR_INVALID_ARG;
  return from_cuda(launch_adam(n, width, param, grad, exp_avg, exp_avg_sq, count, opt->lr, opt->beta1,
                               opt->beta2, opt->eps, opt->step, reinterpret_cast<cudaStream_t>(stream)));
}

gs2d_status gs2d_merge(const gs2d_config* cfg, int32_t n, const float* xy, const float* shape,
                       const float* rgb, const gs2d_record* rec, const int32_t* count,
                       const int32_t* tile_ranges, const int32_t* sorted_gid, int32_t max_merges,
                       float* out_xy, float* out_shape, float* out_rgb, int32_t* merges_out,
                       void* merge_workspace, gs2d_stream_t stream) {
  if (!config_ok(cfg) || n < 0 || max_merges < 0) return GS2D_ERR_INVALID_ARG;
  if (cfg->mode != GS2D_MODE_SUM) return GS2D_ERR_INVALID_ARG;
  if (!merge_workspace || !aligned(merge_workspace, 256)) return GS2D_ERR_INVALID_ARG;
  if (n > 0 && (!xy || !shape || !rgb || !rec || !count || !tile_ranges || !sorted_gid ||
                !out_xy || !out_shape || !out_rgb || !aligned(rec, 16) ||
                !aligned(tile_ranges, 8) || !aligned(xy, 4) || !aligned(shape, 4) ||
                !aligned(rgb, 4) || !aligned(count, 4) || !aligned(sorted_gid, 4) ||
                !aligned(out_xy, 4) || !aligned(out_shape, 4) || !aligned(out_rgb, 4)))
    return GS2D_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned char* ws = static_cast<unsigned char*>(merge_workspace);
  cudaError_t e = launch_merge(*cfg, n, xy, shape, rgb, rec, count, tile_ranges, sorted_gid,
                               max_merges, out_xy, out_shape, out_rgb, ws, nullptr, s);
  if (e != cudaSuccess) return GS2D_ERR_CUDA;
  if (merges_out) {
    int m = 0;
    if (n > 0) {
      e = cudaMemcpyAsync(&m, ws + offsetof(MergeHeader, merges), sizeof(int),
                          cudaMemcpyDeviceToHost, s);
      if (e == cudaSuccess) e = cudaStreamSynchronize(s);
      if (e != cudaSuccess) return GS2D_ERR_CUDA;
    }
    *merges_out = m;
  }
  return GS2D_OK;
}

gs2d_status gs2d_read_status(const void* workspace, int64_t* pairs, uint32_t* flags,
                             gs2d_stream_t stream) {
  if (!workspace || !aligned(workspace, 16)) return GS2D_ERR_INVALID_ARG;
  Header h;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&h, workspace, sizeof(Header), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return GS2D_ERR_CUDA;
  if (pairs) *pairs = h.pairs;
  if (flags) *flags = h.flags;
  return from_flags(h.flags);
}

const char* gs2d_status_string(gs2d_status status) {
  switch (status) {
    case GS2D_OK: return "ok";
    case GS2D_ERR_INVALID_ARG: return "invalid argument";
    case GS2D_ERR_CAPACITY: return "pair capacity exceeded";
    case GS2D_ERR_CUDA: return "CUDA error";
    case GS2D_ERR_TIMEOUT: return "device wait timed out";
    case GS2D_ERR_OVERFLOW: return "pair count overflow";
    case GS2D_ERR_UNSUPPORTED: return "not supported by this build";
  }
  return "unknown status";
}

gs2d_status gs2d_debug_check_word(uint32_t* word, int32_t clear) {
  if (!word) return GS2D_ERR_INVALID_ARG;
  *word = 0;
#ifdef GS2D_CHECKS
  cudaError_t (*const readers[])(unsigned int*, bool) = {
      gs2d::check_word_project, gs2d::check_word_binning, gs2d::check_word_raster_fwd,
      gs2d::check_word_raster_bwd, gs2d::check_word_fused, gs2d::check_word_merge};
  unsigned int all = 0;
  for (auto read : readers) {
    unsigned int w = 0;
    if (read(&w, clear != 0) != cudaSuccess) return GS2D_ERR_CUDA;
    all |= w;
  }
  *word = all;
  return GS2D_OK;
#else
  (void)clear;
  return GS2D_ERR_UNSUPPORTED;
#endif
}

}  // extern "C"
