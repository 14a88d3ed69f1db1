/*
 * gs2d — tile-based 2D Gaussian-splatting rasterizer for NVIDIA B300 (sm_103a).
 *
 * An image is represented by N Gaussians of 8 parameters each: position
 * (2), covariance (3) given as a lower-triangular Cholesky factor, and RGB
 * colour (3) (GaussianImage project page, Overview; DrawingWithGaussians
 * README, MLX-specific notes).  The forward render is the accumulated sum
 *     C(p) = sum_i rgb_i * exp(-q_i(p)/2),   q_i(p) = d^T Sigma_i^-1 d,  d = p - mu_i
 * (GaussianImage project page, Overview: accumulated-sum rendering; FlashImgs
 * README, Python API: gate folded into the colour, additive RGB), with an
 * optional front-to-back, per-tile depth-ordered alpha-composited variant
 * over a background (DrawingWithGaussians README, Overview, 2D fitting).
 * The backward pass gives the gradient of an L2 image loss (FlashImgs
 * README, Configuration: l2_loss_ratio) with respect to xy, L and RGB (and,
 * composite, opacity and background).  Gaussians are binned into 16x16
 * pixel tiles (fVDB radiance_fields API, GaussianSplatReconstructionConfig
 * tile_size).
 *
 * Conventions shared by every call
 * --------------------------------
 *  Coordinates: pixel units; pixel (row i, column j) has its centre at
 *    (j + 0.5, i + 0.5); x to the right, y down.
 *  Touch rule: Gaussian i touches pixel p when p lies in i's pixel box (the
 *    tight axis-aligned box of the ellipse q <= k^2, k = cutoff_sigma,
 *    clipped to the image) and q_i(p) <= k^2, evaluated in FP32 in a fixed
 *    operation order, so the decision is reproducible bit for bit.
 *  Memory: every pointer argument is DEVICE memory unless marked "host".
 *    The caller owns every buffer; the library allocates nothing and keeps
 *    no state between calls (all per-call state lives in `workspace`; the
 *    one exception is gs2d_loss_l2_noalloc's fixed device array, below).
 *    Buffers are contiguous and element-aligned; gs2d_record arrays, rect,
 *    tile_ranges and the workspace must be 16-byte aligned (cudaMalloc and
 *    torch allocations are 256-byte aligned).  Calls that share a workspace
 *    must be ordered (one stream, or events between streams).
 *  Streams: every call enqueues its kernels on `stream` and returns without
 *    waiting, except gs2d_bin_and_sort with a non-NULL `pairs_out` and
 *    gs2d_read_status, which wait for the stream.  Outputs are complete when
 *    the stream reaches the point after the call.
 *  Errors: arguments are checked on the host before anything is enqueued;
 *    a failed check returns GS2D_ERR_INVALID_ARG and enqueues nothing.  A
 *    CUDA launch failure returns GS2D_ERR_CUDA.  No call aborts, throws or
 *    traps.  Gaussians with non-finite or degenerate parameters are culled
 *    (they touch nothing and get a zero gradient); that is not an error.
 *  Limits: 1 <= width, height <= 32768; tile == 16; 0 <= n < 2^31;
 *    pair capacity < 2^30.
 */
#ifndef GS2D_H
#define GS2D_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GS2D_API __attribute__((visibility("default")))
#else
#define GS2D_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t); NULL is the legacy default stream. */
typedef struct CUstream_st* gs2d_stream_t;
/* A CUDA event (cudaEvent_t). */
typedef struct CUevent_st* gs2d_event_t;

typedef enum gs2d_status {
  GS2D_OK = 0,
  GS2D_ERR_INVALID_ARG = 1, /* a host-side argument check failed; nothing was enqueued */
  GS2D_ERR_CAPACITY = 2,    /* the (tile, Gaussian) pairs exceed pair_capacity */
  GS2D_ERR_CUDA = 3,        /* a CUDA call or kernel launch failed */
  GS2D_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up (results invalid); reserved:
                               no kernel of this version waits on another block */
  GS2D_ERR_OVERFLOW = 5,    /* the pair count reached 2^30 */
  GS2D_ERR_UNSUPPORTED = 6  /* the call needs the bounds-checked build of the library */
} gs2d_status;

enum { GS2D_MODE_SUM = 0, GS2D_MODE_COMPOSITE = 1 };

/*
 * What the three shape parameters of a Gaussian are (the `shape` arrays):
 *   GS2D_PARAM_CHOLESKY   (l11, l21, l22): Sigma = L L^T, L = [[l11, 0], [l21, l22]]
 *                         (DrawingWithGaussians README, MLX-specific notes);
 *   GS2D_PARAM_SCALE_ROT  (s_x, s_y, theta): Sigma = R diag(s_x^2, s_y^2) R^T,
 *                         R = [[cos, -sin], [sin, cos]], theta in radians
 *                         (FlashImgs README, Python API:
 *                         project_gaussians_2d_scale_rot).
 */
enum { GS2D_PARAM_CHOLESKY = 0, GS2D_PARAM_SCALE_ROT = 1 };

/* Device status flags, read back by gs2d_read_status. */
enum {
  GS2D_FLAG_CAPACITY = 1u << 0,
  GS2D_FLAG_OVERFLOW = 1u << 1,
  GS2D_FLAG_TIMEOUT = 1u << 2
};

typedef struct gs2d_config {
  int32_t width;        /* image width in pixels */
  int32_t height;       /* image height in pixels */
  int32_t tile;         /* tile edge in pixels; must be 16 */
  int32_t mode;         /* GS2D_MODE_SUM or GS2D_MODE_COMPOSITE */
  float cutoff_sigma;   /* k > 0, finite: the touch rule is q <= k*k; 3 by default */
  float t_min;          /* composite only, in [0, 1]: a Gaussian contributes only
                           while the transmittance in front of it is >= t_min;
                           1e-4 by default */
  int32_t param;        /* GS2D_PARAM_CHOLESKY (0, the default) or GS2D_PARAM_SCALE_ROT */
  float scale;          /* render at any resolution: output pixels per unit of xy and
                           shape (the mean and the shape's lengths are multiplied by it;
                           rotation and colour unchanged; gradients are with respect to
                           the unscaled parameters).  0 means 1; otherwise finite and
                           > 0.  (FlashImgs README, Lifecycle / building-block API:
                           render at any height.) */
} gs2d_config;

/*
 * Projected record of one Gaussian, written by gs2d_project (48 bytes,
 * 16-byte aligned).  conic = (A, B, C) are the entries of Sigma^-1 =
 * [[A, B], [B, C]] in FP32; box_x = x0 | (x1 << 16) and box_y = y0 | (y1 << 16)
 * are the inclusive pixel box.  A culled Gaussian has an all-zero record
 * except box_x = box_y = 0x0000FFFF (an empty box).
 */
typedef struct gs2d_record {
  float mean_x, mean_y;
  float conic_a, conic_b;
  float conic_c;
  float red, green, blue;
  uint32_t box_x, box_y;
  float opacity;  /* composite: the Gaussian's opacity; 0 in sum mode */
  float depth;    /* composite: the Gaussian's depth; 0 in sum mode */
} gs2d_record;

/*
 * Bytes of device workspace needed by gs2d_bin_and_sort, gs2d_loss_l2,
 * gs2d_render_bwd and gs2d_render_fwd_bwd_l2 for this configuration, n
 * Gaussians and a pair capacity (in sum mode it includes room for the fused
 * pass's dL/dC, 12 bytes per pixel).
 * The same workspace must be passed to gs2d_bin_and_sort and to the
 * gs2d_render_bwd that follows it (the backward reads the per-Gaussian
 * pair offsets the binning left there).  The contents need no
 * initialisation.  Returns 0 for arguments that fail the checks above.
 */
GS2D_API size_t gs2d_workspace_size(const gs2d_config* cfg, int32_t n, int64_t pair_capacity);

/*
 * Projection (one thread per Gaussian).  For each Gaussian i: cull test,
 * Sigma^-1 from the shape parameters, the pixel box, the tile rectangle and
 * the number of tiles it covers.
 *   xy[n,2]       mean in pixels
 *   shape[n,3]    per cfg->param: (l11, l21, l22) -- the signs of l11 and l22
 *                 do not matter, l11 = 0 or l22 = 0 is culled -- or
 *                 (s_x, s_y, theta) -- the signs of the scales do not matter,
 *                 a zero scale or |theta| > 65536 is culled.  With the
 *                 rotation, sin and cos are taken in FP32 by range reduction
 *                 (Cody and Waite, pi/2 in three FP32 parts) and Taylor
 *                 polynomials on [-pi/4, pi/4], within 4e-7 of the exact
 *                 values for |theta| <= 1000.
 *   rgb[n,3]      colour (sum mode: the amplitude; no clamp)
 *   depth[n]      composite only (NULL in sum mode): front-to-back order key
 *   opacity[n]    composite only (NULL in sum mode): in [0, 1), else culled
 *   rec[n]        out: projected records
 *   rect[n,4]     out: tile rectangle (tx0, ty0, tx1, ty1), inclusive;
 *                 (0, 0, -1, -1) when culled
 *   count[n]      out: tiles in rect, 0 when culled
 */
GS2D_API gs2d_status gs2d_project(const gs2d_config* cfg, int32_t n, const float* xy, const float* shape,
                         const float* rgb, const float* depth, const float* opacity,
                         gs2d_record* rec, int32_t* rect, int32_t* count, gs2d_stream_t stream);

/*
 * Tile binning and sort.  Every (tile, Gaussian) pair with the tile inside
 * the Gaussian's rect is listed under its tile; lists are concatenated in
 * row-major tile order.  Sum mode: ascending Gaussian index within a tile.
 * Composite: ascending depth (IEEE order; -0 equals +0), ties by ascending
 * index.  (Per-tile depth sort: DrawingWithGaussians README, Overview,
 * gsplat-style projection/rasterization.)
 *   rec, rect, count   from gs2d_project
 *   pair_capacity      length of sorted_gid and the capacity the workspace
 *                      was sized for
 *   pairs_out          host, may be NULL.  Non-NULL: the call waits for the
 *                      stream, stores the pair count P and returns
 *                      GS2D_ERR_CAPACITY when P > pair_capacity (retry with
 *                      a larger capacity) or GS2D_ERR_OVERFLOW/TIMEOUT.
 *                      NULL: nothing waits; P and the flags stay in the
 *                      workspace for gs2d_read_status, and on overflow the
 *                      lists are left empty so later calls render nothing.
 *   tile_ranges[T,2]   out: [start, end) of tile t in sorted_gid,
 *                      T = ceil(W/16) * ceil(H/16); [0, 0) for an empty tile
 *   sorted_gid[cap]    out: Gaussian indices, the first P entries valid
 *   workspace          gs2d_workspace_size(cfg, n, pair_capacity) bytes
 */
GS2D_API gs2d_status gs2d_bin_and_sort(const gs2d_config* cfg, int32_t n, const gs2d_record* rec,
                              const int32_t* rect, const int32_t* count, int64_t pair_capacity,
                              int64_t* pairs_out, int32_t* tile_ranges, int32_t* sorted_gid,
                              void* workspace, gs2d_stream_t stream);

/*
 * gs2d_project followed by gs2d_bin_and_sort, with the same arguments and
 * results as the two calls (the outputs are bit-identical).  With few tiles
 * (the counting sort: at most 2048 tiles and 2^20 Gaussians) each block of
 * the sort's histogram kernel projects its own Gaussians first, so the
 * projection costs no launch of its own and its outputs are not read back.
 * Argument checks and errors are those of the two calls.
 */
GS2D_API gs2d_status gs2d_project_bin_and_sort(const gs2d_config* cfg, int32_t n, const float* xy,
                                               const float* shape, const float* rgb,
                                               const float* depth, const float* opacity,
                                               gs2d_record* rec, int32_t* rect, int32_t* count,
                                               int64_t pair_capacity, int64_t* pairs_out,
                                               int32_t* tile_ranges, int32_t* sorted_gid,
                                               void* workspace, gs2d_stream_t stream);

/*
 * Forward render, one thread block per 16x16 tile.
 * Sum:        C(p) = sum over touching i of rgb_i * w_i(p), w = exp(-q/2).
 * Composite:  T = 1; for the touching Gaussians in list order, while
 *             T >= t_min: alpha = opacity_i * w_i, C += rgb_i * alpha * T,
 *             T *= (1 - alpha); finally C += T * background.
 *   background[3]  composite: background colour (NULL = black); ignored in sum mode
 *   image[3,H,W]   out: planar RGB
 *   t_final[H,W]   out, composite (required for the backward; may be NULL
 *                  otherwise): final transmittance
 *   last[H,W]      out, composite (same): 1 + position within the tile's list
 *                  of the last Gaussian that contributed, 0 if none
 *   workspace      optional (NULL: tiles in index order): the workspace of
 *                  the gs2d_bin_and_sort / gs2d_project_bin_and_sort call
 *                  that wrote tile_ranges and sorted_gid, with the same cfg
 *                  and n.  With at most 2048 tiles that call also left a
 *                  launch order there (tiles by descending list length, each
 *                  with its range), and the blocks then take the longest
 *                  lists first; the result is the same either way.  Not
 *                  written.
 */
GS2D_API gs2d_status gs2d_render_fwd(const gs2d_config* cfg, int32_t n, const gs2d_record* rec,
                            const int32_t* tile_ranges, const int32_t* sorted_gid,
                            const float* background, float* image, float* t_final, int32_t* last,
                            const void* workspace, gs2d_stream_t stream);

/*
 * L2 image loss: loss = (1/(3HW)) sum (image - target)^2 and
 * d_image = 2 (image - target) / (3HW).  FP32 with a fixed-order two-level
 * reduction, so the result is bit-reproducible.
 *   image, target [3,H,W];  loss: one float (device);  d_image [3,H,W] out
 *   workspace: any workspace from gs2d_workspace_size (uses its first 16 KiB)
 */
GS2D_API gs2d_status gs2d_loss_l2(int32_t height, int32_t width, const float* image, const float* target,
                         float* loss, float* d_image, void* workspace, gs2d_stream_t stream);

/*
 * Backward render: gradients of the loss given d_image = dL/dC.
 * The touch and early-termination decisions are held fixed (their
 * derivative is zero almost everywhere).  Per-pair partial gradients are
 * written to the workspace and then summed per Gaussian in a fixed order,
 * so the result is bit-reproducible.  Every output element is written
 * (culled Gaussians get 0); outputs need no initialisation.
 *   shape[n,3]           the shape parameters given to gs2d_project
 *   rec, rect            from gs2d_project
 *   tile_ranges, sorted_gid, workspace   from gs2d_bin_and_sort
 *   background, t_final, last            composite, as given to / returned by
 *                                        gs2d_render_fwd (ignored in sum mode)
 *   d_image[3,H,W]       dL/dC
 *   d_xy[n,2], d_shape[n,3], d_rgb[n,3]  out (d_shape in the parameters of
 *                                        cfg->param)
 *   d_opacity[n]         out, composite (may be NULL)
 *   d_background[3]      out, composite (may be NULL)
 *   d_xy_abs[n,2]        out, may be NULL (not computed): absgrad, for each
 *                        Gaussian the sum over pixels p of |dL_p/dmu_x| and
 *                        of |dL_p/dmu_y|, L_p being pixel p's share of the
 *                        loss -- the densification signal that does not
 *                        cancel between pixels (DrawingWithGaussians README,
 *                        Fit 3D Gaussians and export to SuperSplat: gsplat-style
 *                        absgrad accumulated in the fused backward)
 */
GS2D_API gs2d_status gs2d_render_bwd(const gs2d_config* cfg, int32_t n, const float* shape,
                            const gs2d_record* rec, const int32_t* rect,
                            const int32_t* tile_ranges, const int32_t* sorted_gid,
                            const float* background, const float* t_final, const int32_t* last,
                            const float* d_image, float* d_xy, float* d_shape, float* d_rgb,
                            float* d_opacity, float* d_background, float* d_xy_abs,
                            void* workspace, gs2d_stream_t stream);

/*
 * Fused training pass: what gs2d_render_fwd, gs2d_loss_l2 and
 * gs2d_render_bwd compute, with dL/dC = 2 (C - target) / (3HW) formed at
 * each pixel as soon as its colour is known (FlashImgs README, Project
 * Structure: training-time rasterization, fused fwd/bwd).  Composite: one
 * per-tile kernel renders and back-propagates, keeping dL/dC on chip.  Sum:
 * the forward kernel also takes the loss and leaves dL/dC in the workspace
 * for the pair-parallel backward.  Results equal the three separate calls
 * up to the order of floating-point additions; every sum is taken in a
 * fixed order, so they are bit-reproducible.
 *   shape, rec, rect     as for gs2d_render_bwd
 *   tile_ranges, sorted_gid, workspace   from gs2d_bin_and_sort
 *   background[3]        composite (NULL: black; ignored in sum mode)
 *   target[3,H,W]        the image to fit
 *   image[3,H,W]         out, may be NULL (not written)
 *   loss                 out: one float (device), (1/(3HW)) sum (C - target)^2
 *   d_xy[n,2], d_shape[n,3], d_rgb[n,3]  out, every element written
 *   d_opacity[n], d_background[3]        out, composite (may be NULL)
 *   d_xy_abs[n,2]        out, may be NULL: absgrad, as for gs2d_render_bwd
 * Errors as for gs2d_render_bwd; target and loss must be non-NULL.
 */
GS2D_API gs2d_status gs2d_render_fwd_bwd_l2(const gs2d_config* cfg, int32_t n, const float* shape,
                                            const gs2d_record* rec, const int32_t* rect,
                                            const int32_t* tile_ranges, const int32_t* sorted_gid,
                                            const float* background, const float* target,
                                            float* image, float* loss, float* d_xy, float* d_shape,
                                            float* d_rgb, float* d_opacity, float* d_background,
                                            float* d_xy_abs, void* workspace, gs2d_stream_t stream);

/*
 * Moment-matching merge, one round, sum mode (FlashImgs README, merge --
 * Best quality pipeline: an overcomplete fit merged down via moment
 * matching).  Each valid Gaussian's most similar neighbour is the one of
 * least cost d^T M^-1 d (d = difference of the means, M = the mean of the two
 * covariances) among the Gaussians listed in the tile of its rendered mean;
 * mutual pairs merge, cheapest first (ordered by the top 16 bits of the FP32
 * cost, ties by index), at most max_merges of them.  A pair becomes one
 * Gaussian with the mass-weighted mean and covariance of the two (weight =
 * sqrt(det Sigma) * (|r| + |g| + |b|)) and each colour channel's mass kept.
 *   xy, shape, rgb       the parameters (cfg->param; cfg->scale is the render
 *                        scale the lists were binned at)
 *   rec, count, tile_ranges, sorted_gid   from gs2d_project and
 *                        gs2d_bin_and_sort of the same parameters and cfg
 *   out_xy[n,2], out_shape[n,3], out_rgb[n,3]   out: the merged set, in index
 *                        order (a pair in the slot of its lower index), its
 *                        first n - merges rows valid; must not alias the inputs
 *   merges_out           host, may be NULL: waits for the stream and stores
 *                        the number of pairs merged
 *   merge_workspace      gs2d_merge_workspace_size(n) bytes, 256-byte aligned
 * Errors: GS2D_ERR_INVALID_ARG for composite mode or bad arguments.
 */
GS2D_API size_t gs2d_merge_workspace_size(int32_t n);
GS2D_API gs2d_status gs2d_merge(const gs2d_config* cfg, int32_t n, const float* xy, const float* shape,
                                const float* rgb, const gs2d_record* rec, const int32_t* count,
                                const int32_t* tile_ranges, const int32_t* sorted_gid,
                                int32_t max_merges, float* out_xy, float* out_shape, float* out_rgb,
                                int32_t* merges_out, void* merge_workspace, gs2d_stream_t stream);

/*
 * Selective Adam step on one parameter array of n rows (one per Gaussian)
 * of `width` floats, with the optimizer's two moments in the same row layout
 * (DrawingWithGaussians README, MLX-specific notes: row-aligned optimizer
 * state for a selective Adam).  With t = opt->step (this step's number,
 * from 1) and g an element's gradient, every updated element does
 *     m = beta1 m + (1 - beta1) g,    v = beta2 v + (1 - beta2) g^2,
 *     p = p - lr (m / (1 - beta1^t)) / (sqrt(v / (1 - beta2^t)) + eps)
 * in FP32 (the bias corrections 1 - beta^t in double on the host).  With
 * count non-NULL (the pair counts of gs2d_project) the step is selective:
 * the rows of Gaussians that touch no tile (count 0) keep their parameters
 * and both moments.  One kernel per call; the arrays are device memory.
 *   param, exp_avg, exp_avg_sq [n, width]  in/out
 *   grad [n, width];  count [n] or NULL
 * Errors: GS2D_ERR_INVALID_ARG for n < 0, width outside 1..16, a NULL or
 * unaligned array (count may be NULL), step < 1, lr negative or not
 * finite, a beta outside [0, 1), eps not > 0 and finite.
 */
typedef struct gs2d_adam {
  float lr;
  float beta1;    /* 0.9 by convention */
  float beta2;    /* 0.999 by convention */
  float eps;      /* 1e-8 by convention */
  int32_t step;   /* 1 on the first step */
} gs2d_adam;

GS2D_API gs2d_status gs2d_adam_step(const gs2d_adam* opt, int32_t n, int32_t width, float* param,
                                    const float* grad, float* exp_avg, float* exp_avg_sq,
                                    const int32_t* count, gs2d_stream_t stream);

/*
 * The L2 loss of gs2d_loss_l2 for callers that cannot supply a workspace.
 * (This call has no counterpart in the method's pages; it serves callers.)
 * Some callers cannot hand the library device memory beyond the image,
 * target and outputs -- code that receives its buffers from another
 * framework and has no allocator to call, or a loop that must not call
 * cudaMalloc (it synchronises the device, and is not allowed while a
 * stream capture is running).  This call allocates nothing: it keeps the
 * reduction's block partial sums in a 4 KiB array in the library's own
 * device memory, one per GPU, held until the process exits.
 *   Same arguments and results as gs2d_loss_l2, without the workspace.
 *   Limits: 1 <= height, width <= 32768, else GS2D_ERR_INVALID_ARG (every
 *   such image fits the fixed array: the reduction uses at most 1024
 *   blocks).
 *   The first call on each device (and again the first after a device
 *   reset, which ends the CUDA context that held the array) looks the
 *   array's address up (cudaGetSymbolAddress); make that first call before
 *   any stream capture.  Later calls only compare the current context with
 *   the one the address belongs to.
 *   All calls on a device share the array: calls that overlap on the GPU
 *   (different streams, no ordering between them) race and give wrong
 *   losses.  Nothing in the array needs clearing between calls: every call
 *   writes each partial it reads.
 */
GS2D_API gs2d_status gs2d_loss_l2_noalloc(int32_t height, int32_t width, const float* image,
                                          const float* target, float* loss, float* d_image,
                                          gs2d_stream_t stream);

/*
 * Waits for `stream`, then reads what the last gs2d_bin_and_sort left in
 * the workspace: the pair count (host *pairs, may be NULL) and the
 * GS2D_FLAG_* bits (host *flags, may be NULL).  Returns the status those
 * flags map to (GS2D_OK when none is set).
 */
GS2D_API gs2d_status gs2d_read_status(const void* workspace, int64_t* pairs, uint32_t* flags,
                             gs2d_stream_t stream);

/* A static, human-readable name for a status code. */
GS2D_API const char* gs2d_status_string(gs2d_status status);

/*
 * Kernel trace: the device time of each kernel the library enqueues, for
 * profiling a pass from inside the program that runs it.  (No counterpart in
 * the method's pages, which time whole renders -- FlashImgs README, Python
 * API: benchmark_render; the trace splits such a time by kernel.)  While a
 * trace is active on the calling
 * host thread, every kernel any gs2d call launches from that thread is
 * bracketed on its stream by two of the caller's events: events[2k] is
 * recorded just before the k-th traced kernel and events[2k + 1] just after
 * it, so cudaEventElapsedTime(events[2k], events[2k + 1]) is that kernel's
 * duration.  During a stream capture the records are captured as event
 * nodes of the graph (cudaEventRecordExternal) and are recorded again on
 * every replay, so the durations are the last replay's.  Kernels, results
 * and the other calls' behaviour are unchanged; memory copies and sets are
 * not traced.
 *   events        host array of 2 * max_kernels events, created by the
 *                 caller with timing enabled and owned by it; it must stay
 *                 valid until gs2d_trace_end
 *   max_kernels   1 .. 4096: kernels that get events; later launches are
 *                 counted but not bracketed
 * gs2d_trace_begin returns GS2D_ERR_INVALID_ARG for a NULL array, a NULL
 * event or max_kernels out of range, and starts a new trace otherwise (an
 * active one is discarded).  gs2d_trace_end stops the trace and returns the
 * number of kernels launched while it was active (0 if none was).
 * gs2d_trace_kernel_name(k) returns the k-th traced kernel's name with its
 * template arguments (e.g. "k_render_bwd_sum<false>") in a per-thread
 * buffer valid until the next call, or NULL when k was not traced or a
 * trace is active.
 */
GS2D_API gs2d_status gs2d_trace_begin(const gs2d_event_t* events, int32_t max_kernels);
GS2D_API int32_t gs2d_trace_end(void);
GS2D_API const char* gs2d_trace_kernel_name(int32_t k);

/*
 * Bounds-check word of the checked build (libgs2d_checked.so, compiled with
 * GS2D_CHECKS).  In that build every index the kernels take from data -- a
 * tile id, a list range, a Gaussian index from a tile list, a pair's
 * destination or partial-gradient slot, a merge partner -- is tested before
 * the memory access it guards; a failed test skips the access and sets one
 * bit in a device word instead of faulting.  Bits: 1 tile id, 2 pair
 * destination, 3 list range, 4 Gaussian index, 5 partial slot, 6 merge
 * index, 7 shared-memory index.
 *   word   host out: the OR of the bits set since the last clear (0: every
 *          checked access stayed in bounds)
 *   clear  nonzero: zero the bits after reading them
 * Synchronizes the device.  Returns GS2D_ERR_UNSUPPORTED (and *word = 0) in
 * the normal build, whose kernels carry no checks; GS2D_ERR_INVALID_ARG for
 * a NULL word; GS2D_ERR_CUDA if a copy fails.
 */
GS2D_API gs2d_status gs2d_debug_check_word(uint32_t* word, int32_t clear);

#ifdef __cplusplus
}
#endif

#endif /* GS2D_H */
