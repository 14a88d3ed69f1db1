/*
 * gs2d_probe: throughput probes for the rasterizer's roofline.
 *
 * The raster kernels are bound by FP32 arithmetic and by the special-function
 * unit's 2^x (the Gaussian weight exp(-q/2) is one ex2.approx per touching
 * pixel).  The FP32/SFU peaks used for their roofline are derived from the
 * SM count, the per-SM rates per clock (128 FP32 FMAs; 32 ex2 results, the
 * figure the ex2 probe below supports on a B300: it measures 28 to 30 per
 * SM per clock, more than 16 could give) and the SM clock.  These two
 * kernels measure what the GPU actually delivers, as a cross-check of that
 * derivation.  They are separate from libgs2d.so
 * (built as libgs2d_probe.so) and take no part in the rasterizer.
 *
 * Both calls only enqueue one kernel on `stream`; the caller times them
 * (CUDA events around the call) and derives the rate from the counts below.
 * `out` is a device buffer of blocks * 256 floats that receives one value per
 * thread, so that the compiler cannot drop the arithmetic.
 * Returns 0 on success, 1 for invalid arguments (nothing enqueued), 3 if the
 * launch fails.
 */
#ifndef GS2D_PROBE_H
#define GS2D_PROBE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(_WIN32)
#define GS2D_PROBE_API __declspec(dllexport)
#else
#define GS2D_PROBE_API __attribute__((visibility("default")))
#endif

typedef struct CUstream_st* gs2d_probe_stream_t;

/*
 * FP32 fused multiply-add throughput: every thread of `blocks` blocks of 256
 * threads runs 8 independent chains of `iters` FMAs (a = a * m + c with m and
 * c passed in at run time).  Work = blocks * 256 * 8 * iters FMAs
 * = 2 * that in flops.  1 <= blocks <= 65535, 1 <= iters <= 2^20.
 */
GS2D_PROBE_API int gs2d_probe_fp32_fma(float* out, int32_t blocks, int32_t iters, float m, float c,
                                       gs2d_probe_stream_t stream);

/*
 * SFU 2^x throughput: every thread runs 8 independent chains of `iters`
 * steps x = 2^(-x) (the PTX ex2.approx.ftz.f32 instruction the raster
 * kernels use; the negation is an operand modifier).  Work = blocks * 256 *
 * 8 * iters evaluations.  Same limits as above.
 */
GS2D_PROBE_API int gs2d_probe_ex2(float* out, int32_t blocks, int32_t iters,
                                  gs2d_probe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GS2D_PROBE_H */
