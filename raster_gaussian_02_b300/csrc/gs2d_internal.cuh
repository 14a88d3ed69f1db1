// Internal declarations of the gs2d CUDA library: workspace layout, device
// helpers for the FP32 touch rule, and the kernel launchers each .cu file
// provides.  Not part of the public interface (include/gs2d.h is).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gs2d.h"

namespace gs2d {

constexpr int kTile = 16;
constexpr int kTilePixels = kTile * kTile;

// Workspace layout (byte offsets; every region 256-byte aligned).  The
// regions the backward reads come before every region whose size depends on
// the pair capacity, so their offsets follow from (cfg, n) alone; the one
// exception, the sorted keys, is located through Header::keys_final.
//   [0, 256)          Header
//   [256, 4352)       loss partial sums (kLossMaxBlocks floats)
//   [4352, 12544)     radix digit totals [kMaxPasses][kMaxRadix]
//   then              per-block pair totals, then offsets [ceil(n / kScanItems) + 1] (int64)
//   then              per-Gaussian pair offsets [n] (int32)
//   then              background partials [T] x 4 floats (composite)
//   then              backward partials [cap] x 8 floats (sum) or x 12 (composite)
//   then              radix count tables [passes][radix][partitions(cap) rounded up to 4]
//   then              keys A, keys B [cap] (uint32 sum, uint64 composite)
//   then              values scratch [cap] (uint32)
struct Header {
  long long pairs;                 // P, written by the binning
  unsigned int flags;              // GS2D_FLAG_*
  unsigned int blocks_done;        // count of finished blocks (last one finishes the scan)
  unsigned long long keys_final;   // byte offset of the sorted keys
  unsigned int blocks_done2;       // the same for a second kernel
};

constexpr int kMaxPasses = 8;
constexpr int kMaxDigitBits = 8;
constexpr int kMaxRadix = 1 << kMaxDigitBits;
constexpr size_t kOffLoss = 256;
constexpr int kLossMaxBlocks = 1024;
constexpr size_t kOffHist = kOffLoss + kLossMaxBlocks * 4;           // 4352
constexpr size_t kOffScan = kOffHist + size_t(kMaxPasses) * kMaxRadix * 4;  // 12544

constexpr int kScanThreads = 256;
constexpr int kScanItems = kScanThreads;  // Gaussians per scan block, one per thread

constexpr int kRadixThreads = 256;
// With at most this many tiles (and Gaussians) the lists are sorted by counting:
// the per-tile Gaussian masks of one 256-Gaussian block take 32 bytes per
// tile of shared memory.
constexpr int kCountSortMaxTiles = 2048;
constexpr long long kCountSortMaxGaussians = 1 << 20;

struct Layout {
  size_t block_off, offsets, tile_partials, loss_partials, dimage, tile_order, tile_hist, partials, tables, keys_a, keys_b, vals_tmp, total;
  int passes, digit_bits, tile_bits, key_bits, key_bytes, partial_floats, radix_per_thread;
  bool count_sort;  // few tiles: counting sort by tile (composite: then by depth per tile)
  long long partitions, partitions4;  // radix partitions, and rounded up to a multiple of 4
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline int tiles_x(const gs2d_config& c) { return (c.width + kTile - 1) / kTile; }
inline int tiles_y(const gs2d_config& c) { return (c.height + kTile - 1) / kTile; }
inline int num_tiles(const gs2d_config& c) { return tiles_x(c) * tiles_y(c); }

// Render scale (output pixels per unit of xy and shape); 0 means 1.
__host__ __device__ inline float render_scale(const gs2d_config& c) {
  return c.scale == 0.0f ? 1.0f : c.scale;
}

// Streaming multiprocessors of the current device (148 if the query fails).
inline int sm_count() {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 148;
  return sms;
}

inline int bits_for(long long values) {  // bits needed to hold 0 .. values-1
  int b = 0;
  while ((1ll << b) < values) ++b;
  return b;
}

// Keys per radix partition = kRadixThreads * radix_per_thread.  Measured on a
// B300 at 1.2e5 pairs: 2048-key partitions beat 1024 (the look-back chain is
// shorter) and match 4096.
inline int radix_per_thread(long long) { return 8; }

inline Layout layout_of(const gs2d_config& c, long long n, long long cap) {
  Layout L{};
  const int T = num_tiles(c);
  L.tile_bits = bits_for(T);
  const bool comp = c.mode == GS2D_MODE_COMPOSITE;
  L.key_bits = L.tile_bits + (comp ? 32 : 0);
  L.passes = (L.key_bits + kMaxDigitBits - 1) / kMaxDigitBits;
  L.digit_bits = kMaxDigitBits;  // every pass sorts a full 8-bit digit (256 buckets)
  L.key_bytes = comp ? 8 : 4;
  // per pair: 8 floats (sum) or 9 (composite) of partial derivatives, plus
  // 2 absgrad sums; slots of 3 float4 (sum without absgrad uses 2 of them)
  L.partial_floats = 12;
  L.radix_per_thread = radix_per_thread(cap);
  const long long items = (long long)kRadixThreads * L.radix_per_thread;
  L.partitions = (cap + items - 1) / items;
  L.partitions4 = (L.partitions + 3) & ~3ll;
  const size_t radix = kMaxRadix;
  size_t o = kOffScan;
  L.block_off = o;
  o = align256(o + 8 * size_t((n + kScanItems - 1) / kScanItems + 1));
  L.offsets = o;
  o = align256(o + 4 * size_t(n));
  L.tile_partials = o;  // per tile: background gradient (x, y, z)
  o = align256(o + 16 * size_t(T));
  L.loss_partials = o;  // fused pass: per block (at most two per tile) loss sums
  o = align256(o + 8 * size_t(T));
  L.dimage = o;  // fused pass, sum mode: dL/dC [3,H,W]
  if (!comp) o = align256(o + 12 * size_t(c.width) * size_t(c.height));
  L.tile_order = o;  // counting sort: (tile, start, end, 0) by descending list length (launch order)
  o = align256(o + 16 * size_t(T));
  L.tile_hist = o;  // counting sort by tile: [T][blocks] counts, then row totals [T]
  L.count_sort = T <= kCountSortMaxTiles && n <= kCountSortMaxGaussians;
  if (L.count_sort) {
    const long long B = n > 0 ? (n + kScanItems - 1) / kScanItems : 1;
    o = align256(o + 4 * size_t(T) * size_t(B) + 4 * size_t(T));
  }
  L.partials = o;
  o = align256(o + 4 * size_t(L.partial_floats) * size_t(cap));
  L.tables = o;
  o = align256(o + 4 * size_t(L.passes) * size_t(L.partitions4) * radix);
  L.keys_a = o;
  o = align256(o + size_t(L.key_bytes) * size_t(cap));
  L.keys_b = o;
  o = align256(o + size_t(L.key_bytes) * size_t(cap));
  L.vals_tmp = o;
  o = align256(o + 4 * size_t(cap));
  L.total = o < 16384 ? 16384 : o;  // the loss alone needs the first 16 KiB
  return L;
}

// ------------------------------------------------------------ device side --

// The FP32 touch rule.  Every operation is an explicitly rounded intrinsic so
// that the compiler can neither contract nor reorder it; the oracle evaluates
// the same sequence on the CPU.
//   q = fma(dx, fma(A, dx, (2B) * dy), (C * dy) * dy)
__device__ __forceinline__ float touch_q(float dx, float dy, float A, float B2, float C) {
  const float cdy = __fmul_rn(C, dy);
  const float cdydy = __fmul_rn(cdy, dy);
  const float inner = __fmaf_rn(A, dx, __fmul_rn(B2, dy));
  return __fmaf_rn(dx, inner, cdydy);
}

// 2^x with the hardware approximation (the PTX ex2.approx instruction).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 1/x with the hardware approximation (the PTX rcp.approx instruction, about
// one ulp); used only in gradient arithmetic, never in a touch or
// termination decision.
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// exp(-q/2) = 2^(q * (-log2(e)/2)).
constexpr float kNegHalfLog2e = -0.72134752044448170368f;

__device__ __forceinline__ unsigned int box_lo(unsigned int b) { return b & 0xFFFFu; }
__device__ __forceinline__ unsigned int box_hi(unsigned int b) { return b >> 16; }

// The lanes of a warp whose pixel lies in the box [x0, x1] x [y0, y1]; the
// warp covers columns bx0..bx0+7 and rows by0..by0+3, lane = 8 * row + col.
// Returns 0 when the box misses the sub-block.
__device__ __forceinline__ unsigned int box_lanes(uint2 b, int bx0, int by0) {
  const int cl = max(int(box_lo(b.x)) - bx0, 0), ch = min(int(box_hi(b.x)) - bx0, 7);
  const int rl = max(int(box_lo(b.y)) - by0, 0), rh = min(int(box_hi(b.y)) - by0, 3);
  if (cl > ch || rl > rh) return 0u;
  const unsigned int cols = (0xFFu >> (7 - ch)) & (0xFFu << cl);
  const unsigned int rows = (0xFFFFFFFFu >> (8 * (3 - rh))) & (0xFFFFFFFFu << (8 * rl));
  return (cols * 0x01010101u) & rows;
}

// sin and cos of theta in FP32 for the scale-rotation shape: Cody and Waite's
// additive range reduction, theta = k (pi/2) + r with k = rint(theta * 2/pi)
// and pi/2 split into three FP32 parts (fused products, so r carries no
// rounding of k * pi/2), |r| <= pi/4; the Taylor polynomials of sin r (to
// r^9) and cos r (to r^10) in Horner form with the FP32 values of 1/n!; the
// quadrant k mod 4 then swaps and negates them.  Every step is an explicitly
// rounded operation so that the result is the same FP32 value wherever the
// sequence is evaluated.  For |theta| <= 65536, k is an exact integer.
__device__ __forceinline__ void sincos_fp32(float th, float* sn, float* cs) {
  const float k = rintf(__fmul_rn(th, 0.636619747f));
  float r = __fmaf_rn(-k, 1.57079637f, th);
  r = __fmaf_rn(-k, -4.37113883e-08f, r);
  r = __fmaf_rn(-k, -1.71512451e-15f, r);
  const float r2 = __fmul_rn(r, r);
  float p = __fmaf_rn(2.75573188e-06f, r2, -1.98412701e-04f);
  p = __fmaf_rn(p, r2, 8.33333377e-03f);
  p = __fmaf_rn(p, r2, -1.66666672e-01f);
  const float s = __fmaf_rn(__fmul_rn(p, r2), r, r);
  float q = __fmaf_rn(-2.75573200e-07f, r2, 2.48015876e-05f);
  q = __fmaf_rn(q, r2, -1.38888892e-03f);
  q = __fmaf_rn(q, r2, 4.16666679e-02f);
  q = __fmaf_rn(q, r2, -0.5f);
  const float c = __fmaf_rn(q, r2, 1.0f);
  const int quad = int(__fsub_rn(k, __fmul_rn(4.0f, floorf(__fmul_rn(k, 0.25f)))));
  switch (quad) {
    case 0: *sn = s; *cs = c; break;
    case 1: *sn = c; *cs = -s; break;
    case 2: *sn = -s; *cs = -c; break;
    default: *sn = -c; *cs = s; break;
  }
}

// ------------------------------------------------------- checked build --
// Built with -DGS2D_CHECKS (libgs2d_checked.so), every index that comes from
// data -- a list entry, an offset, a tile id, a destination slot -- is tested
// before the access it guards.  A failed test sets bit `site` of its
// translation unit's check word and the access is skipped: nothing traps, and
// gs2d_debug_check_word() reads the bits back.  The normal build compiles the
// tests away.  Sites:
enum CheckSite {
  kCheckTile = 1,      // tile id outside [0, T)
  kCheckPairSlot = 2,  // pair destination outside [0, capacity)
  kCheckRange = 3,     // a tile's list range outside [0, pairs]
  kCheckGaussian = 4,  // Gaussian index outside [0, n)
  kCheckPartial = 5,   // partial-gradient slot outside [0, pairs)
  kCheckMerge = 6,     // merge index outside [0, n)
  kCheckShared = 7,    // shared-memory index outside its array
};
#ifdef GS2D_CHECKS
static __device__ unsigned int g_check_word;
__device__ __forceinline__ bool check_ok(bool cond, int site) {
  if (!cond) atomicOr(&g_check_word, 1u << site);
  return cond;
}
// Defines check_word_<name>(): reads (and with clear, zeroes) this
// translation unit's check word.
#define GS2D_CHECK_WORD_READER(name)                                                   \
  cudaError_t check_word_##name(unsigned int* out, bool clear) {                      \
    cudaError_t e = cudaMemcpyFromSymbol(out, g_check_word, sizeof(unsigned int));    \
    if (e == cudaSuccess && clear) {                                                   \
      const unsigned int zero = 0u;                                                    \
      e = cudaMemcpyToSymbol(g_check_word, &zero, sizeof(unsigned int));              \
    }                                                                                  \
    return e;                                                                          \
  }
#else
__device__ __forceinline__ bool check_ok(bool cond, int) {
  (void)cond;
  return true;
}
#define GS2D_CHECK_WORD_READER(name)
#endif

// Sums a Gaussian's cnt per-pair partial slots (kStride float4 each, in
// emission order) starting at p: s[0..7] from the first two float4, s[8]
// (kOpacity) from the third's .x, the absgrad sums (kAbs) from its .y, .z.
// The loads of four slots are issued before their adds, which keep the slot
// order.
template <int kStride, bool kOpacity, bool kAbs>
__device__ __forceinline__ void sum_pair_partials(const float4* __restrict__ p, int cnt,
                                                  float (&s)[9], float& ax, float& ay) {
  constexpr int kBatch = 4;  // slots whose loads are issued together; the adds stay in slot order
  constexpr int kUsed = (kOpacity || kAbs) ? 3 : 2;
  for (int k0 = 0; k0 < cnt; k0 += kBatch, p += kBatch * kStride) {
    float4 q[kBatch][kUsed];
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      if (k0 + j < cnt)
#pragma unroll
        for (int u = 0; u < kUsed; ++u) q[j][u] = p[j * kStride + u];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      if (k0 + j >= cnt) break;
      const float4 u = q[j][0], v = q[j][1];
      s[0] += u.x; s[1] += u.y; s[2] += u.z; s[3] += u.w;
      s[4] += v.x; s[5] += v.y; s[6] += v.z; s[7] += v.w;
      if constexpr (kOpacity || kAbs) {
        const float4 x = q[j][kUsed - 1];
        if (kOpacity) s[8] += x.x;
        if (kAbs) {
          ax += x.y;
          ay += x.z;
        }
      }
    }
  }
}

// Writes Gaussian i's gradients with respect to the caller's parameters,
// given its derivatives at the rendered (scaled) values: s[0..1] the mean,
// s[2..4] the inverse covariance (A, B, C), s[5..7] the colour, s[8] the
// opacity, and (ax, ay) its absgrad sums.  A is the record's A and shp the
// caller's three shape parameters of Gaussian i (loaded by the caller, so
// that its loads can be issued early).  ok false
// (a culled Gaussian, or no valid binning): zeros.  d_opacity and d_xy_abs
// may be NULL (not written).  The chain rule to the shape parameters:
// Cholesky:
//   dA/da = -2A/a,        dA/db = 2b/(a^2 c^2),  dA/dc = -2b^2/(a^2 c^3)
//   dB/da = b/(a^2 c^2),  dB/db = -1/(a c^2),    dB/dc = 2b/(a c^3)
//   dC/dc = -2/c^3.
// Scale-rotation (u = 1/s_x^2, v = 1/s_y^2, c = cos theta, s = sin theta):
//   d(A, B, C)/du = (c^2, c s, s^2),  d(A, B, C)/dv = (s^2, -c s, c^2),
//   du/ds_x = -2/s_x^3,  dv/ds_y = -2/s_y^3,
//   d(A, B, C)/dtheta = (-2B, (c^2 - s^2)(u - v), 2B).
// d(xy) = d(mean).  With render scale sc the derivatives are taken at the
// scaled shape and multiplied back by sc (lengths and the mean only).
__device__ __forceinline__ void write_gaussian_grads(int i, bool ok, float (&s)[9], float ax, float ay,
                                                     float A, float3 shp, int param, float sc,
                                                     float* __restrict__ d_xy,
                                                     float* __restrict__ d_shape,
                                                     float* __restrict__ d_rgb,
                                                     float* __restrict__ d_opacity,
                                                     float* __restrict__ d_xy_abs) {
  float g0 = 0.f, g1 = 0.f, g2 = 0.f;
  if (ok) {
    const bool rot = param == GS2D_PARAM_SCALE_ROT;
    const float a = sc * shp.x, b = sc * shp.y;
    const float c = rot ? shp.z : sc * shp.z;
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
    ax = ay = 0.f;
  }
  d_xy[2 * i] = s[0];
  d_xy[2 * i + 1] = s[1];
  d_shape[3 * i] = g0;
  d_shape[3 * i + 1] = g1;
  d_shape[3 * i + 2] = g2;
  d_rgb[3 * i] = s[5];
  d_rgb[3 * i + 1] = s[6];
  d_rgb[3 * i + 2] = s[7];
  if (d_opacity) d_opacity[i] = s[8];
  if (d_xy_abs) {
    d_xy_abs[2 * i] = ax;
    d_xy_abs[2 * i + 1] = ay;
  }
}

// Monotone map of a finite float to uint32 (IEEE order, -0 mapped as +0).
__device__ __forceinline__ unsigned int depth_key(float d) {
  unsigned int u = __float_as_uint(d);
  if ((u << 1) == 0u) u = 0u;  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ------------------------------------------------- dependent launches --
// Every kernel is launched with programmatic stream serialization: its
// blocks may be scheduled while the kernel before it on the stream drains,
// and each kernel starts with pdl_wait(), which returns once that kernel
// has completed and its writes are visible (a no-op for launches without
// the attribute).  pdl_trigger() then lets the next kernel start scheduling.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// The tile a block takes and that tile's list range.  With the counting
// sort's launch order (one int4 per slot: tile, start, end, 0; longest lists
// first) both come from one 16-byte load; without it slot i is tile i and
// its range is read from the ranges array.  A slot naming no tile of the
// T (a workspace the binning has not written) gives -1, and the caller's
// block does nothing.
__device__ __forceinline__ int tile_of_slot(const int4* __restrict__ order, int i,
                                            const int2* __restrict__ ranges, int T, int2* rg) {
  if (order) {
    const int4 o = order[i];
    *rg = make_int2(o.y, o.z);
    return (o.x >= 0 && o.x < T) ? o.x : -1;
  }
  *rg = ranges[i];
  return i;
}

__device__ __forceinline__ void pdl_enter() {
  pdl_wait();
  pdl_trigger();
}

// Measured on a B300 (768x512 and 2048x2048 steps in CUDA graphs): within
// +-1.5 % of plain stream order, so it is left off.
constexpr bool kDependentLaunch = false;

// ------------------------------------------------------------- tracing --
// Kernel trace (gs2d_trace_begin / gs2d_trace_end, csrc/trace.cu): while a
// trace is active on the calling host thread, launch() records one of the
// caller's events just before each kernel and one just after it on the
// kernel's stream, so the pair brackets that kernel alone.  During a stream
// capture the records become event nodes of the graph and are re-recorded on
// every replay.
struct Trace {
  const cudaEvent_t* events = nullptr;  // 2 per kernel: before, after
  int capacity = 0;                     // kernels that can be bracketed
  int launched = 0;                     // kernels launched while active
  bool active = false;
};
constexpr int kTraceMaxKernels = 4096;
Trace& trace_state();                              // this host thread's trace
void trace_set_kernel(int i, const void* kernel);  // the i-th traced kernel's host stub
cudaError_t trace_record(cudaEvent_t e, cudaStream_t s);

template <typename... KArgs, typename... Args>
inline cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, Args... args) {
  Trace& tr = trace_state();
  const bool traced = tr.active && tr.launched < tr.capacity;
  if (traced) {
    const cudaError_t e = trace_record(tr.events[2 * tr.launched], s);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = kDependentLaunch ? 1 : 0;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
  if (e != cudaSuccess || !tr.active) return e;
  if (traced) {
    trace_set_kernel(tr.launched, reinterpret_cast<const void*>(kernel));
    const cudaError_t e2 = trace_record(tr.events[2 * tr.launched + 1], s);
    if (e2 != cudaSuccess) return e2;
  }
  ++tr.launched;
  return cudaSuccess;
}

#define GS2D_TRY(expr)                    \
  do {                                    \
    const cudaError_t err_ = (expr);      \
    if (err_ != cudaSuccess) return err_; \
  } while (0)

// ------------------------------------------------------------- launchers --
// Each returns cudaGetLastError() after enqueueing.

cudaError_t launch_project(const gs2d_config& c, int n, const float* xy, const float* chol,
                           const float* rgb, const float* depth, const float* opacity,
                           gs2d_record* rec, int* rect, int* count, cudaStream_t s);

cudaError_t launch_binning(const gs2d_config& c, int n, const gs2d_record* rec, const int* rect,
                           const int* count, long long cap, int* tile_ranges, int* sorted_gid,
                           unsigned char* ws, cudaStream_t s);

// The projection's inputs, for the fused projection + binning.
struct ProjectIn {
  const float *xy, *shape, *rgb, *depth, *opacity;
};

// launch_project followed by launch_binning, with the projection folded into
// the counting sort's histogram kernel where that sort is used.
cudaError_t launch_project_binning(const gs2d_config& c, int n, const ProjectIn& in, gs2d_record* rec,
                                   int* rect, int* count, long long cap, int* tile_ranges,
                                   int* sorted_gid, unsigned char* ws, cudaStream_t s);

cudaError_t launch_render_fwd(const gs2d_config& c, int n, const gs2d_record* rec, const int* ranges,
                              const int* sorted_gid, const float* bg, float* image, float* t_final,
                              int* last, const unsigned char* ws, cudaStream_t s);

cudaError_t launch_loss_l2(int h, int w, const float* image, const float* target, float* loss,
                           float* d_image, unsigned char* ws, cudaStream_t s);

// loss (may be NULL): the fused pass's loss, the sum of the first
// loss_blocks entries of the workspace's loss partials divided by 3HW.
cudaError_t launch_gather(const gs2d_config& c, int n, const float* chol, const gs2d_record* rec,
                          const int* rect, const unsigned char* ws, float* d_xy, float* d_chol,
                          float* d_rgb, float* d_opacity, float* d_bg, float* d_xy_abs, float* loss,
                          int loss_blocks, cudaStream_t s);

cudaError_t launch_render_bwd(const gs2d_config& c, int n, const float* chol,
                              const gs2d_record* rec, const int* rect, const int* ranges,
                              const int* sorted_gid, const float* bg, const float* t_final,
                              const int* last, const float* d_image, float* d_xy, float* d_chol,
                              float* d_rgb, float* d_opacity, float* d_bg, float* d_xy_abs,
                              unsigned char* ws, cudaStream_t s, float* loss = nullptr,
                              int loss_blocks = 0);

// Sum forward that also takes the L2 loss: writes image (if non-NULL),
// dL/dC = scale (C - target) to d_image and one loss partial per block to
// loss_partials; returns the number of blocks in *blocks.  order (may be
// NULL): the tiles in the order their blocks are launched.
// Selective Adam step (csrc/adam.cu): param, m, v [n, width]; rows with
// count[row] == 0 untouched when count is non-NULL.
cudaError_t launch_adam(int n, int width, float* param, const float* grad, float* m, float* v,
                        const int* count, float lr, float beta1, float beta2, float eps, int step,
                        cudaStream_t s);

cudaError_t launch_render_fwd_loss(const gs2d_config& c, int n, const gs2d_record* rec, const int* ranges,
                                   const int* sorted_gid, const float* target, float scale,
                                   float* image, float* d_image, float* loss_partials, int* blocks,
                                   const int4* order, cudaStream_t s);

cudaError_t launch_render_fused_l2(const gs2d_config& c, int n, const float* chol,
                                   const gs2d_record* rec, const int* rect, const int* ranges,
                                   const int* sorted_gid, const float* bg, const float* target,
                                   float* image, float* loss, float* d_xy, float* d_chol,
                                   float* d_rgb, float* d_opacity, float* d_bg, float* d_xy_abs,
                                   unsigned char* ws, cudaStream_t s);

// Start of the merge workspace.
struct MergeHeader {
  int boundary;     // key bin at which the selection stops
  int need;         // pairs to take from the boundary bin, in index order
  int pairs;        // mutual pairs found
  int merges;       // pairs merged
  unsigned int done_a, done_b;
};

#ifdef GS2D_CHECKS
cudaError_t check_word_project(unsigned int* out, bool clear);
cudaError_t check_word_binning(unsigned int* out, bool clear);
cudaError_t check_word_raster_fwd(unsigned int* out, bool clear);
cudaError_t check_word_raster_bwd(unsigned int* out, bool clear);
cudaError_t check_word_fused(unsigned int* out, bool clear);
cudaError_t check_word_merge(unsigned int* out, bool clear);
#endif

size_t merge_workspace_size(long long n);

cudaError_t launch_merge(const gs2d_config& c, int n, const float* xy, const float* shape,
                         const float* rgb, const gs2d_record* rec, const int* count,
                         const int* ranges, const int* sorted_gid, int max_merges, float* out_xy,
                         float* out_shape, float* out_rgb, unsigned char* ws, int* merges_dev,
                         cudaStream_t s);

}  // namespace gs2d
