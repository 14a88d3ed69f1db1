// Per-tile bodies shared by the forward, backward and fused kernels: one
// block per 16x16 tile, one pixel per thread, each warp owning an 8x4-pixel
// sub-block (warp w covers columns 8 (w & 1) .. +7 and rows 4 (w >> 1) .. +3
// of the tile).
//
// The tile's Gaussian list is staged through shared memory (one coalesced
// record gather per thread); each warp then culls a window of staged
// entries with one lane per entry, keeping, in list order, those whose
// pixel box meets its sub-block together with a 32-bit mask of the warp's
// lanes inside the box, so that the per-pixel box test is a single bit test.
#pragma once

#include "gs2d_internal.cuh"

namespace gs2d {

constexpr int kWindow = 64;  // entries culled per warp at a time
constexpr int kCompBatch = 4;  // composite backward: list entries per warp reduction

struct Staged {
  float4 mc;  // mean_x, mean_y, A, 2B
  float4 cr;  // C, r, g, b
};

// Staging area of the sum forward (kWarps warps per block).
template <int kWarps>
struct SumSmem {
  Staged g[256];
  uint2 box[256];
  uint2 list[kWarps][kWindow];  // (staged index, lane mask)
  float red[kWarps];
};

// Loads records sorted_gid[rb .. rb + cnt) into the staging area (cnt <= 256).
template <typename Smem>
__device__ __forceinline__ void stage_records(Smem& sm, int rb, int cnt, int tid, int nthreads, int n,
                                              const float4* __restrict__ rec,
                                              const int* __restrict__ sorted_gid) {
  for (int k = tid; k < cnt; k += nthreads) {
    int g = sorted_gid[rb + k];
    if (!check_ok(g >= 0 && g < n, kCheckGaussian)) g = 0;
    const float4* r = rec + 3 * size_t(g);
    const float4 p0 = r[0], p1 = r[1], p2 = r[2];
    sm.g[k].mc = make_float4(p0.x, p0.y, p0.z, 2.0f * p0.w);
    sm.g[k].cr = p1;
    sm.box[k] = make_uint2(__float_as_uint(p2.x), __float_as_uint(p2.y));
  }
}

// Sum forward over the list [rg.x, rg.y) for the calling thread's pixel
// (pixel centre pxf, pyf; the warp's sub-block starts at bx0, by0):
//     C(p) = sum over touching Gaussians i of rgb_i * exp(-q/2)
// (GaussianImage project page, Overview: accumulated-sum rendering; FlashImgs
// README: additive RGB, gate folded into the colour).  Every thread of the
// block must call it.
template <int kWarps>
__device__ __forceinline__ float3 sum_tile_forward(SumSmem<kWarps>& sm, int2 rg, int bx0, int by0,
                                                   float pxf, float pyf, float kk, int n,
                                                   const float4* __restrict__ rec,
                                                   const int* __restrict__ sorted_gid) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const unsigned int lt = (1u << lane) - 1u, bit = 1u << lane;
  uint2* list = sm.list[warp];
  float ar = 0.f, ag = 0.f, ab = 0.f;
  for (int rb = rg.x; rb < rg.y; rb += 256) {
    const int cnt = min(256, rg.y - rb);
    if (rb != rg.x) __syncthreads();  // the previous round is no longer read
    stage_records(sm, rb, cnt, tid, kWarps * 32, n, rec, sorted_gid);
    __syncthreads();
    for (int wb = 0; wb < cnt; wb += kWindow) {
      const int wend = min(wb + kWindow, cnt);
      int nl = 0;
#pragma unroll
      for (int j0 = 0; j0 < kWindow; j0 += 32) {
        const int j = wb + j0 + lane;
        unsigned int m = 0;
        if (j < wend) m = box_lanes(sm.box[j], bx0, by0);
        const unsigned int hits = __ballot_sync(0xffffffffu, m != 0u);
        if (m) list[nl + __popc(hits & lt)] = make_uint2(unsigned(j), m);
        nl += __popc(hits);
      }
      __syncwarp();
      int e = 0;
      for (; e + 1 < nl; e += 2) {
        const uint2 u0 = list[e], u1 = list[e + 1];
        const Staged s0 = sm.g[u0.x], s1 = sm.g[u1.x];
        const float q0 = touch_q(__fsub_rn(pxf, s0.mc.x), __fsub_rn(pyf, s0.mc.y), s0.mc.z, s0.mc.w, s0.cr.x);
        const float q1 = touch_q(__fsub_rn(pxf, s1.mc.x), __fsub_rn(pyf, s1.mc.y), s1.mc.z, s1.mc.w, s1.cr.x);
        float w0 = ex2_approx(q0 * kNegHalfLog2e);
        float w1 = ex2_approx(q1 * kNegHalfLog2e);
        w0 = (q0 <= kk && (u0.y & bit)) ? w0 : 0.f;
        w1 = (q1 <= kk && (u1.y & bit)) ? w1 : 0.f;
        ar = fmaf(s0.cr.y, w0, ar);
        ag = fmaf(s0.cr.z, w0, ag);
        ab = fmaf(s0.cr.w, w0, ab);
        ar = fmaf(s1.cr.y, w1, ar);
        ag = fmaf(s1.cr.z, w1, ag);
        ab = fmaf(s1.cr.w, w1, ab);
      }
      if (e < nl) {
        const uint2 u0 = list[e];
        const Staged s0 = sm.g[u0.x];
        const float q0 = touch_q(__fsub_rn(pxf, s0.mc.x), __fsub_rn(pyf, s0.mc.y), s0.mc.z, s0.mc.w, s0.cr.x);
        float w0 = ex2_approx(q0 * kNegHalfLog2e);
        w0 = (q0 <= kk && (u0.y & bit)) ? w0 : 0.f;
        ar = fmaf(s0.cr.y, w0, ar);
        ag = fmaf(s0.cr.z, w0, ag);
        ab = fmaf(s0.cr.w, w0, ab);
      }
      __syncwarp();
    }
  }
  return make_float3(ar, ag, ab);
}

struct CompSmem {
  Staged g[256];
  uint2 box[256];
  float op[256];
  uint2 list[8][kWindow];
};

struct CompFwdOut {
  float r, g, b;  // colour before the background term
  float T;        // transmittance after the last contributor
  int last;       // 1 + list position of the last contributor (0: none)
  // kMid: the state in front of list position `mid` (after every entry
  // before it): transmittance and colour so far
  float Tm, mr, mg, mb;
};

// Composite forward for the calling thread's pixel (256 threads), front to
// back in list (depth) order (DrawingWithGaussians README, Overview: alpha
// compositing over a trainable background):
//     while T >= t_min: alpha = o_i exp(-q/2); C += rgb_i alpha T; T *= 1 - alpha
// The caller adds T * background.  kMid: also records the state in front of
// list position `mid` (CompFwdOut::Tm, mr, mg, mb).  Every thread of the
// block must call it.
template <bool kMid = false>
__device__ __forceinline__ CompFwdOut comp_tile_forward(CompSmem& sm, const gs2d_config& c, int2 rg,
                                                        int bx0, int by0, float pxf, float pyf,
                                                        bool inside, float kk, int n,
                                                        const float4* __restrict__ rec,
                                                        const int* __restrict__ sorted_gid,
                                                        int mid = 0) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const unsigned int lt = (1u << lane) - 1u, bit = 1u << lane;
  uint2* list = sm.list[warp];
  float ar = 0.f, ag = 0.f, ab = 0.f, T = 1.f;
  float Tm = 1.f, mr = 0.f, mg = 0.f, mb = 0.f;
  bool have_mid = false;
  int lst = 0;
  bool done = !inside;
  for (int rb = rg.x; rb < rg.y; rb += 256) {
    if (__syncthreads_and(done)) break;
    const int cnt = min(256, rg.y - rb);
    if (tid < cnt) {
      int g = sorted_gid[rb + tid];
      if (!check_ok(g >= 0 && g < n, kCheckGaussian)) g = 0;
      const float4* r = rec + 3 * size_t(g);
      const float4 p0 = r[0], p1 = r[1], p2 = r[2];
      sm.g[tid].mc = make_float4(p0.x, p0.y, p0.z, 2.0f * p0.w);
      sm.g[tid].cr = p1;
      sm.box[tid] = make_uint2(__float_as_uint(p2.x), __float_as_uint(p2.y));
      sm.op[tid] = p2.z;
    }
    __syncthreads();
    for (int wb = 0; wb < cnt; wb += kWindow) {
      if (__all_sync(0xffffffffu, done)) break;
      const int wend = min(wb + kWindow, cnt);
      int nl = 0;
#pragma unroll
      for (int j0 = 0; j0 < kWindow; j0 += 32) {
        const int j = wb + j0 + lane;
        unsigned int m = 0;
        if (j < wend) m = box_lanes(sm.box[j], bx0, by0);
        const unsigned int hits = __ballot_sync(0xffffffffu, m != 0u);
        if (m) list[nl + __popc(hits & lt)] = make_uint2(unsigned(j), m);
        nl += __popc(hits);
      }
      __syncwarp();
      // front to back; the weights of two entries are formed together (they
      // do not depend on T), then the transmittance steps run in order
      auto step = [&](uint2 u, const Staged& s, float q, float w) {
        if constexpr (kMid) {
          if (!have_mid && rb - rg.x + int(u.x) >= mid) {  // entries from here on are at or past mid
            have_mid = true;
            Tm = T;
            mr = ar;
            mg = ag;
            mb = ab;
          }
        }
        if (q <= kk && (u.y & bit) && !done) {
          if (T < c.t_min) {
            done = true;
          } else {
            const float alpha = sm.op[u.x] * w;
            const float aT = alpha * T;
            ar = fmaf(s.cr.y, aT, ar);
            ag = fmaf(s.cr.z, aT, ag);
            ab = fmaf(s.cr.w, aT, ab);
            T = T * (1.0f - alpha);
            lst = rb - rg.x + int(u.x) + 1;
          }
        }
      };
      int e = 0;
      for (; e + 1 < nl; e += 2) {
        const uint2 u0 = list[e], u1 = list[e + 1];
        const Staged s0 = sm.g[u0.x], s1 = sm.g[u1.x];
        const float q0 = touch_q(__fsub_rn(pxf, s0.mc.x), __fsub_rn(pyf, s0.mc.y), s0.mc.z, s0.mc.w, s0.cr.x);
        const float q1 = touch_q(__fsub_rn(pxf, s1.mc.x), __fsub_rn(pyf, s1.mc.y), s1.mc.z, s1.mc.w, s1.cr.x);
        const float w0 = ex2_approx(q0 * kNegHalfLog2e), w1 = ex2_approx(q1 * kNegHalfLog2e);
        step(u0, s0, q0, w0);
        step(u1, s1, q1, w1);
      }
      if (e < nl) {
        const uint2 u = list[e];
        const Staged s = sm.g[u.x];
        const float q = touch_q(__fsub_rn(pxf, s.mc.x), __fsub_rn(pyf, s.mc.y), s.mc.z, s.mc.w, s.cr.x);
        step(u, s, q, ex2_approx(q * kNegHalfLog2e));
      }
      __syncwarp();
    }
    __syncthreads();
  }
  if (kMid && !have_mid) {  // no entry at or past mid reached this pixel's warp
    Tm = T;
    mr = ar;
    mg = ag;
    mb = ab;
  }
  return CompFwdOut{ar, ag, ab, T, lst, Tm, mr, mg, mb};
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Butterfly reduce-scatter of N = 2^m (m <= 5) per-lane values over the
// warp: returns, in lane L, the warp total of value L >> (5 - m), each value
// summed in the same fixed order on every run.  The first m steps halve the
// values a lane carries (lane bit 4 picks the upper half first, then bit 3,
// ...); the remaining steps add whole totals.
template <int N>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[N], int lane) {
  static_assert(N >= 1 && N <= 32 && (N & (N - 1)) == 0, "N must be a power of two <= 32");
#pragma unroll
  for (int half = N / 2, o = 16; half >= 1; half >>= 1, o >>= 1) {
    const bool up = lane & o;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float keep = up ? v[i + half] : v[i], send = up ? v[i] : v[i + half];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  float c = v[0];
#pragma unroll
  for (int o = 16 / N; o >= 1; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  return c;
}

// Sum of one value over the kWarps warps of a block: warp totals, then the
// warps in order.  The result is valid in thread 0.  `red` holds kWarps
// floats; the caller synchronises before reusing it.
template <int kWarps>
__device__ __forceinline__ float block_sum_ordered(float v, float* red) {
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.f;
  if (threadIdx.x == 0)
    for (int w = 0; w < kWarps; ++w) s += red[w];
  return s;
}

constexpr int kCompChunk = 128;
constexpr int kCompVals = 9;

template <bool kAbs>
struct CompStage {
  float4 mc[kCompChunk];  // mean_x, mean_y, A, 2B
  float4 cr[kCompChunk];  // C, r, g, b
  uint2 box[kCompChunk];
  float op[kCompChunk];
  int gid[kCompChunk];
  uint2 list[8][kCompChunk];            // (chunk index, lane mask) per warp
  float acc[8][kCompChunk][kCompVals];  // per-warp partials, summed over warps in order
  float acc_abs[kAbs ? 8 : 1][kAbs ? kCompChunk : 1][2];  // per-warp absgrad sums
  float bgred[8][3];
};

// Composite backward for the calling thread's pixel (256 threads), walking
// the tile's list back to front from the pixel's last contributor, over the
// list positions [lo, hi) only (the whole list by default).  T is the
// transmittance behind position hi - 1 (the pixel's final transmittance when
// hi is the list's end), (Sr0, Sg0, Sb0) the colour accumulated behind it
// including T_final * bg (T * bg when hi is the end), lst the pixel's last
// contributor, (gr, gg, gb) its dL/dC.  with_bg: also write the tile's
// background partial (T is then the final transmittance).  With alpha = o w, T_i the transmittance in front of Gaussian i and
// S the colour accumulated behind it (including T_final * bg):
//     dL/dalpha = sum_k g_k (rgb_k T_i - S_k / (1 - alpha)),
//     dL/do = w dL/dalpha,  dL/dw = o dL/dalpha,  dL/drgb_k = g_k alpha T_i,
//     dL/dbg_k = sum over pixels of T_final g_k.
// Per (warp, Gaussian) the nine partial derivatives are reduced over the
// warp and kept in a per-warp slot; the slots are summed in warp order and
// written to the pair's emission slot (3 float4 per pair).  The tile's
// background partial goes to tile_partials[tile].  kAbs: also the absgrad
// sums, over the pair's pixels, of |each pixel's share of dL/dmu_x| and of
// dL/dmu_y (slot's third float4, .y and .z).
template <bool kAbs>
__device__ __forceinline__ void comp_tile_backward(
    CompStage<kAbs>& sm, const gs2d_config& c, int tile, int tx, int ty, int2 rg, int bx0, int by0,
    float pxf, float pyf, bool inside, float kk, float T, int lst, float gr, float gg, float gb,
    int n, long long pairs, const float* __restrict__ bg, const float4* __restrict__ rec,
    const int4* __restrict__ rect, const int* __restrict__ sorted_gid,
    const int* __restrict__ offsets, float4* __restrict__ partials,
    float4* __restrict__ tile_partials, int lo = 0, int hi = 0x7fffffff, bool with_bg = true,
    float Sr0 = 0.f, float Sg0 = 0.f, float Sb0 = 0.f) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const unsigned int lt = (1u << lane) - 1u, bit = 1u << lane;
  const float bgr = bg ? bg[0] : 0.f, bgg = bg ? bg[1] : 0.f, bgb = bg ? bg[2] : 0.f;
  uint2* list = sm.list[warp];
  // background gradient: T_final * g summed over the tile, fixed order
  if (with_bg) {
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
      tile_partials[tile] = make_float4(x, y, z, 0.f);
    }
  }
  float Sr = with_bg ? T * bgr : Sr0, Sg = with_bg ? T * bgg : Sg0, Sb = with_bg ? T * bgb : Sb0;
  const int len = rg.y - rg.x;
  hi = min(hi, len);
  lo = max(lo, 0);
  for (int ci = (hi - 1) / kCompChunk; lo < hi && ci >= lo / kCompChunk; --ci) {
    const int cb = rg.x + ci * kCompChunk;
    const int cnt = min(kCompChunk, rg.y - cb);
    // the chunk's entries in [lo, hi)
    const int jlo = max(0, lo - ci * kCompChunk), jhi = min(cnt, hi - ci * kCompChunk);
    if (tid >= jlo && tid < jhi) {
      int gid = sorted_gid[cb + tid];
      if (!check_ok(gid >= 0 && gid < n, kCheckGaussian)) gid = 0;
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
    for (int j0 = jlo; j0 < jhi; j0 += 32) {
      const int j = j0 + lane;
      unsigned int m = 0;
      if (j < jhi) {
        m = box_lanes(sm.box[j], bx0, by0);
        if (!m) {
#pragma unroll
          for (int v = 0; v < kCompVals; ++v) sm.acc[warp][j][v] = 0.f;
          if constexpr (kAbs) sm.acc_abs[warp][j][0] = sm.acc_abs[warp][j][1] = 0.f;
        }
      }
      const unsigned int hits = __ballot_sync(0xffffffffu, m != 0u);
      if (m) list[nl + __popc(hits & lt)] = make_uint2(unsigned(j), m);
      nl += __popc(hits);
    }
    __syncwarp();
    // Four list entries at a time, back to front: each lane's transmittance
    // and colour-behind chain runs through them in order, then the warp
    // reduces the four entries' values together (one reduce-scatter of 32
    // values and one of the rest) instead of one reduction chain per entry.
    for (int e0 = nl - 1; e0 >= 0; e0 -= kCompBatch) {
      float v[kCompBatch * 8];
      float x[kCompBatch * (kAbs ? 4 : 1)];  // v8 per entry, then (kAbs) absgrad x, y per entry
      int jj[kCompBatch];
#pragma unroll
      for (int k = 0; k < kCompBatch; ++k) {
        const int e = e0 - k;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) v[k * 8 + c8] = 0.f;
        x[k] = 0.f;
        if constexpr (kAbs) x[kCompBatch + 2 * k] = x[kCompBatch + 2 * k + 1] = 0.f;
        jj[k] = -1;
        if (e < 0) continue;  // warp-uniform
        const uint2 u = list[e];
        const int j = int(u.x);
        jj[k] = j;
        const int idx = cb - rg.x + j;  // position in the tile's list
        const float4 mc = sm.mc[j];
        const float4 cr = sm.cr[j];
        const float dx = __fsub_rn(pxf, mc.x);
        const float dy = __fsub_rn(pyf, mc.y);
        const float q = touch_q(dx, dy, mc.z, mc.w, cr.x);
        const bool act = inside && (u.y & bit) && idx < lst && q <= kk;
        if (act) {
          const float o = sm.op[j];
          const float w = ex2_approx(q * kNegHalfLog2e);
          const float alpha = o * w;
          const float inv = rcp_approx(1.0f - alpha);
          const float Tb = T * inv;  // transmittance in front of this Gaussian
          const float aT = alpha * Tb;
          const float dal = gr * (cr.y * Tb - Sr * inv) + gg * (cr.z * Tb - Sg * inv) +
                            gb * (cr.w * Tb - Sb * inv);
          const float t = w * o * dal;
          const float t0x = t * dx, t0y = t * dy;
          v[k * 8 + 0] = t0x;
          v[k * 8 + 1] = t0y;
          v[k * 8 + 2] = t0x * dx;
          v[k * 8 + 3] = t0x * dy;
          v[k * 8 + 4] = t0y * dy;
          v[k * 8 + 5] = gr * aT;
          v[k * 8 + 6] = gg * aT;
          v[k * 8 + 7] = gb * aT;
          x[k] = dal * w;
          if constexpr (kAbs) {
            const float Bh = 0.5f * mc.w;
            x[kCompBatch + 2 * k] = fabsf(fmaf(mc.z, t0x, Bh * t0y));
            x[kCompBatch + 2 * k + 1] = fabsf(fmaf(Bh, t0x, cr.x * t0y));
          }
          Sr = fmaf(cr.y, aT, Sr);
          Sg = fmaf(cr.z, aT, Sg);
          Sb = fmaf(cr.w, aT, Sb);
          T = Tb;
        }
      }
      // lane L: the total of v[L] = entry L / 8, value L % 8
      const float tot = warp_reduce_scatter<kCompBatch * 8>(v, lane);
      {
        const int k = lane >> 3;
        const int j = k == 0 ? jj[0] : k == 1 ? jj[1] : k == 2 ? jj[2] : jj[3];
        if (j >= 0) sm.acc[warp][j][lane & 7] = tot;
      }
      constexpr int kX = kCompBatch * (kAbs ? 4 : 1);
      const float totx = warp_reduce_scatter<kX>(x, lane);  // lane L: x[L >> (5 - log2 kX)]
      if ((lane & (32 / kX - 1)) == 0) {
        const int m = lane / (32 / kX);
        const int k = m < kCompBatch ? m : (m - kCompBatch) >> 1;
        const int j = k == 0 ? jj[0] : k == 1 ? jj[1] : k == 2 ? jj[2] : jj[3];
        if (j >= 0) {
          if (m < kCompBatch)
            sm.acc[warp][j][8] = totx;
          else if constexpr (kAbs)
            sm.acc_abs[warp][j][(m - kCompBatch) & 1] = totx;
        }
      }
    }
    __syncthreads();
    if (tid >= jlo && tid < jhi) {
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
      float ax = 0.f, ay = 0.f;
      if constexpr (kAbs)
        for (int w = 0; w < 8; ++w) {
          ax += sm.acc_abs[w][tid][0];
          ay += sm.acc_abs[w][tid][1];
        }
      if (check_ok(slot >= 0 && slot < pairs, kCheckPartial)) {
        float4* out = partials + 3 * size_t(slot);
        out[0] = make_float4(fmaf(A, s[0], B * s[1]), fmaf(B, s[0], C * s[1]), -0.5f * s[2], -s[3]);
        out[1] = make_float4(-0.5f * s[4], s[5], s[6], s[7]);
        out[2] = make_float4(s[8], ax, ay, 0.f);
      }
    }
    __syncthreads();
  }
}

}  // namespace gs2d
