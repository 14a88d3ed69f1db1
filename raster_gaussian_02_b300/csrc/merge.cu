// Moment-matching merge, one round (FlashImgs README, merge -- Best quality
// pipeline: an overcomplete fit merged down "via moment-matching"; the CUDA
// library's merge_gaussians).  Sum mode.
//
// The pages leave the choice of pairs and the weights open; this follows one
// reading, step for step:
//   Sigma per Gaussian (scale-rotation: cos and sin from sincos_fp32);
//   cost(i, j) = d^T M^-1 d, d = mu_i - mu_j, M = (Sigma_i + Sigma_j) / 2, in a
//   fixed FP32 sequence (+inf when det M <= 0, the quadratic form clamped at
//   0) so that the pairing, an integer decision, is the same wherever the
//   sequence is evaluated;
//   candidates of i: the Gaussians listed in the tile of its rendered mean
//   (clamped to the image); nn(i): least cost, ties to the smaller index;
//   pairs: i < j = nn(i) with nn(j) = i; at most max_merges of them, ordered
//   by the top 16 bits of the FP32 cost, ties by index;
//   weights w = sqrt(det Sigma) (|r| + |g| + |b|); the merged mean and
//   covariance are the w-weighted moments; each colour channel keeps its
//   mass; the output lists the Gaussians in index order, a pair in the slot
//   of its lower index.
// Every operation of the decision is explicitly rounded (no contraction).
// The merged values are computed in double.
//
// Kernels: k_merge_prep, k_merge_nn (one block per tile: the tile's list is
// staged in shared memory once and searched by the Gaussians whose mean lies
// in the tile), k_merge_pairs (+ key histogram),
// k_merge_threshold (one block), k_merge_count/k_merge_take (rank among the
// boundary key's pairs in index order), k_merge_count/k_merge_write (output
// slots, merged values).  The counts use the reduce-then-scan pattern of the
// binning: no block waits on another.
#include "gs2d_internal.cuh"

namespace gs2d {

namespace {

constexpr int kMergeThreads = 256;
constexpr int kKeyBins = 1 << 16;

struct MergeLayout {
  size_t hist, mrec, msyy, mtile, cost, nn, key, take, drop, block_a, block_b, total;
};

MergeLayout merge_layout(long long n) {
  MergeLayout L{};
  const long long nb = (n + kMergeThreads - 1) / kMergeThreads + 1;
  size_t o = 256;
  L.hist = o;
  o = align256(o + 4 * size_t(kKeyBins));
  L.mrec = o;  // (x, y, Sxx, Sxy) FP32
  o = align256(o + 16 * size_t(n));
  L.msyy = o;  // Syy FP32
  o = align256(o + 4 * size_t(n));
  L.mtile = o;  // tile of the rendered mean, -1 when culled
  o = align256(o + 4 * size_t(n));
  L.cost = o;
  o = align256(o + 4 * size_t(n));
  L.nn = o;
  o = align256(o + 4 * size_t(n));
  L.key = o;
  o = align256(o + 4 * size_t(n));
  L.take = o;
  o = align256(o + 4 * size_t(n));
  L.drop = o;
  o = align256(o + 4 * size_t(n));
  L.block_a = o;
  o = align256(o + 4 * size_t(nb));
  L.block_b = o;
  o = align256(o + 4 * size_t(nb));
  L.total = o;
  return L;
}

__device__ __forceinline__ double dmul(double a, double b) { return __dmul_rn(a, b); }
__device__ __forceinline__ double dadd(double a, double b) { return __dadd_rn(a, b); }
__device__ __forceinline__ double dsub(double a, double b) { return __dsub_rn(a, b); }
__device__ __forceinline__ double ddiv(double a, double b) { return __ddiv_rn(a, b); }

__device__ __forceinline__ float fmul(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ float fadd(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float fsub(float a, float b) { return __fsub_rn(a, b); }

// Sigma (FP32, each product rounded) for the pairing cost, the mean, and the
// tile of the rendered mean (clamped to the image); nn/cost start empty.
__global__ void __launch_bounds__(kMergeThreads)
k_merge_prep(gs2d_config c, int n, int tiles_x, const float* __restrict__ xy,
             const float* __restrict__ shape, const float4* __restrict__ rec,
             const int* __restrict__ count, float4* __restrict__ mrec, float* __restrict__ msyy,
             int* __restrict__ mtile, int* __restrict__ nn, float* __restrict__ cost) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float p0 = shape[3 * i], p1 = shape[3 * i + 1], p2 = shape[3 * i + 2];
  float sxx, sxy, syy;
  if (c.param == GS2D_PARAM_SCALE_ROT) {
    float sn, cs;
    sincos_fp32(p2, &sn, &cs);
    const float x2 = fmul(p0, p0), y2 = fmul(p1, p1);
    sxx = fadd(fmul(fmul(cs, cs), x2), fmul(fmul(sn, sn), y2));
    sxy = fmul(fmul(cs, sn), fsub(x2, y2));
    syy = fadd(fmul(fmul(sn, sn), x2), fmul(fmul(cs, cs), y2));
  } else {
    sxx = fmul(p0, p0);
    sxy = fmul(p0, p1);
    syy = fadd(fmul(p1, p1), fmul(p2, p2));
  }
  mrec[i] = make_float4(xy[2 * i], xy[2 * i + 1], sxx, sxy);
  msyy[i] = syy;
  int t = -1;
  if (count[i] > 0) {
    const float4 r0 = rec[3 * size_t(i)];  // the rendered (scaled) mean
    const float px = floorf(r0.x), py = floorf(r0.y);
    const int col = px < 0.0f ? 0 : (px > float(c.width - 1) ? c.width - 1 : int(px));
    const int row = py < 0.0f ? 0 : (py > float(c.height - 1) ? c.height - 1 : int(py));
    t = (row / kTile) * tiles_x + col / kTile;
  }
  mtile[i] = t;
  nn[i] = -1;
  cost[i] = __int_as_float(0x7f800000);  // +inf
}

// cost(i, j) = max(m2 dx^2 - 2 m1 dx dy + m0 dy^2, 0) / (m0 m2 - m1^2) with
// M = (Si + Sj) / 2, in this FP32 order; +inf when det M <= 0.
__device__ __forceinline__ float merge_cost(float4 a, float ayy, float4 b, float byy) {
  const float m0 = fmul(0.5f, fadd(a.z, b.z));
  const float m1 = fmul(0.5f, fadd(a.w, b.w));
  const float m2 = fmul(0.5f, fadd(ayy, byy));
  const float dx = fsub(a.x, b.x), dy = fsub(a.y, b.y);
  const float det = fsub(fmul(m0, m2), fmul(m1, m1));
  if (!(det > 0.0f)) return __int_as_float(0x7f800000);
  const float num = fadd(fsub(fmul(fmul(m2, dx), dx), fmul(fmul(fmul(2.0f, m1), dx), dy)),
                         fmul(fmul(m0, dy), dy));
  return __fdiv_rn(num > 0.0f ? num : 0.0f, det);  // (-0 and NaN clamp to +0)
}

// One block per tile.  Thread k of a member round owns list entry k of the
// round when that Gaussian's mean lies in this tile (every valid Gaussian is
// listed in its mean's tile: its box holds the pixel nearest its mean), and
// finds its least-cost candidate over the whole list, staged 256 at a time.
__global__ void __launch_bounds__(kMergeThreads)
k_merge_nn(int n, const int2* __restrict__ ranges, const int* __restrict__ sorted_gid,
           const float4* __restrict__ mrec, const float* __restrict__ msyy,
           const int* __restrict__ mtile, int* __restrict__ nn, float* __restrict__ cost) {
  __shared__ float4 s_rec[kMergeThreads];
  __shared__ float s_syy[kMergeThreads];
  __shared__ int s_gid[kMergeThreads];
  const int t = blockIdx.x, tid = threadIdx.x;
  int2 rg = ranges[t];
  if (!check_ok(rg.x >= 0 && rg.x <= rg.y, kCheckRange)) rg = make_int2(0, 0);
  for (int mc = rg.x; mc < rg.y; mc += kMergeThreads) {
    const int k = mc + tid;
    int g = k < rg.y ? sorted_gid[k] : -1;
    if (g >= 0 && !check_ok(g < n, kCheckMerge)) g = -1;
    const bool member = g >= 0 && mtile[g] == t;
    float4 me = make_float4(0.f, 0.f, 0.f, 0.f);
    float myy = 0.f;
    if (member) {
      me = mrec[g];
      myy = msyy[g];
    }
    int best = -1;
    float bc = __int_as_float(0x7f800000);
    for (int cc = rg.x; cc < rg.y; cc += kMergeThreads) {
      const int cnt = min(kMergeThreads, rg.y - cc);
      __syncthreads();  // the previous chunk is no longer read
      if (tid < cnt) {
        int j = sorted_gid[cc + tid];
        if (!check_ok(j >= 0 && j < n, kCheckMerge)) j = 0;
        s_rec[tid] = mrec[j];
        s_syy[tid] = msyy[j];
        s_gid[tid] = j;
      }
      __syncthreads();
      if (member)
        for (int q = 0; q < cnt; ++q) {
          const int j = s_gid[q];
          if (j == g) continue;
          const float cj = merge_cost(me, myy, s_rec[q], s_syy[q]);
          if (cj < bc || (cj == bc && j < best)) {
            bc = cj;
            best = j;
          }
        }
    }
    if (member) {
      nn[g] = best;
      cost[g] = bc;
    }
  }
}

// Mutual pairs (lower index) get a key (top 16 bits of the FP32 cost) and a
// histogram count; other Gaussians get key kKeyBins (none).
__global__ void __launch_bounds__(kMergeThreads)
k_merge_pairs(int n, const int* __restrict__ nn, const float* __restrict__ cost,
              unsigned int* __restrict__ key, unsigned int* __restrict__ hist) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int j = nn[i];
  unsigned int k = kKeyBins;
  if (j > i && check_ok(j < n, kCheckMerge) && nn[j] == i) {
    k = __float_as_uint(cost[i]) >> 16;
    atomicAdd(&hist[k], 1u);
  }
  key[i] = k;
}

// One block of 1024 threads: the first bin b at which the cumulative pair
// count reaches max_merges; pairs below b all merge, `need` more from b.
__global__ void __launch_bounds__(1024)
k_merge_threshold(int max_merges, const unsigned int* __restrict__ hist, MergeHeader* hdr) {
  __shared__ unsigned int s_tot[1024];
  const int tid = threadIdx.x;
  constexpr int kPer = kKeyBins / 1024;
  unsigned int sum = 0;
  for (int k = 0; k < kPer; ++k) sum += hist[tid * kPer + k];
  s_tot[tid] = sum;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {  // inclusive scan (Hillis-Steele)
    const unsigned int v = tid >= o ? s_tot[tid - o] : 0u;
    __syncthreads();
    s_tot[tid] += v;
    __syncthreads();
  }
  const unsigned int total = s_tot[1023];
  const unsigned int want = max_merges < 0 ? 0u : unsigned(max_merges);
  if (tid == 0) {
    hdr->pairs = int(total);
    hdr->merges = int(total < want ? total : want);
    if (total <= want) {
      hdr->boundary = kKeyBins;  // take every pair
      hdr->need = 0;
    }
  }
  if (total <= want) return;
  const unsigned int before = tid > 0 ? s_tot[tid - 1] : 0u;
  if (before < want && s_tot[tid] >= want) {  // the crossing lies in this thread's bins
    unsigned int run = before;
    for (int k = 0; k < kPer; ++k) {
      const unsigned int h = hist[tid * kPer + k];
      if (run + h >= want) {
        hdr->boundary = tid * kPer + k;
        hdr->need = int(want - run);
        break;
      }
      run += h;
    }
  }
  if (want == 0 && tid == 0) {
    hdr->boundary = 0;
    hdr->need = 0;
  }
}

__device__ __forceinline__ int block_excl_scan_int(int x, int* total) {
  __shared__ int warp_tot[kMergeThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kMergeThreads / 32; ++w) {
    const int v = warp_tot[w];
    if (w < warp) before += v;
    all += v;
  }
  __syncthreads();
  *total = all;
  return before + incl - x;
}

// Flags of a count: 0 = boundary pairs (key == boundary), 1 = kept Gaussians.
template <int kWhich>
__device__ __forceinline__ int merge_flag(int i, int n, const MergeHeader* hdr,
                                          const unsigned int* key, const int* drop) {
  if (i >= n) return 0;
  if (kWhich == 0) return key[i] == unsigned(hdr->boundary) ? 1 : 0;
  return drop[i] ? 0 : 1;
}

// Block totals of a flag; the last block scans them into block offsets.
template <int kWhich>
__global__ void __launch_bounds__(kMergeThreads)
k_merge_count(int n, MergeHeader* hdr, const unsigned int* __restrict__ key,
              const int* __restrict__ drop, int* __restrict__ block_off) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  int total;
  block_excl_scan_int(merge_flag<kWhich>(i, n, hdr, key, drop), &total);
  __shared__ bool last;
  unsigned int* done = kWhich == 0 ? &hdr->done_a : &hdr->done_b;
  if (threadIdx.x == 0) {
    block_off[blockIdx.x] = total;
    __threadfence();
    last = atomicAdd(done, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  const volatile int* bo = block_off;
  int carry = 0;
  for (int b0 = 0; b0 < int(gridDim.x); b0 += kMergeThreads) {
    const int b = b0 + threadIdx.x;
    const int v = b < int(gridDim.x) ? bo[b] : 0;
    int chunk;
    const int ex = block_excl_scan_int(v, &chunk);
    if (b < int(gridDim.x)) block_off[b] = carry + ex;
    carry += chunk;
  }
}

// take[i]: i is the lower index of a merged pair; its partner is dropped.
__global__ void __launch_bounds__(kMergeThreads)
k_merge_take(int n, const MergeHeader* __restrict__ hdr, const unsigned int* __restrict__ key,
             const int* __restrict__ nn, const int* __restrict__ block_off, int* __restrict__ take,
             int* __restrict__ drop) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  int total;
  const int rank = block_off[blockIdx.x] + block_excl_scan_int(merge_flag<0>(i, n, hdr, key, nullptr), &total);
  if (i >= n) return;
  const unsigned int k = key[i];
  const unsigned int b = unsigned(hdr->boundary);
  const bool t = k < unsigned(kKeyBins) && (k < b || (k == b && rank < hdr->need));
  take[i] = t ? 1 : 0;
  if (t && check_ok(nn[i] >= 0 && nn[i] < n, kCheckMerge)) drop[nn[i]] = 1;  // pairs are disjoint: every partner is dropped once
}

// Sigma in double from the shape, in the order the merged values use it.
__device__ __forceinline__ void sigma_double(int param, const float* P, double S[3]) {
  if (param == GS2D_PARAM_SCALE_ROT) {
    float sn, cs;
    sincos_fp32(P[2], &sn, &cs);
    const double c = cs, s = sn;
    const double x2 = dmul(double(P[0]), double(P[0])), y2 = dmul(double(P[1]), double(P[1]));
    S[0] = dadd(dmul(dmul(c, c), x2), dmul(dmul(s, s), y2));
    S[1] = dmul(dmul(c, s), dsub(x2, y2));
    S[2] = dadd(dmul(dmul(s, s), x2), dmul(dmul(c, c), y2));
  } else {
    const double a = P[0], b = P[1], c = P[2];
    S[0] = dmul(a, a);
    S[1] = dmul(a, b);
    S[2] = dadd(dmul(b, b), dmul(c, c));
  }
}

__global__ void __launch_bounds__(kMergeThreads)
k_merge_write(int n, int param, const float* __restrict__ xy, const float* __restrict__ shape,
              const float* __restrict__ rgb,
              const int* __restrict__ nn, const int* __restrict__ take, const int* __restrict__ drop,
              const int* __restrict__ block_off, float* __restrict__ out_xy,
              float* __restrict__ out_shape, float* __restrict__ out_rgb) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  int total;
  const int keep = (i < n && !drop[i]) ? 1 : 0;
  const int o = block_off[blockIdx.x] + block_excl_scan_int(keep, &total);
  if (!keep || !check_ok(o >= 0 && o < n, kCheckMerge)) return;
  if (!take[i]) {
    out_xy[2 * o] = xy[2 * i];
    out_xy[2 * o + 1] = xy[2 * i + 1];
    for (int d = 0; d < 3; ++d) {
      out_shape[3 * o + d] = shape[3 * i + d];
      out_rgb[3 * o + d] = rgb[3 * i + d];
    }
    return;
  }
  const int j = nn[i];
  if (!check_ok(j >= 0 && j < n, kCheckMerge)) return;
  double Si[3], Sj[3];
  sigma_double(param, shape + 3 * i, Si);
  sigma_double(param, shape + 3 * j, Sj);
  const double ri = sqrt(dsub(dmul(Si[0], Si[2]), dmul(Si[1], Si[1])));
  const double rj = sqrt(dsub(dmul(Sj[0], Sj[2]), dmul(Sj[1], Sj[1])));
  const float* ci = rgb + 3 * i;
  const float* cj = rgb + 3 * j;
  double wi = dmul(ri, dadd(dadd(fabs(double(ci[0])), fabs(double(ci[1]))), fabs(double(ci[2]))));
  double wj = dmul(rj, dadd(dadd(fabs(double(cj[0])), fabs(double(cj[1]))), fabs(double(cj[2]))));
  if (dadd(wi, wj) == 0.0) wi = wj = 1.0;
  const double W = dadd(wi, wj);
  const double xi0 = xy[2 * i], xi1 = xy[2 * i + 1], xj0 = xy[2 * j], xj1 = xy[2 * j + 1];
  const double m0 = ddiv(dadd(dmul(wi, xi0), dmul(wj, xj0)), W);
  const double m1 = ddiv(dadd(dmul(wi, xi1), dmul(wj, xj1)), W);
  const double di0 = dsub(xi0, m0), di1 = dsub(xi1, m1), dj0 = dsub(xj0, m0), dj1 = dsub(xj1, m1);
  const double sxx = ddiv(dadd(dmul(wi, dadd(Si[0], dmul(di0, di0))), dmul(wj, dadd(Sj[0], dmul(dj0, dj0)))), W);
  const double sxy = ddiv(dadd(dmul(wi, dadd(Si[1], dmul(di0, di1))), dmul(wj, dadd(Sj[1], dmul(dj0, dj1)))), W);
  const double syy = ddiv(dadd(dmul(wi, dadd(Si[2], dmul(di1, di1))), dmul(wj, dadd(Sj[2], dmul(dj1, dj1)))), W);
  const double r = sqrt(dsub(dmul(sxx, syy), dmul(sxy, sxy)));
  out_xy[2 * o] = __double2float_rn(m0);
  out_xy[2 * o + 1] = __double2float_rn(m1);
  for (int d = 0; d < 3; ++d)
    out_rgb[3 * o + d] = __double2float_rn(ddiv(dadd(dmul(double(ci[d]), ri), dmul(double(cj[d]), rj)), r));
  if (param == GS2D_PARAM_SCALE_ROT) {
    // theta = atan2(2 Sxy, Sxx - Syy) / 2; eigenvalue along theta = the
    // quadratic form of (cos, sin), the other = the trace minus it
    const double th = dmul(0.5, atan2(dmul(2.0, sxy), dsub(sxx, syy)));
    double s, c;
    sincos(th, &s, &c);
    const double l1 = dadd(dadd(dmul(dmul(c, c), sxx), dmul(dmul(dmul(2.0, c), s), sxy)), dmul(dmul(s, s), syy));
    const double l2 = dsub(dadd(sxx, syy), l1);
    out_shape[3 * o] = __double2float_rn(sqrt(l1));
    out_shape[3 * o + 1] = __double2float_rn(sqrt(l2 > 0.0 ? l2 : 0.0));
    out_shape[3 * o + 2] = __double2float_rn(th);
  } else {
    const double a = sqrt(sxx);
    const double b = ddiv(sxy, a);
    out_shape[3 * o] = __double2float_rn(a);
    out_shape[3 * o + 1] = __double2float_rn(b);
    out_shape[3 * o + 2] = __double2float_rn(sqrt(dsub(syy, dmul(b, b))));
  }
}

}  // namespace

size_t merge_workspace_size(long long n) { return merge_layout(n).total; }

cudaError_t launch_merge(const gs2d_config& c, int n, const float* xy, const float* shape,
                         const float* rgb, const gs2d_record* rec, const int* count,
                         const int* ranges, const int* sorted_gid, int max_merges, float* out_xy,
                         float* out_shape, float* out_rgb, unsigned char* ws, int* merges_dev,
                         cudaStream_t s) {
  const MergeLayout L = merge_layout(n);
  MergeHeader* hdr = reinterpret_cast<MergeHeader*>(ws);
  GS2D_TRY(cudaMemsetAsync(ws, 0, L.mrec, s));  // header and key histogram
  if (n == 0) return cudaGetLastError();
  GS2D_TRY(cudaMemsetAsync(ws + L.drop, 0, 4 * size_t(n), s));
  unsigned int* hist = reinterpret_cast<unsigned int*>(ws + L.hist);
  float4* mrec = reinterpret_cast<float4*>(ws + L.mrec);
  float* msyy = reinterpret_cast<float*>(ws + L.msyy);
  int* mtile = reinterpret_cast<int*>(ws + L.mtile);
  float* cost = reinterpret_cast<float*>(ws + L.cost);
  int* nn = reinterpret_cast<int*>(ws + L.nn);
  unsigned int* key = reinterpret_cast<unsigned int*>(ws + L.key);
  int* take = reinterpret_cast<int*>(ws + L.take);
  int* drop = reinterpret_cast<int*>(ws + L.drop);
  int* block_a = reinterpret_cast<int*>(ws + L.block_a);
  int* block_b = reinterpret_cast<int*>(ws + L.block_b);
  const int blocks = (n + kMergeThreads - 1) / kMergeThreads;
  const dim3 g(blocks), b(kMergeThreads);
  GS2D_TRY(launch(k_merge_prep, g, b, 0, s, c, n, tiles_x(c), xy, shape,
                  reinterpret_cast<const float4*>(rec), count, mrec, msyy, mtile, nn, cost));
  GS2D_TRY(launch(k_merge_nn, dim3(num_tiles(c)), b, 0, s, n, reinterpret_cast<const int2*>(ranges),
                  sorted_gid, static_cast<const float4*>(mrec), static_cast<const float*>(msyy),
                  static_cast<const int*>(mtile), nn, cost));
  GS2D_TRY(launch(k_merge_pairs, g, b, 0, s, n, static_cast<const int*>(nn),
                  static_cast<const float*>(cost), key, hist));
  GS2D_TRY(launch(k_merge_threshold, dim3(1), dim3(1024), 0, s, max_merges,
                  static_cast<const unsigned int*>(hist), hdr));
  GS2D_TRY(launch(k_merge_count<0>, g, b, 0, s, n, hdr, static_cast<const unsigned int*>(key),
                  static_cast<const int*>(drop), block_a));
  GS2D_TRY(launch(k_merge_take, g, b, 0, s, n, static_cast<const MergeHeader*>(hdr),
                  static_cast<const unsigned int*>(key), static_cast<const int*>(nn),
                  static_cast<const int*>(block_a), take, drop));
  GS2D_TRY(launch(k_merge_count<1>, g, b, 0, s, n, hdr, static_cast<const unsigned int*>(key),
                  static_cast<const int*>(drop), block_b));
  GS2D_TRY(launch(k_merge_write, g, b, 0, s, n, int(c.param), xy, shape, rgb,
                  static_cast<const int*>(nn), static_cast<const int*>(take),
                  static_cast<const int*>(drop), static_cast<const int*>(block_b), out_xy, out_shape,
                  out_rgb));
  if (merges_dev)
    GS2D_TRY(cudaMemcpyAsync(merges_dev, &hdr->merges, sizeof(int), cudaMemcpyDeviceToDevice, s));
  return cudaGetLastError();
}

GS2D_CHECK_WORD_READER(merge)

}  // namespace gs2d
