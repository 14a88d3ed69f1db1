// Tile binning and sort, as reduce-then-scan steps that never wait on
// another block.  With few tiles the counting sort further down is taken
// (composite: then a per-tile depth sort); otherwise:
//
//   k_count_scan   sum of the tile counts of every 256-Gaussian block (eight
//                  such blocks per thread block); the last thread block to
//                  finish scans the sums into block offsets and writes the
//                  pair count P (and the flags).
//   k_emit         per block: Gaussian pair offsets, then the (key, Gaussian
//                  index) pairs of its Gaussians in index order -- key = tile
//                  id (sum) or (tile id << 32 | depth key) (composite) -- plus
//                  the digit counts of every 2048-key partition for the first
//                  pass.
//   per radix pass (8-bit digits, least significant first):
//     k_radix_count    (passes after the first) digit counts of every
//                      partition of the pass's input;
//     k_digit_offsets  (more than 128 partitions) per digit: exclusive scan
//                      of its partition counts and the digit's total;
//     k_radix_scatter  per partition: each digit's output start (a block
//                      scan of the digit totals) plus the partition's prefix
//                      (both summed by the block itself when partitions are
//                      few), stable
//                      ranks within the partition (lane groups by digit from
//                      ballots + per-warp counts), the keys reordered by digit
//                      in shared memory, and the scatter from there in runs
//                      of consecutive slots.
//   k_tile_bounds  [start, end) of every non-empty tile from the places where
//                  the tile id changes along the sorted keys (empty tiles keep
//                  the [0, 0) written by k_count_scan).
// Emission in index order plus stable passes gives ascending index within
// equal keys.
//
// Tile size 16 (fVDB radiance_fields API, GaussianSplatReconstructionConfig
// tile_size); per-tile depth order for compositing (DrawingWithGaussians
// README, Overview: gsplat-style projection/rasterization).
#include <type_traits>

#include "project_body.cuh"

namespace gs2d {

namespace {

constexpr int kPartKeys = kRadixThreads * 8;  // keys per radix partition
constexpr int kSpan = 4;                     // partitions one emit block counts in shared memory
constexpr unsigned int kBadFlags = GS2D_FLAG_CAPACITY | GS2D_FLAG_OVERFLOW | GS2D_FLAG_TIMEOUT;

__device__ __forceinline__ unsigned int lanemask_lt() {
  unsigned int m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Exclusive scan over the 256 threads of a block; returns the thread's
// exclusive prefix and writes the block total to *total.
template <typename T>
__device__ __forceinline__ T block_exclusive_scan_256(T x, T* total) {
  __shared__ T warp_tot[8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  T before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const T v = warp_tot[w];
    if (w < warp) before += v;
    all += v;
  }
  __syncthreads();
  *total = all;
  return before + incl - x;
}

// The pair count, unless the flags say the lists are not usable.
__device__ __forceinline__ long long usable_pairs(const Header* hdr, long long cap) {
  const unsigned int f = *reinterpret_cast<const volatile unsigned int*>(&hdr->flags);
  const long long P = hdr->pairs;
  return (f & kBadFlags) ? 0 : (P < cap ? P : cap);
}

template <bool kComposite>
using KeyOf = typename std::conditional<kComposite, unsigned long long, unsigned int>::type;

// Called by every thread of every block once the block has written its
// sub-block totals (each writer fenced its write): the last block to arrive
// scans all nsub totals into exclusive offsets and writes P, the flags and the
// offset of the final keys.
__device__ __forceinline__ void finish_block_totals(Header* hdr, long long* __restrict__ block_off,
                                                    long long nsub, long long cap,
                                                    unsigned long long keys_final) {
  const int tid = threadIdx.x;
  __shared__ bool last;
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    last = atomicAdd(&hdr->blocks_done, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!last) return;
  // The last block: exclusive scan of all block sums.  Thread t takes the
  // contiguous run [t per, (t + 1) per), loads it 8 at a time, and one block
  // scan of the runs' sums gives every run's start (a scan per chunk of 256
  // sums, each behind its own loads and barriers, made this block the
  // kernel's tail at 2M Gaussians).
  __threadfence();
  const volatile long long* bo = block_off;
  const long long B = nsub;
  const long long per = (B + kScanThreads - 1) / kScanThreads;
  const long long a = tid * per, b = a + per < B ? a + per : B;
  long long sum = 0;
  for (long long p0 = a; p0 < b; p0 += 8) {
    long long v8[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v8[j] = (p0 + j < b) ? bo[p0 + j] : 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) sum += v8[j];
  }
  long long carry;
  long long run = block_exclusive_scan_256<long long>(sum, &carry);
  for (long long p0 = a; p0 < b; p0 += 8) {
    long long v8[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v8[j] = (p0 + j < b) ? bo[p0 + j] : 0;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (p0 + j < b) {
        block_off[p0 + j] = run;
        run += v8[j];
      }
  }
  if (tid == 0) {
    hdr->pairs = carry;
    hdr->keys_final = keys_final;
    unsigned int f = 0;
    if (carry > cap) f |= GS2D_FLAG_CAPACITY;
    if (carry >= (1ll << 30)) f |= GS2D_FLAG_OVERFLOW;
    if (f) atomicOr(&hdr->flags, f);
  }
}

// Sums of the tile counts of every 256-Gaussian sub-block (kCountSubs of
// them per block, so that only one block in kCountSubs takes a turn at the
// arrival counter: with one block per sub-block, the 7,813 atomics of 2M
// Gaussians on that one address set the kernel's length); the last block
// scans them.  Also clears the first pass's count table (k_emit adds to it;
// the later passes' tables are written whole by k_radix_count) and the tile
// ranges for the kernels that follow.
constexpr int kCountSubs = 8;

__global__ void __launch_bounds__(kScanThreads)
k_count_scan(int n, long long cap, const int* __restrict__ count, Header* hdr,
             long long* __restrict__ block_off, unsigned int* __restrict__ zero_a,
             long long zero_a_words, unsigned int* __restrict__ zero_b, long long zero_b_words,
             unsigned long long keys_final) {
  pdl_enter();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long gstride = (long long)gridDim.x * blockDim.x;
  for (long long k = (long long)blockIdx.x * blockDim.x + tid; k < zero_a_words; k += gstride)
    zero_a[k] = 0u;
  for (long long k = (long long)blockIdx.x * blockDim.x + tid; k < zero_b_words; k += gstride)
    zero_b[k] = 0u;
  __shared__ long long s_sum[kCountSubs][kScanThreads / 32];
  const long long nsub = (n + kScanItems - 1) / kScanItems;
  const long long sub0 = (long long)blockIdx.x * kCountSubs;
  int c[kCountSubs];
#pragma unroll
  for (int j = 0; j < kCountSubs; ++j) {
    const long long g = (sub0 + j) * kScanItems + tid;
    c[j] = g < n ? count[g] : 0;
  }
#pragma unroll
  for (int j = 0; j < kCountSubs; ++j) {
    long long v = c[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) s_sum[j][warp] = v;
  }
  __syncthreads();
  if (tid < kCountSubs && sub0 + tid < nsub) {
    long long t = 0;
#pragma unroll
    for (int w = 0; w < kScanThreads / 32; ++w) t += s_sum[tid][w];
    block_off[sub0 + tid] = t;
    __threadfence();
  }
  finish_block_totals(hdr, block_off, nsub, cap, keys_final);
}

// ---------------------------------------------------------------------------
// With at most kCountSortMaxTiles tiles: a counting sort by tile in three
// kernels, writing the final lists directly.  No block waits for another or
// finishes for the others: what every block needs is recomputed by each.
//   k_tile_hist     per 256-Gaussian block b: H[t][b] = how many of the
//                   block's Gaussians cover tile t, and the block's pair
//                   total.
//   k_tile_scan     per tile t (one warp): exclusive scan of H[t][.] over the
//                   blocks, in place, and the row total R[t].
//   k_tile_scatter  per block: the block's pair offset (sum of the totals of
//                   the blocks before it) and the tile starts (exclusive scan
//                   of R); the pair (Gaussian g, tile t) goes to start(t) +
//                   H[t][b] + the number of the block's Gaussians before g
//                   that cover t, read off a per-tile 256-bit mask of the
//                   block's Gaussians.  One extra block, the last, emits no
//                   pair: it writes the tile ranges (empty tiles [0, 0), as
//                   the radix path leaves them), the tiles' launch order, P
//                   and the flags, beside the others instead of lengthening
//                   block 0 (768x512 step 64.1 -> 63.6 us).
// Within a tile the list comes out in ascending index, as the radix passes
// give it; the sorted tile ids are written too (the backward reads them).

// kProject: the block first projects its Gaussians (project_one), so the
// projection and the histogram are one launch.
template <bool kProject>
__global__ void __launch_bounds__(kScanThreads)
k_tile_hist(int n, int T, int tiles_x, gs2d_config c, ProjectIn in, float4* __restrict__ rec,
            int4* __restrict__ rect, int* __restrict__ count, long long* __restrict__ block_tot,
            unsigned int* __restrict__ H) {
  pdl_enter();
  __shared__ unsigned int s_h[kCountSortMaxTiles];
  const int tid = threadIdx.x;
  for (int t = tid; t < T; t += blockDim.x) s_h[t] = 0u;
  const long long g = (long long)blockIdx.x * kScanItems + tid;
  int cnt = 0;
  int4 r = make_int4(0, 0, -1, -1);
  if (g < n) {
    if constexpr (kProject) {
      r = project_one(c, int(g), in.xy, in.shape, in.rgb, in.depth, in.opacity, rec, rect, count);
      cnt = r.z >= r.x ? (r.z - r.x + 1) * (r.w - r.y + 1) : 0;
    } else {
      cnt = count[g];
      r = rect[g];
    }
  }
  long long total;
  block_exclusive_scan_256<long long>(cnt, &total);  // its barriers order the clears
  if (cnt > 0)
    for (int y = r.y; y <= r.w; ++y)
      for (int x = r.x; x <= r.z; ++x)
        if (check_ok(y * tiles_x + x < T, kCheckTile)) atomicAdd(&s_h[y * tiles_x + x], 1u);
  __syncthreads();
  const size_t B = gridDim.x;
  for (int t = tid; t < T; t += blockDim.x) H[size_t(t) * B + blockIdx.x] = s_h[t];
  if (tid == 0) block_tot[blockIdx.x] = total;
}

__global__ void __launch_bounds__(256)
k_tile_scan(int T, int B, unsigned int* __restrict__ H, unsigned int* __restrict__ R) {
  pdl_enter();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t = blockIdx.x * 8 + warp;
  if (t < T) {
    unsigned int* row = H + size_t(t) * B;
    unsigned int carry = 0;
    for (int b0 = 0; b0 < B; b0 += 256) {  // lane: 8 consecutive entries
      unsigned int v[8], ex[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int b = b0 + lane * 8 + j;
        v[j] = b < B ? row[b] : 0u;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        ex[j] = sum;
        sum += v[j];
      }
      unsigned int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned int before = carry + incl - sum;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int b = b0 + lane * 8 + j;
        if (b < B) row[b] = before + ex[j];
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) R[t] = carry;
  }
}

__global__ void __launch_bounds__(kScanThreads)
k_tile_scatter(int n, int T, int tiles_x, long long cap, Header* __restrict__ hdr,
               const int4* __restrict__ rect, const int* __restrict__ count,
               const long long* __restrict__ block_tot, const unsigned int* __restrict__ H,
               const unsigned int* __restrict__ R, int2* __restrict__ ranges, int4* __restrict__ order,
               int* __restrict__ offsets, int* __restrict__ sorted_gid,
               unsigned int* __restrict__ keys_out, unsigned long long keys_final) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned int s_mask[];  // [T][8]: bit i = local Gaussian i covers t
  __shared__ int s_excl[kScanItems + 1];  // block-local pair offsets (P < 2^31 here)
  __shared__ int4 s_rect[kScanItems];
  __shared__ float s_rcpw[kScanItems];   // 1 / rectangle width
  __shared__ unsigned int s_base[kCountSortMaxTiles];  // where the block's part of list t starts
  constexpr int kTilesPer = kCountSortMaxTiles / kScanThreads;  // tiles per thread, consecutive
  const int tid = threadIdx.x;
  const size_t B = gridDim.x - 1;  // the last block only writes the ranges, the order and the header
  const long long g0 = (long long)blockIdx.x * kScanItems;
  const long long g = g0 + tid;
  const int cnt = g < n ? count[g] : 0;
  const int4 r = g < n ? rect[g] : make_int4(0, 0, -1, -1);
  // this thread's tiles: row totals and the block's offsets within them
  unsigned int v[kTilesPer], hb[kTilesPer];
#pragma unroll
  for (int j = 0; j < kTilesPer; ++j) {
    const int u = tid * kTilesPer + j;
    v[j] = u < T ? R[u] : 0u;
    hb[j] = (u < T && blockIdx.x < B) ? H[size_t(u) * B + blockIdx.x] : 0u;
  }
  long long before_blocks = 0;  // pairs of the blocks before this one (loads issued 4 at a time)
  for (int k0 = tid; k0 < int(blockIdx.x); k0 += 4 * blockDim.x) {
    long long v4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = k0 + j * int(blockDim.x);
      v4[j] = k < int(blockIdx.x) ? block_tot[k] : 0;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) before_blocks += v4[j];
  }
  {  // the per-tile masks cleared with 16-byte stores, after the loads above
     // are issued (768x512 step 60.5 -> 60.0 us, render path 39.0 -> 37.6 us)
    uint4* m4 = reinterpret_cast<uint4*>(s_mask);
    for (int k = tid; k < T * 2; k += blockDim.x) m4[k] = make_uint4(0u, 0u, 0u, 0u);
  }
  s_rect[tid] = r;
  s_rcpw[tid] = 1.0f / float(max(r.z - r.x + 1, 1));
  long long total;
  const long long excl = block_exclusive_scan_256<long long>(cnt, &total);  // orders the clears
  s_excl[tid] = int(excl);
  if (tid == 0) s_excl[kScanItems] = int(total);
  long long boff;
  block_exclusive_scan_256<long long>(before_blocks, &boff);
  // tile starts: exclusive scan of the row totals (P fits 32 bits: n <= 2^20, T <= 2^11)
  unsigned int ex[kTilesPer], sum = 0;
#pragma unroll
  for (int j = 0; j < kTilesPer; ++j) {
    ex[j] = sum;
    sum += v[j];
  }
  unsigned int P32;
  const unsigned int before = block_exclusive_scan_256<unsigned int>(sum, &P32);
  const long long P = P32;
  unsigned int flags = 0;
  if (P > cap) flags |= GS2D_FLAG_CAPACITY;
  if (P >= (1ll << 30)) flags |= GS2D_FLAG_OVERFLOW;
  const bool ok = flags == 0;
#pragma unroll
  for (int j = 0; j < kTilesPer; ++j) {
    const int u = tid * kTilesPer + j;
    if (u < T) s_base[u] = before + ex[j] + hb[j];
  }
  if (g < n) {
    const long long o = boff + excl;
    offsets[g] = o < (1ll << 31) ? int(o) : 0x7fffffff;
  }
  if (cnt > 0) {
    const unsigned int bit = 1u << (tid & 31);
    for (int y = r.y; y <= r.w; ++y)
      for (int x = r.x; x <= r.z; ++x)
        if (check_ok(y * tiles_x + x < T, kCheckTile))
          atomicOr(&s_mask[(y * tiles_x + x) * 8 + (tid >> 5)], bit);
  }
  if (blockIdx.x == B) {
#pragma unroll
    for (int j = 0; j < kTilesPer; ++j) {
      const int u = tid * kTilesPer + j;
      if (u < T) {
        const unsigned int start = before + ex[j];
        ranges[u] = (ok && v[j]) ? make_int2(int(start), int(start + v[j])) : make_int2(0, 0);
      }
    }
    if (tid == 0) {
      hdr->pairs = P;
      hdr->flags = flags;
      hdr->blocks_done = 0u;
      hdr->blocks_done2 = 0u;
      hdr->keys_final = keys_final;
    }
    // Launch order for the raster: tiles bucketed by floor(log2(list
    // length)), longest first, so that the heaviest tiles start early
    // instead of finishing last.  The order within a bucket does not matter
    // (it only affects scheduling; every tile's result is the same).
    __shared__ unsigned int s_cnt[33], s_pos[33];
    if (tid < 33) s_cnt[tid] = 0u;
    __syncthreads();
    int bk[kTilesPer];
#pragma unroll
    for (int j = 0; j < kTilesPer; ++j) {
      const int u = tid * kTilesPer + j;
      bk[j] = (u < T && ok && v[j]) ? 32 - __clz(v[j]) : 0;
      if (u < T) atomicAdd(&s_cnt[bk[j]], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      unsigned int run = 0;
      for (int k = 32; k >= 0; --k) {
        s_pos[k] = run;
        run += s_cnt[k];
      }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kTilesPer; ++j) {
      const int u = tid * kTilesPer + j;
      if (u < T) {
        const int start = int(before + ex[j]);
        const bool used = ok && v[j];
        order[atomicAdd(&s_pos[bk[j]], 1u)] =
            make_int4(u, used ? start : 0, used ? start + int(v[j]) : 0, 0);
      }
    }
  }
  __syncthreads();
  if (!ok || P == 0) return;  // P > capacity, overflow, or no pairs
  const int total32 = int(total);
  for (int e = tid; e < total32; e += blockDim.x) {
    int lo = 0, hi = kScanItems - 1;  // the local Gaussian of pair e (as in k_emit)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_excl[mid] <= e) lo = mid; else hi = mid - 1;
    }
    const int k = e - s_excl[lo];
    const int4 q = s_rect[lo];
    const int rw = q.z - q.x + 1;
    int qy = int(float(k) * s_rcpw[lo]);  // k / rw as in k_emit
    int qx = k - qy * rw;
    if (qx >= rw) { ++qy; qx -= rw; }
    if (qx < 0) { --qy; qx += rw; }
    const int t = (q.y + qy) * tiles_x + q.x + qx;
    if (!check_ok(t >= 0 && t < T, kCheckTile)) continue;
    const unsigned int* m = s_mask + t * 8;
    unsigned int rank = __popc(m[lo >> 5] & ((1u << (lo & 31)) - 1u));
    for (int j = 0; j < (lo >> 5); ++j) rank += __popc(m[j]);
    const long long dst = (long long)s_base[t] + rank;
    if (!check_ok(dst >= 0 && dst < cap, kCheckPairSlot)) continue;
    sorted_gid[dst] = int(g0 + lo);
    keys_out[dst] = unsigned(t);
  }
}

template <bool kComposite>
__global__ void __launch_bounds__(kScanThreads)
k_emit(int n, int tiles_x, int passes, long long cap, long long partitions4,
       const int4* __restrict__ rect, const int* __restrict__ count,
       const float4* __restrict__ rec, const long long* __restrict__ block_off,
       unsigned int* __restrict__ table0, int* __restrict__ offsets,
       KeyOf<kComposite>* __restrict__ keys, unsigned int* __restrict__ vals) {
  pdl_enter();
  using Key = KeyOf<kComposite>;
  __shared__ int s_excl[kScanItems + 1];  // block-local pair offsets (below 2^30)
  __shared__ int4 s_rect[kScanItems];
  __shared__ float s_rcpw[kScanItems];   // 1 / rectangle width
  __shared__ unsigned int s_dkey[kComposite ? kScanItems : 1];
  __shared__ unsigned int s_part[kSpan][kMaxRadix];
  const int tid = threadIdx.x;
  const long long g = (long long)blockIdx.x * kScanItems + tid;
  for (int k = tid; k < kSpan * kMaxRadix; k += blockDim.x) (&s_part[0][0])[k] = 0u;
  const int cnt = (g < n) ? count[g] : 0;
  const int4 myrect = (g < n) ? rect[g] : make_int4(0, 0, -1, -1);
  s_rect[tid] = myrect;
  s_rcpw[tid] = 1.0f / float(max(myrect.z - myrect.x + 1, 1));
  if constexpr (kComposite) s_dkey[tid] = (g < n) ? depth_key(rec[3 * g + 2].w) : 0u;
  long long total;
  const long long excl = block_exclusive_scan_256<long long>(cnt, &total);
  s_excl[tid] = int(excl);
  if (tid == 0) s_excl[kScanItems] = int(total);
  const long long base = block_off[blockIdx.x];
  if (g < n) {
    const long long o = base + excl;
    offsets[g] = o < (1ll << 31) ? int(o) : 0x7fffffff;
  }
  __syncthreads();
  const long long part0 = base / kPartKeys;
  // Pair e of this block belongs to the last local Gaussian whose exclusive
  // offset is <= e (that one has a non-zero count).
  const int total32 = int(total);
  for (int e = tid; e < total32; e += blockDim.x) {
    int lo = 0, hi = kScanItems - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_excl[mid] <= e) lo = mid; else hi = mid - 1;
    }
    const int k = e - s_excl[lo];
    const int4 r = s_rect[lo];
    const int rw = r.z - r.x + 1;
    // k / rw by the rounded reciprocal (k < 2^24, exact in FP32) and one
    // correction step, in place of an integer division (4096x4096 / 2M:
    // emission with 64-bit offsets and the division 60.2 us, now 55.6 us)
    int qy = int(float(k) * s_rcpw[lo]);
    int qx = k - qy * rw;
    if (qx >= rw) { ++qy; qx -= rw; }
    if (qx < 0) { --qy; qx += rw; }
    const int ty = r.y + qy, tx = r.x + qx;
    const unsigned int tile = unsigned(ty) * unsigned(tiles_x) + unsigned(tx);
    Key key;
    if constexpr (kComposite)
      key = (Key(tile) << 32) | Key(s_dkey[lo]);
    else
      key = Key(tile);
    const long long slot = base + e;
    if (slot < cap) {
      keys[slot] = key;
      vals[slot] = unsigned(g - tid + lo);
      if (passes > 0) {
        const unsigned int d = unsigned(key) & 255u;
        const long long part = slot / kPartKeys;
        if (part - part0 < kSpan)
          atomicAdd(&s_part[part - part0][d], 1u);
        else
          atomicAdd(&table0[(long long)d * partitions4 + part], 1u);
      }
    }
  }
  __syncthreads();
  if (passes > 0) {
    for (int k = tid; k < kSpan * kMaxRadix; k += blockDim.x) {
      const unsigned int v = (&s_part[0][0])[k];
      if (v) atomicAdd(&table0[(long long)(k % kMaxRadix) * partitions4 + part0 + k / kMaxRadix], v);
    }
  }
}

// Per digit (one block each): every used partition's offset for the digit
// within the digit's run (the counts of the digit in the partitions before
// it), over the counts it replaces, and the digit's total, to totals[d]
// (each scatter block scans the totals into the digits' starts: as a
// last-block tail here the scan cost as much as it saved).
__global__ void __launch_bounds__(256)
k_digit_offsets(int pass, long long cap, long long partitions4, const Header* __restrict__ hdr,
                unsigned int* __restrict__ totals, unsigned int* __restrict__ table) {
  pdl_enter();
  const long long n = usable_pairs(hdr, cap);
  if (n == 0) return;
  const long long partitions = (n + kPartKeys - 1) / kPartKeys;  // the used ones
  const int d = blockIdx.x, tid = threadIdx.x;
  unsigned int* row = table + (long long)d * partitions4;
  const long long per = (partitions + blockDim.x - 1) / blockDim.x;
  const long long a = (long long)tid * per;
  const long long b = a + per < partitions ? a + per : partitions;
  // the thread's run of counts, loaded 8 at a time (one round trip per 8)
  unsigned int sum = 0;
  for (long long p0 = a; p0 < b; p0 += 8) {
    unsigned int c8[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) c8[j] = (p0 + j < b) ? row[p0 + j] : 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) sum += c8[j];
  }
  unsigned int tot;
  unsigned int run = block_exclusive_scan_256<unsigned int>(sum, &tot);
  if (tid == 0) totals[d] = tot;
  for (long long p0 = a; p0 < b; p0 += 8) {
    unsigned int c8[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) c8[j] = (p0 + j < b) ? row[p0 + j] : 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (p0 + j < b) {
        row[p0 + j] = run;
        run += c8[j];
      }
  }
}

// One stable LSD pass over the digit at bits [8 pass, 8 pass + 8).  A
// digit's output run starts after the runs of the digits below it (a block
// scan of the digit totals), and the partition's part of it after the
// digit's keys in the partitions before it.  With own_offsets the table
// still holds counts and every block sums them itself (the totals and its
// own prefix): cheaper than a separate k_digit_offsets launch when
// partitions are few.  Otherwise k_digit_offsets left the prefix in the table
// and the totals in `totals`.
template <typename Key, int kPerThread>
__global__ void __launch_bounds__(kRadixThreads)
k_radix_scatter(int pass, long long cap, long long partitions4, bool own_offsets,
                const unsigned int* __restrict__ totals,
                const Header* __restrict__ hdr, const unsigned int* __restrict__ table,
                const Key* __restrict__ keys_in,
                const unsigned int* __restrict__ vals_in, Key* __restrict__ keys_out,
                unsigned int* __restrict__ vals_out) {
  pdl_enter();
  constexpr int kItems = kRadixThreads * kPerThread;
  __shared__ unsigned short s_whist[8][kMaxRadix];  // per-warp counts, then exclusive offsets
  __shared__ unsigned int s_base[kMaxRadix];
  __shared__ Key s_k[kItems];            // the partition's keys in output order
  __shared__ unsigned int s_v[kItems];
  __shared__ unsigned int s_dstart[kMaxRadix];  // where each digit's run starts in s_k
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long n = usable_pairs(hdr, cap);
  const long long part = blockIdx.x;
  const long long base = part * kItems;
  if (base >= n) return;
  // The partition's keys and values are loaded first, so that their round
  // trip overlaps the digit-offset loads and scan below (4096x4096 / 2M:
  // both passes 118.4 -> 95.9 us); the digits are formed after the scan.
  Key k[kPerThread];
  unsigned int v[kPerThread], d[kPerThread], rank[kPerThread];
  const long long wbase = base + (long long)warp * (32 * kPerThread);
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const long long idx = wbase + j * 32 + lane;
    const bool ok = idx < n;
    k[j] = ok ? keys_in[idx] : Key(0);
    v[j] = ok ? vals_in[idx] : 0u;
  }
  for (int q = tid; q < 8 * kMaxRadix; q += blockDim.x) (&s_whist[0][0])[q] = 0;
  {
    unsigned int total = 0u, prefix = 0u;  // digit tid: keys in all partitions, in those before this one
    if (own_offsets) {
      const long long used = (n + kItems - 1) / kItems;
      const uint4* row4 = reinterpret_cast<const uint4*>(table + (long long)tid * partitions4);
      for (long long p = 0; p < used; p += 4) {  // the row is padded to a multiple of 4 (zeros)
        const uint4 c = row4[p >> 2];
        const unsigned int cc[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (p + j < part) prefix += cc[j];
          if (p + j < used) total += cc[j];
        }
      }
    } else {
      total = totals[tid];
      prefix = table[(long long)tid * partitions4 + part];
    }
    unsigned int all;
    s_base[tid] = block_exclusive_scan_256<unsigned int>(total, &all) + prefix;
  }
  __syncthreads();
  const int shift = 8 * pass;
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const long long idx = wbase + j * 32 + lane;
    d[j] = idx < n ? (unsigned(k[j] >> shift) & 255u) : 256u;
  }
  // Stable rank within the warp: item j of lane l precedes item j of lane
  // l+1 and every item j+1.  The lanes sharing a digit come from nine
  // ballots, one per bit of the digit (256 marks a key past the end): faster
  // than __match_any_sync over ~28 distinct digits per warp (4096x4096 / 2M:
  // both passes 169.4 -> 149.2 us).
  const unsigned int lt = lanemask_lt();
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    // the lanes holding the same digit (d <= 256): one ballot per bit of d
    unsigned int peers = 0xffffffffu;
#pragma unroll
    for (int b = 0; b < 9; ++b) {
      const bool bit = (d[j] >> b) & 1u;
      const unsigned int bal = __ballot_sync(0xffffffffu, bit);
      peers &= bit ? bal : ~bal;
    }
    const int leader = 31 - __clz(peers);
    const unsigned int prev = (d[j] < 256u) ? s_whist[warp][d[j]] : 0u;
    __syncwarp();
    if (lane == leader && d[j] < 256u) s_whist[warp][d[j]] = (unsigned short)(prev + __popc(peers));
    __syncwarp();
    rank[j] = prev + __popc(peers & lt);
  }
  __syncthreads();
  // The keys are first placed in shared memory in their output order (digit
  // by digit) and then written out from there, so that consecutive threads
  // store consecutive slots of a digit's run: one slot per lane scattered over
  // ~28 runs per store took 4096x4096 / 2M from 149.2 to 104.1 us for both
  // passes.  Same positions as a direct scatter, so the lists are unchanged.
  unsigned int dtot = 0;
  {  // per digit (one per thread): exclusive offsets across warps
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const unsigned int c = s_whist[w][tid];
      s_whist[w][tid] = (unsigned short)dtot;
      dtot += c;
    }
  }
  unsigned int all;
  s_dstart[tid] = block_exclusive_scan_256<unsigned int>(dtot, &all);
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    if (d[j] < 256u) {
      const unsigned int lpos = s_dstart[d[j]] + s_whist[warp][d[j]] + rank[j];
      if (check_ok(lpos < unsigned(kItems), kCheckPairSlot)) {
        s_k[lpos] = k[j];
        s_v[lpos] = v[j];
      }
    }
  }
  __syncthreads();
  const int cnt = int(n - base < kItems ? n - base : kItems);
  for (int i = tid; i < cnt; i += kRadixThreads) {
    const Key kk = s_k[i];
    const unsigned int dd = unsigned(kk >> shift) & 255u;
    const unsigned int dst = s_base[dd] + (unsigned(i) - s_dstart[dd]);
    if (check_ok((long long)dst < cap, kCheckPairSlot)) {
      keys_out[dst] = kk;
      vals_out[dst] = s_v[i];
    }
  }
}

// Digit counts of one pass for every partition of its input (the previous
// pass's output): table[d][partition].
template <typename Key>
__global__ void __launch_bounds__(kRadixThreads)
k_radix_count(int pass, long long cap, long long partitions4, const Header* __restrict__ hdr,
              const Key* __restrict__ keys, unsigned int* __restrict__ table) {
  pdl_enter();
  __shared__ unsigned int s_cnt[kMaxRadix];
  const long long n = usable_pairs(hdr, cap);
  const long long part = blockIdx.x;
  const long long base = part * kPartKeys;
  if (base >= n) return;
  const int tid = threadIdx.x;
  s_cnt[tid] = 0u;
  __syncthreads();
  const int shift = 8 * pass;
  // all of the thread's keys are loaded before the first count: with each
  // load followed by its atomic, the loads went out one after another
  constexpr int kPer = kPartKeys / kRadixThreads;
  unsigned int d[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const long long idx = base + j * kRadixThreads + tid;
    d[j] = idx < n ? unsigned(keys[idx] >> shift) & 255u : 256u;
  }
#pragma unroll
  for (int j = 0; j < kPer; ++j)
    if (d[j] < 256u) atomicAdd(&s_cnt[d[j]], 1u);
  __syncthreads();
  table[(long long)tid * partitions4 + part] = s_cnt[tid];
}

constexpr int kBoundsPer = 8;  // sorted keys per thread and step in k_tile_bounds

// Each thread takes kBoundsPer consecutive keys per step (16-byte loads),
// with the key before them and the key after them, and compares neighbours
// in registers (one key per thread with both neighbours reloaded took
// 23.4 us for 4.3M keys at 4096x4096).
template <typename Key>
__global__ void __launch_bounds__(256)
k_tile_bounds(long long cap, const Header* __restrict__ hdr, const Key* __restrict__ keys,
              int2* __restrict__ ranges, int tile_shift, int T) {
  pdl_enter();
  const long long n = usable_pairs(hdr, cap);
  int* rg = reinterpret_cast<int*>(ranges);
  const long long stride = (long long)gridDim.x * blockDim.x * kBoundsPer;
  for (long long b = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * kBoundsPer; b < n; b += stride) {
    unsigned int t[kBoundsPer + 2];  // t[0]: key b - 1, t[1 + j]: key b + j, t[kBoundsPer + 1]: the key after
    t[0] = b > 0 ? unsigned(keys[b - 1] >> tile_shift) : 0xFFFFFFFFu;
    t[kBoundsPer + 1] = b + kBoundsPer < n ? unsigned(keys[b + kBoundsPer] >> tile_shift) : 0xFFFFFFFFu;
    if (b + kBoundsPer <= n) {  // the run in 16-byte loads (b is a multiple of kBoundsPer)
      constexpr int kVec = 16 / int(sizeof(Key));
      const uint4* v = reinterpret_cast<const uint4*>(keys + b);
#pragma unroll
      for (int q = 0; q < kBoundsPer / kVec; ++q) {
        const uint4 u = v[q];
        const Key* k = reinterpret_cast<const Key*>(&u);
#pragma unroll
        for (int e = 0; e < kVec; ++e) t[1 + q * kVec + e] = unsigned(k[e] >> tile_shift);
      }
    } else {
#pragma unroll
      for (int j = 0; j < kBoundsPer; ++j)
        t[1 + j] = b + j < n ? unsigned(keys[b + j] >> tile_shift) : 0xFFFFFFFFu;
    }
#pragma unroll
    for (int j = 1; j <= kBoundsPer; ++j) {
      const long long i = b - 1 + j;
      if (i >= n || !check_ok(t[j] < unsigned(T), kCheckTile)) continue;
      if (t[j - 1] != t[j]) rg[2 * size_t(t[j])] = int(i);
      if (t[j + 1] != t[j]) rg[2 * size_t(t[j]) + 1] = int(i + 1);
    }
  }
}

constexpr int kSegSmem = 4096;  // tile lists up to this long are depth-sorted in shared memory

// Composite: each tile's list, in ascending index after the counting sort,
// into ascending (depth, index), one block per tile, longest lists first
// (the scatter's launch order: composite 768x512 step 151.6 -> 148.1 us).
// The keys (depth_key << 32 | index) are unique, so any sorting network
// gives the order of a stable sort by depth (ties by index).  (Sorting by
// rank -- each key's place is the number of smaller keys, no barriers --
// measured slower: 29.5 against 21.3 us up to 1024 entries, 149.6 against
// 148.1 us of step up to 256.)  The network is the bitonic merge sort with every
// comparator ascending -- the first step of each merge compares mirrored
// positions -- so positions past the list's end act as +inf and their
// comparators are skipped.  Lists longer than kSegSmem are sorted in place in
// a workspace buffer.
__global__ void __launch_bounds__(256)
k_tile_depth_sort(int n, int T, long long cap, const Header* __restrict__ hdr,
                  const int2* __restrict__ ranges, const float4* __restrict__ rec,
                  int* __restrict__ sorted_gid, unsigned long long* __restrict__ temp,
                  const int4* __restrict__ order) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned long long s_key[];  // kSegSmem
  const long long P = usable_pairs(hdr, cap);
  if (P == 0) return;
  int2 rg;
  const int tile = tile_of_slot(order, int(blockIdx.x), ranges, T, &rg);  // longest lists first
  if (!check_ok(tile >= 0 && tile < T, kCheckTile) || tile < 0) return;
  const int len = rg.y - rg.x;
  if (len <= 1) return;
  if (!check_ok(rg.x >= 0 && rg.y <= P, kCheckRange)) return;
  unsigned long long* key = len <= kSegSmem ? s_key : temp + rg.x;
  for (int k = threadIdx.x; k < len; k += blockDim.x) {
    int g = sorted_gid[rg.x + k];
    if (!check_ok(g >= 0 && g < n, kCheckGaussian)) g = 0;
    key[k] = ((unsigned long long)depth_key(rec[3 * size_t(g) + 2].w) << 32) | unsigned(g);
  }
  __syncthreads();
  int n2 = 2, l2 = 1;
  while (n2 < len) {
    n2 <<= 1;
    ++l2;
  }
  for (int lk = 1; lk <= l2; ++lk) {  // merge size k = 2^lk
    const int k = 1 << lk;
    for (int lj = lk - 1; lj >= 0; --lj) {  // comparator distance j = 2^lj
      const int j = 1 << lj;
      for (int i = threadIdx.x; i < (n2 >> 1); i += blockDim.x) {
        // comparator i: block i >> lj of width 2j, offset i & (j - 1)
        const int lo = ((i >> lj) << (lj + 1)) + (i & (j - 1));
        // first step of a merge: mirrored partner (merges two ascending runs)
        const int hi = (lj == lk - 1) ? (lo ^ (k - 1)) : (lo + j);
        if (hi < len) {
          const unsigned long long a = key[lo], b = key[hi];
          if (a > b) {
            key[lo] = b;
            key[hi] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int k = threadIdx.x; k < len; k += blockDim.x)
    sorted_gid[rg.x + k] = int(unsigned(key[k] & 0xFFFFFFFFull));
}

template <bool kComposite>
cudaError_t launch_binning_t(const gs2d_config& c, int n, const ProjectIn* proj, gs2d_record* rec,
                             int* rect, int* count, long long cap, int* tile_ranges, int* sorted_gid,
                             unsigned char* ws, cudaStream_t s) {
  using Key = KeyOf<kComposite>;
  const Layout L = layout_of(c, n, cap);
  // the kernels below use fixed 256-bucket digits and kPartKeys-key partitions
  if (L.digit_bits != 8 || (long long)kRadixThreads * L.radix_per_thread != kPartKeys)
    return cudaErrorInvalidConfiguration;
  const int T = num_tiles(c);
  Header* hdr = reinterpret_cast<Header*>(ws);
  unsigned int* hist = reinterpret_cast<unsigned int*>(ws + kOffHist);
  long long* block_off = reinterpret_cast<long long*>(ws + L.block_off);
  int* offsets = reinterpret_cast<int*>(ws + L.offsets);
  unsigned int* tables = reinterpret_cast<unsigned int*>(ws + L.tables);
  const long long table_words = (long long)kMaxRadix * L.partitions4;
  unsigned int* vals_a = (L.passes % 2 == 0) ? reinterpret_cast<unsigned int*>(sorted_gid)
                                             : reinterpret_cast<unsigned int*>(ws + L.vals_tmp);
  unsigned int* vals_b = (L.passes % 2 == 0) ? reinterpret_cast<unsigned int*>(ws + L.vals_tmp)
                                             : reinterpret_cast<unsigned int*>(sorted_gid);
  Key* ka = reinterpret_cast<Key*>(ws + L.keys_a);
  Key* kb = reinterpret_cast<Key*>(ws + L.keys_b);
  const size_t keys_final = (L.passes % 2 == 0) ? L.keys_a : L.keys_b;
  const int blocks = n > 0 ? (n + kScanItems - 1) / kScanItems : 1;
  {
    if (L.count_sort) {
      unsigned int* H = reinterpret_cast<unsigned int*>(ws + L.tile_hist);
      unsigned int* R = H + size_t(T) * size_t(blocks);
      const int2* rg = reinterpret_cast<const int2*>(tile_ranges);
      // every header field is written by the scatter: no clearing pass
      // with proj the projection runs inside the histogram kernel
      GS2D_TRY(launch(proj ? k_tile_hist<true> : k_tile_hist<false>, dim3(blocks), dim3(kScanThreads), 0,
                      s, n, T, tiles_x(c), c, proj ? *proj : ProjectIn{},
                      reinterpret_cast<float4*>(rec), reinterpret_cast<int4*>(rect), count, block_off,
                      H));
      GS2D_TRY(launch(k_tile_scan, dim3((T + 7) / 8), dim3(256), 0, s, T, blocks, H, R));
      const size_t smem = size_t(T) * 8 * sizeof(unsigned int);
      GS2D_TRY(cudaFuncSetAttribute(k_tile_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    int(size_t(kCountSortMaxTiles) * 8 * sizeof(unsigned int))));
      GS2D_TRY(launch(k_tile_scatter, dim3(blocks + 1), dim3(kScanThreads), smem, s, n, T, tiles_x(c), cap,
                      hdr, reinterpret_cast<const int4*>(rect), count,
                      static_cast<const long long*>(block_off), static_cast<const unsigned int*>(H),
                      static_cast<const unsigned int*>(R), reinterpret_cast<int2*>(tile_ranges),
                      reinterpret_cast<int4*>(ws + L.tile_order), offsets, sorted_gid,
                      reinterpret_cast<unsigned int*>(ws + L.keys_a), (unsigned long long)L.keys_a));
      if (kComposite) {
        const size_t dsmem = size_t(kSegSmem) * sizeof(unsigned long long);
        GS2D_TRY(cudaFuncSetAttribute(k_tile_depth_sort, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      int(dsmem)));
        GS2D_TRY(launch(k_tile_depth_sort, dim3(T), dim3(256), dsmem, s, n, T, cap,
                        static_cast<const Header*>(hdr), rg, reinterpret_cast<const float4*>(rec),
                        sorted_gid, reinterpret_cast<unsigned long long*>(ws + L.keys_b),
                        reinterpret_cast<const int4*>(ws + L.tile_order)));
      }
      return cudaGetLastError();
    }
  }
  if (proj)
    GS2D_TRY(launch_project(c, n, proj->xy, proj->shape, proj->rgb, proj->depth, proj->opacity, rec,
                            rect, count, s));
  GS2D_TRY(cudaMemsetAsync(ws, 0, kOffScan, s));  // header, loss partials and digit totals
  GS2D_TRY(launch(k_count_scan, dim3((blocks + kCountSubs - 1) / kCountSubs), dim3(kScanThreads), 0, s, n, cap, count, hdr, block_off, tables,
                                               L.passes > 0 ? table_words : 0,  // pass 0's counts (atomics)
                                               reinterpret_cast<unsigned int*>(tile_ranges), 2ll * T,
                                               (unsigned long long)keys_final));
  GS2D_TRY(launch(k_emit<kComposite>, dim3(blocks), dim3(kScanThreads), 0, s, n, tiles_x(c), L.passes, cap, L.partitions4, reinterpret_cast<const int4*>(rect), count,
      reinterpret_cast<const float4*>(rec), block_off, tables, offsets, ka, vals_a));
  // Up to 128 partitions each scatter block sums its own offsets (at most 128
  // counts per digit); beyond that one k_digit_offsets launch per pass does.
  const bool own = L.partitions <= 128;
  for (int p = 0; p < L.passes && L.partitions > 0; ++p) {
    const bool even = (p % 2) == 0;
    unsigned int* table = tables + p * table_words;
    if (p > 0)  // pass 0 counts come from k_emit
      GS2D_TRY(launch(k_radix_count<Key>, dim3(int(L.partitions)), dim3(kRadixThreads), 0, s, p, cap, L.partitions4, hdr,
                                                                    even ? ka : kb, table));
    unsigned int* totals = hist + p * kMaxRadix;  // this pass's digit totals
    if (!own)
      GS2D_TRY(launch(k_digit_offsets, dim3(kMaxRadix), dim3(256), 0, s, p, cap, L.partitions4, hdr, totals, table));
    GS2D_TRY(launch(k_radix_scatter<Key, 8>, dim3(int(L.partitions)), dim3(kRadixThreads), 0, s, p, cap, L.partitions4, own, totals, hdr, table, even ? ka : kb, even ? vals_a : vals_b,
        even ? kb : ka, even ? vals_b : vals_a));
  }
  if (cap > 0) {
    long long tb = (cap + 256 * kBoundsPer - 1) / (256 * kBoundsPer);
    if (tb > 148 * 16) tb = 148 * 16;
    GS2D_TRY(launch(k_tile_bounds<Key>, dim3(int(tb)), dim3(256), 0, s, cap, hdr, reinterpret_cast<const Key*>(ws + keys_final),
                                              reinterpret_cast<int2*>(tile_ranges),
                                              kComposite ? 32 : 0, T));
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_binning(const gs2d_config& c, int n, const gs2d_record* rec, const int* rect,
                           const int* count, long long cap, int* tile_ranges, int* sorted_gid,
                           unsigned char* ws, cudaStream_t s) {
  // without a projection the kernels only read rec, rect and count
  gs2d_record* r = const_cast<gs2d_record*>(rec);
  int* rc = const_cast<int*>(rect);
  int* ct = const_cast<int*>(count);
  if (c.mode == GS2D_MODE_COMPOSITE)
    return launch_binning_t<true>(c, n, nullptr, r, rc, ct, cap, tile_ranges, sorted_gid, ws, s);
  return launch_binning_t<false>(c, n, nullptr, r, rc, ct, cap, tile_ranges, sorted_gid, ws, s);
}

cudaError_t launch_project_binning(const gs2d_config& c, int n, const ProjectIn& in, gs2d_record* rec,
                                   int* rect, int* count, long long cap, int* tile_ranges,
                                   int* sorted_gid, unsigned char* ws, cudaStream_t s) {
  if (c.mode == GS2D_MODE_COMPOSITE)
    return launch_binning_t<true>(c, n, &in, rec, rect, count, cap, tile_ranges, sorted_gid, ws, s);
  return launch_binning_t<false>(c, n, &in, rec, rect, count, cap, tile_ranges, sorted_gid, ws, s);
}

}  // namespace gs2d

namespace gs2d {
GS2D_CHECK_WORD_READER(binning)
}  // namespace gs2d
