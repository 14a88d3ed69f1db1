// Tile binning and sort.
//
//   1. k_scan_emit: exclusive scan of the per-Gaussian tile counts (block
//      scan + decoupled look-back across blocks), then every block emits the
//      (key, Gaussian index) pairs of its Gaussians in index order: key =
//      tile id (sum) or (tile id << 32 | depth key) (composite).  It also
//      builds the digit histograms of every radix pass.
//   2. k_radix_pass (one launch per 8-bit digit): stable LSD radix sort,
//      one pass per launch, ranks by warp-level match + per-digit look-back
//      across partitions.  Emission in index order plus stable passes gives
//      ascending index within equal keys.
//   3. k_tile_ranges: [start, end) of every tile by binary search.
//
// Tile size 16 (fVDB radiance_fields API, GaussianSplatReconstructionConfig
// tile_size); per-tile depth order for compositing (DrawingWithGaussians
// README, Overview: gsplat-style projection/rasterization).
//
// Every cross-block wait polls a status word at most kSpinLimit times; a
// wait that runs out sets GS2D_FLAG_TIMEOUT in the header and carries on, so
// the kernels always terminate.  Forward progress: blocks take their
// partition index from an atomic ticket when they start, so every block
// waited on has already started and publishes its aggregate before it waits
// on anything itself.
#include <type_traits>

#include "gs2d_internal.cuh"

namespace gs2d {

namespace {

constexpr unsigned long long kScanAgg = 1ull << 62;
constexpr unsigned long long kScanInc = 2ull << 62;
constexpr unsigned long long kScanVal = (1ull << 62) - 1;
constexpr unsigned int kRadAgg = 1u << 30;
constexpr unsigned int kRadInc = 2u << 30;
constexpr unsigned int kRadVal = (1u << 30) - 1;

__device__ __forceinline__ unsigned long long ld_volatile(const unsigned long long* p) {
  return *reinterpret_cast<const volatile unsigned long long*>(p);
}
__device__ __forceinline__ unsigned int ld_volatile(const unsigned int* p) {
  return *reinterpret_cast<const volatile unsigned int*>(p);
}
__device__ __forceinline__ void st_volatile(unsigned long long* p, unsigned long long v) {
  *reinterpret_cast<volatile unsigned long long*>(p) = v;
}
__device__ __forceinline__ void st_volatile(unsigned int* p, unsigned int v) {
  *reinterpret_cast<volatile unsigned int*>(p) = v;
}

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

template <bool kComposite>
__global__ void __launch_bounds__(kScanThreads)
k_scan_emit(int n, int tiles_x, int passes, long long cap, const int4* __restrict__ rect,
            const int* __restrict__ count, const float4* __restrict__ rec, Header* hdr,
            unsigned long long* scan_status, unsigned int* __restrict__ hist,
            int* __restrict__ offsets,
            typename std::conditional<kComposite, unsigned long long, unsigned int>::type* __restrict__ keys,
            unsigned int* __restrict__ vals, unsigned int* __restrict__ zero_ptr,
            long long zero_words) {
  using Key = typename std::conditional<kComposite, unsigned long long, unsigned int>::type;
  __shared__ long long s_excl[kScanItems + 1];
  __shared__ int4 s_rect[kScanItems];
  __shared__ unsigned int s_dkey[kComposite ? kScanItems : 1];
  __shared__ unsigned int s_hist[kMaxPasses][256];
  __shared__ long long s_base;
  __shared__ unsigned int s_part;
  const int tid = threadIdx.x;

  // Clear the look-back words of the radix passes that follow.
  for (long long k = (long long)blockIdx.x * blockDim.x + tid; k < zero_words;
       k += (long long)gridDim.x * blockDim.x)
    zero_ptr[k] = 0u;

  if (tid == 0) s_part = atomicAdd(&hdr->scan_ticket, 1u);
  for (int k = tid; k < kMaxPasses * 256; k += blockDim.x) (&s_hist[0][0])[k] = 0u;
  __syncthreads();
  const long long part = s_part;
  const long long g0 = part * kScanItems;

  long long mine = 0;
  int cnt[kScanPerThread];
#pragma unroll
  for (int j = 0; j < kScanPerThread; ++j) {
    const long long g = g0 + tid * kScanPerThread + j;
    cnt[j] = (g < n) ? count[g] : 0;
    mine += cnt[j];
    s_rect[tid * kScanPerThread + j] = (g < n) ? rect[g] : make_int4(0, 0, -1, -1);
    if (kComposite) s_dkey[tid * kScanPerThread + j] = (g < n) ? depth_key(rec[3 * g + 2].w) : 0u;
  }
  long long total;
  long long excl = block_exclusive_scan_256<long long>(mine, &total);
#pragma unroll
  for (int j = 0; j < kScanPerThread; ++j) {
    s_excl[tid * kScanPerThread + j] = excl;
    excl += cnt[j];
  }
  if (tid == 0) {
    s_excl[kScanItems] = total;
    long long prefix = 0;
    if (part == 0) {
      st_volatile(&scan_status[0], kScanInc | (unsigned long long)total);
    } else {
      st_volatile(&scan_status[part], kScanAgg | (unsigned long long)total);
      for (long long j = part - 1; j >= 0; --j) {
        unsigned long long v = 0;
        unsigned int it = 0;
        while (((v = ld_volatile(&scan_status[j])) >> 62) == 0ull) {
          if (++it >= kSpinLimit) {
            atomicOr(&hdr->flags, (unsigned)GS2D_FLAG_TIMEOUT);
            break;
          }
          __nanosleep(32);
        }
        prefix += (long long)(v & kScanVal);
        if ((v >> 62) == 2ull || it >= kSpinLimit) break;
      }
      st_volatile(&scan_status[part], kScanInc | (unsigned long long)(prefix + total));
    }
    s_base = prefix;
    if (part == gridDim.x - 1) {
      const long long P = prefix + total;
      hdr->pairs = P;
      unsigned int f = 0;
      if (P > cap) f |= GS2D_FLAG_CAPACITY;
      if (P >= (1ll << 30)) f |= GS2D_FLAG_OVERFLOW;
      if (f) atomicOr(&hdr->flags, f);
    }
  }
  __syncthreads();
  const long long base = s_base;
#pragma unroll
  for (int j = 0; j < kScanPerThread; ++j) {
    const long long g = g0 + tid * kScanPerThread + j;
    if (g < n) {
      const long long o = base + s_excl[tid * kScanPerThread + j];
      offsets[g] = o < (1ll << 31) ? int(o) : 0x7fffffff;
    }
  }

  // Emission: pair e of this block belongs to the last local Gaussian whose
  // exclusive offset is <= e (that one has a non-zero count).
  for (long long e = tid; e < total; e += blockDim.x) {
    int lo = 0, hi = kScanItems - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_excl[mid] <= e) lo = mid; else hi = mid - 1;
    }
    const int k = int(e - s_excl[lo]);
    const int4 r = s_rect[lo];
    const int rw = r.z - r.x + 1;
    const int ty = r.y + k / rw, tx = r.x + k % rw;
    const unsigned int tile = unsigned(ty) * unsigned(tiles_x) + unsigned(tx);
    Key key;
    if constexpr (kComposite)
      key = (Key(tile) << 32) | Key(s_dkey[lo]);
    else
      key = Key(tile);
    const long long slot = base + e;
    if (slot < cap) {
      keys[slot] = key;
      vals[slot] = unsigned(g0 + lo);
    }
    for (int p = 0; p < passes; ++p) atomicAdd(&s_hist[p][unsigned(key >> (8 * p)) & 255u], 1u);
  }
  __syncthreads();
  for (int p = 0; p < passes; ++p) {
    const unsigned int v = s_hist[p][tid];
    if (v) atomicAdd(&hist[p * 256 + tid], v);
  }
}

// One stable LSD pass over the digit at bits [8*pass, 8*pass + 8).
template <typename Key>
__global__ void __launch_bounds__(kRadixThreads)
k_radix_pass(int pass, long long cap, Header* hdr, const unsigned int* __restrict__ hist,
             unsigned int* status, const Key* __restrict__ keys_in,
             const unsigned int* __restrict__ vals_in, Key* __restrict__ keys_out,
             unsigned int* __restrict__ vals_out) {
  __shared__ unsigned int s_whist[8][256];
  __shared__ unsigned int s_gbase[256];
  __shared__ unsigned int s_part;
  __shared__ long long s_n;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_part = atomicAdd(&hdr->radix_ticket[pass], 1u);
    const unsigned int f = ld_volatile(&hdr->flags);
    const long long P = hdr->pairs;
    s_n = (f & (GS2D_FLAG_CAPACITY | GS2D_FLAG_OVERFLOW | GS2D_FLAG_TIMEOUT)) ? 0 : (P < cap ? P : cap);
  }
  for (int k = tid; k < 8 * 256; k += blockDim.x) (&s_whist[0][0])[k] = 0u;
  __syncthreads();
  const long long n = s_n;
  const long long part = s_part;
  const long long base = part * kRadixItems;
  if (base >= n) return;
  const int shift = 8 * pass;

  Key k[kRadixPerThread];
  unsigned int v[kRadixPerThread], d[kRadixPerThread], rank[kRadixPerThread];
  const long long wbase = base + (long long)warp * (32 * kRadixPerThread);
#pragma unroll
  for (int j = 0; j < kRadixPerThread; ++j) {
    const long long idx = wbase + j * 32 + lane;
    const bool ok = idx < n;
    k[j] = ok ? keys_in[idx] : Key(0);
    v[j] = ok ? vals_in[idx] : 0u;
    d[j] = ok ? (unsigned(k[j] >> shift) & 255u) : 256u;
  }
  // Stable rank within the warp: item j of lane l precedes item j of lane
  // l+1 and every item j+1.
  const unsigned int lt = lanemask_lt();
#pragma unroll
  for (int j = 0; j < kRadixPerThread; ++j) {
    const unsigned int peers = __match_any_sync(0xffffffffu, d[j]);
    const int leader = 31 - __clz(peers);
    const unsigned int prev = (d[j] < 256u) ? s_whist[warp][d[j]] : 0u;
    __syncwarp();
    if (lane == leader && d[j] < 256u) s_whist[warp][d[j]] = prev + __popc(peers);
    __syncwarp();
    rank[j] = prev + __popc(peers & lt);
  }
  __syncthreads();
  // Per digit (thread tid = digit): exclusive offsets across warps and the
  // partition's total, then the look-back for the partitions before it.
  const unsigned int dg = tid;
  unsigned int run = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const unsigned int c = s_whist[w][dg];
    s_whist[w][dg] = run;
    run += c;
  }
  unsigned int* my = status + part * 256 + dg;
  unsigned int prefix = 0;
  if (part == 0) {
    st_volatile(my, kRadInc | run);
  } else {
    st_volatile(my, kRadAgg | run);
    for (long long j = part - 1; j >= 0; --j) {
      unsigned int s = 0, it = 0;
      while (((s = ld_volatile(status + j * 256 + dg)) >> 30) == 0u) {
        if (++it >= kSpinLimit) {
          atomicOr(&hdr->flags, (unsigned)GS2D_FLAG_TIMEOUT);
          break;
        }
        __nanosleep(32);
      }
      prefix += s & kRadVal;
      if ((s >> 30) == 2u || it >= kSpinLimit) break;
    }
    st_volatile(my, kRadInc | (prefix + run));
  }
  unsigned int gtot;
  const unsigned int gstart = block_exclusive_scan_256<unsigned int>(hist[pass * 256 + dg], &gtot);
  s_gbase[dg] = gstart + prefix;
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kRadixPerThread; ++j) {
    if (d[j] < 256u) {
      const unsigned int dst = s_gbase[d[j]] + s_whist[warp][d[j]] + rank[j];
      keys_out[dst] = k[j];
      vals_out[dst] = v[j];
    }
  }
}

template <typename Key>
__global__ void __launch_bounds__(256)
k_tile_ranges(int T, long long cap, const Header* __restrict__ hdr, const Key* __restrict__ keys,
              int2* __restrict__ ranges, int tile_shift) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const unsigned int f = hdr->flags;
  const long long P = hdr->pairs;
  const long long n =
      (f & (GS2D_FLAG_CAPACITY | GS2D_FLAG_OVERFLOW | GS2D_FLAG_TIMEOUT)) ? 0 : (P < cap ? P : cap);
  auto lower = [&](unsigned long long tile) {
    long long lo = 0, hi = n;
    while (lo < hi) {
      const long long mid = (lo + hi) >> 1;
      if ((unsigned long long)(keys[mid] >> tile_shift) < tile) lo = mid + 1; else hi = mid;
    }
    return lo;
  };
  ranges[t] = make_int2(int(lower(unsigned(t))), int(lower(unsigned(t) + 1ull)));
}

}  // namespace

cudaError_t launch_binning(const gs2d_config& c, int n, const gs2d_record* rec, const int* rect,
                           const int* count, long long cap, int* tile_ranges, int* sorted_gid,
                           unsigned char* ws, cudaStream_t s) {
  const Layout L = layout_of(c, n, cap);
  const bool comp = c.mode == GS2D_MODE_COMPOSITE;
  const int T = num_tiles(c);
  Header* hdr = reinterpret_cast<Header*>(ws);
  cudaError_t e = cudaMemsetAsync(ws, 0, L.offsets, s);  // header, histograms, scan words
  if (e != cudaSuccess) return e;
  unsigned int* hist = reinterpret_cast<unsigned int*>(ws + kOffHist);
  unsigned long long* scan_status = reinterpret_cast<unsigned long long*>(ws + L.scan);
  int* offsets = reinterpret_cast<int*>(ws + L.offsets);
  unsigned int* rstatus = reinterpret_cast<unsigned int*>(ws + L.radix_status);
  const long long zero_words = (long long)L.passes * L.partitions * 256;
  unsigned int* vals_a = (L.passes % 2 == 0) ? reinterpret_cast<unsigned int*>(sorted_gid)
                                             : reinterpret_cast<unsigned int*>(ws + L.vals_tmp);
  unsigned int* vals_b = (L.passes % 2 == 0) ? reinterpret_cast<unsigned int*>(ws + L.vals_tmp)
                                             : reinterpret_cast<unsigned int*>(sorted_gid);
  const int scan_blocks = n > 0 ? (n + kScanItems - 1) / kScanItems : 1;
  const int tx = tiles_x(c);
  const int radix_blocks = int(L.partitions);
  const int range_blocks = (T + 255) / 256;
  if (comp) {
    using Key = unsigned long long;
    Key* ka = reinterpret_cast<Key*>(ws + L.keys_a);
    Key* kb = reinterpret_cast<Key*>(ws + L.keys_b);
    k_scan_emit<true><<<scan_blocks, kScanThreads, 0, s>>>(
        n, tx, L.passes, cap, reinterpret_cast<const int4*>(rect), count,
        reinterpret_cast<const float4*>(rec), hdr, scan_status, hist, offsets, ka, vals_a, rstatus,
        zero_words);
    for (int p = 0; p < L.passes && radix_blocks > 0; ++p) {
      const bool even = (p % 2) == 0;
      k_radix_pass<Key><<<radix_blocks, kRadixThreads, 0, s>>>(
          p, cap, hdr, hist, rstatus + (size_t)p * L.partitions * 256, even ? ka : kb,
          even ? vals_a : vals_b, even ? kb : ka, even ? vals_b : vals_a);
    }
    k_tile_ranges<Key><<<range_blocks, 256, 0, s>>>(T, cap, hdr, (L.passes % 2 == 0) ? ka : kb,
                                                    reinterpret_cast<int2*>(tile_ranges), 32);
  } else {
    using Key = unsigned int;
    Key* ka = reinterpret_cast<Key*>(ws + L.keys_a);
    Key* kb = reinterpret_cast<Key*>(ws + L.keys_b);
    k_scan_emit<false><<<scan_blocks, kScanThreads, 0, s>>>(
        n, tx, L.passes, cap, reinterpret_cast<const int4*>(rect), count,
        reinterpret_cast<const float4*>(rec), hdr, scan_status, hist, offsets, ka, vals_a, rstatus,
        zero_words);
    for (int p = 0; p < L.passes && radix_blocks > 0; ++p) {
      const bool even = (p % 2) == 0;
      k_radix_pass<Key><<<radix_blocks, kRadixThreads, 0, s>>>(
          p, cap, hdr, hist, rstatus + (size_t)p * L.partitions * 256, even ? ka : kb,
          even ? vals_a : vals_b, even ? kb : ka, even ? vals_b : vals_a);
    }
    k_tile_ranges<Key><<<range_blocks, 256, 0, s>>>(T, cap, hdr, (L.passes % 2 == 0) ? ka : kb,
                                                    reinterpret_cast<int2*>(tile_ranges), 0);
  }
  return cudaGetLastError();
}

}  // namespace gs2d
