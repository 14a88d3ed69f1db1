// Tile binning and sort.
//
//   1. k_scan_emit: exclusive scan of the per-Gaussian tile counts (block
//      scan + decoupled look-back across blocks), then every block emits the
//      (key, Gaussian index) pairs of its Gaussians in index order: key =
//      tile id (sum) or (tile id << 32 | depth key) (composite).  It also
//      builds the digit histograms of every radix pass and clears the state
//      the later kernels count on.
//   2. k_radix_pass (one launch per digit of up to 8 bits): stable LSD radix
//      sort, ranks by warp-level match plus a per-digit look-back across
//      partitions.  Emission in index order plus stable passes gives
//      ascending index within equal keys.
//   3. k_tile_bounds: [start, end) of every non-empty tile from the places
//      where the tile id changes along the sorted keys (empty tiles keep the
//      [0, 0) the first kernel wrote).
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
constexpr unsigned int kBadFlags = GS2D_FLAG_CAPACITY | GS2D_FLAG_OVERFLOW | GS2D_FLAG_TIMEOUT;

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

__device__ __forceinline__ uint4 ld_volatile4(const unsigned int* p) {
  uint4 v;
  asm volatile("ld.volatile.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Sum of the published counts of partitions [0, j) of one digit, whose
// look-back words lie contiguously in col[] (16-byte aligned, length a
// multiple of 4).  Reads 32 partitions per step with eight vector loads,
// from partition j-1 downwards, and stops at the first inclusive word.
__device__ unsigned int radix_lookback(const unsigned int* col, long long j, unsigned int* flags) {
  unsigned int prefix = 0, spins = 0;
  long long hi = j - 1;  // highest partition not counted yet
  while (hi >= 0) {
    const long long base = (hi | 3) - 31;  // window [base, base + 31], 4-aligned groups
    unsigned int s[32];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const long long gi = base + 4 * g;
      uint4 v = make_uint4(kRadInc, kRadInc, kRadInc, kRadInc);  // before partition 0: count 0
      if (gi >= 0) v = ld_volatile4(col + gi);
      s[4 * g] = v.x;
      s[4 * g + 1] = v.y;
      s[4 * g + 2] = v.z;
      s[4 * g + 3] = v.w;
    }
    unsigned int acc = 0;
    bool done = false, ready = true;
#pragma unroll
    for (int i = 31; i >= 0; --i) {
      if (base + i > hi || done || !ready) continue;
      const unsigned int st = s[i] >> 30;
      if (st == 0u) {
        ready = false;
        continue;
      }
      acc += s[i] & kRadVal;
      if (st == 2u) done = true;
    }
    if (!ready) {
      if (++spins >= kSpinLimit) {
        atomicOr(flags, (unsigned)GS2D_FLAG_TIMEOUT);
        return prefix + acc;
      }
      __nanosleep(32);
      continue;
    }
    prefix += acc;
    if (done) break;
    hi = base - 1;
  }
  return prefix;
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
using KeyOf = typename std::conditional<kComposite, unsigned long long, unsigned int>::type;

template <bool kComposite>
__global__ void __launch_bounds__(kScanThreads)
k_scan_emit(int n, int tiles_x, int passes, int digit_bits, long long cap,
            const int4* __restrict__ rect, const int* __restrict__ count,
            const float4* __restrict__ rec, Header* hdr, unsigned long long* scan_status,
            unsigned int* __restrict__ hist, int* __restrict__ offsets,
            KeyOf<kComposite>* __restrict__ keys, unsigned int* __restrict__ vals,
            unsigned int* __restrict__ zero_a, long long zero_a_words,
            unsigned int* __restrict__ zero_b, long long zero_b_words,
            unsigned long long keys_final) {
  using Key = KeyOf<kComposite>;
  extern __shared__ unsigned int s_hist[];  // [passes][1 << digit_bits]
  __shared__ long long s_excl[kScanItems + 1];
  __shared__ int4 s_rect[kScanItems];
  __shared__ unsigned int s_dkey[kComposite ? kScanItems : 1];
  __shared__ long long s_base;
  __shared__ unsigned int s_part;
  const int tid = threadIdx.x;
  const int radix = 1 << digit_bits;

  // Clear what the later kernels count on: the radix look-back words and
  // the tile ranges (empty tiles must read [0, 0)).
  const long long gstride = (long long)gridDim.x * blockDim.x;
  for (long long k = (long long)blockIdx.x * blockDim.x + tid; k < zero_a_words; k += gstride)
    zero_a[k] = 0u;
  for (long long k = (long long)blockIdx.x * blockDim.x + tid; k < zero_b_words; k += gstride)
    zero_b[k] = 0u;

  if (tid == 0) {
    s_part = atomicAdd(&hdr->scan_ticket, 1u);
    if (blockIdx.x == 0) hdr->keys_final = keys_final;
  }
  for (int k = tid; k < passes * radix; k += blockDim.x) s_hist[k] = 0u;
  __syncthreads();
  const long long part = s_part;
  const long long g = part * kScanItems + tid;

  const int cnt = (g < n) ? count[g] : 0;
  s_rect[tid] = (g < n) ? rect[g] : make_int4(0, 0, -1, -1);
  if constexpr (kComposite) s_dkey[tid] = (g < n) ? depth_key(rec[3 * g + 2].w) : 0u;
  long long total;
  const long long excl = block_exclusive_scan_256<long long>(cnt, &total);
  s_excl[tid] = excl;
  if (tid == 0) {
    s_excl[kScanItems] = total;
    st_volatile(&scan_status[part], (part == 0 ? kScanInc : kScanAgg) | (unsigned long long)total);
  }
  if (tid < 32) {
    // Warp-wide look-back: lane l reads the word of partition hi - l.
    const int lane = tid;
    long long prefix = 0, hi = part - 1;
    unsigned int spins = 0;
    while (hi >= 0) {
      const long long idx = hi - lane;
      const unsigned long long v = (idx >= 0) ? ld_volatile(&scan_status[idx]) : kScanInc;
      const unsigned int st = unsigned(v >> 62);
      const unsigned int inc = __ballot_sync(0xffffffffu, st == 2u);
      const unsigned int notready = __ballot_sync(0xffffffffu, st == 0u);
      const int first = inc ? __ffs(inc) - 1 : 31;  // lanes [0, first] are needed
      const unsigned int need = first >= 31 ? 0xffffffffu : ((2u << first) - 1u);
      if (notready & need) {
        if (++spins >= kSpinLimit) {
          if (lane == 0) atomicOr(&hdr->flags, (unsigned)GS2D_FLAG_TIMEOUT);
          break;
        }
        __nanosleep(32);
        continue;
      }
      long long val = (lane <= first) ? (long long)(v & kScanVal) : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) val += __shfl_xor_sync(0xffffffffu, val, o);
      prefix += val;
      if (inc) break;
      hi -= 32;
    }
    if (lane == 0) {
      if (part > 0) st_volatile(&scan_status[part], kScanInc | (unsigned long long)(prefix + total));
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
  }
  __syncthreads();
  const long long base = s_base;
  if (g < n) {
    const long long o = base + excl;
    offsets[g] = o < (1ll << 31) ? int(o) : 0x7fffffff;
  }

  // Emission: pair e of this block belongs to the last local Gaussian whose
  // exclusive offset is <= e (that one has a non-zero count).
  const unsigned int dmask = unsigned(radix - 1);
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
      vals[slot] = unsigned(part * kScanItems + lo);
    }
    for (int p = 0; p < passes; ++p)
      atomicAdd(&s_hist[p * radix + (unsigned(key >> (digit_bits * p)) & dmask)], 1u);
  }
  __syncthreads();
  for (int k = tid; k < passes * radix; k += blockDim.x) {
    const unsigned int v = s_hist[k];
    if (v) atomicAdd(&hist[(k / radix) * kMaxRadix + (k % radix)], v);
  }
}

// One stable LSD pass over the digit at bits [digit_bits * pass, + digit_bits).
// kRadix is the bucket capacity; the pass uses 1 << digit_bits buckets.
template <typename Key, int kRadix, int kPerThread>
__global__ void __launch_bounds__(kRadixThreads)
k_radix_pass(int pass, int digit_bits, long long cap, long long partitions4, Header* hdr,
             const unsigned int* __restrict__ hist, unsigned int* status,
             const Key* __restrict__ keys_in, const unsigned int* __restrict__ vals_in,
             Key* __restrict__ keys_out, unsigned int* __restrict__ vals_out) {
  constexpr int kDigitsPerThread = kRadix / kRadixThreads;
  constexpr int kItems = kRadixThreads * kPerThread;
  __shared__ unsigned short s_whist[8][kRadix];  // per-warp counts, then exclusive offsets
  __shared__ unsigned int s_gbase[kRadix];
  __shared__ unsigned int s_part;
  __shared__ long long s_n;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int radix = 1 << digit_bits;
  if (tid == 0) {
    s_part = atomicAdd(&hdr->radix_ticket[pass], 1u);
    const unsigned int f = ld_volatile(&hdr->flags);
    const long long P = hdr->pairs;
    s_n = (f & kBadFlags) ? 0 : (P < cap ? P : cap);
  }
  for (int k = tid; k < 8 * kRadix; k += blockDim.x) (&s_whist[0][0])[k] = 0;
  __syncthreads();
  const long long n = s_n;
  const long long part = s_part;
  const long long base = part * kItems;
  if (base >= n) return;
  const int shift = digit_bits * pass;
  const unsigned int dmask = unsigned(radix - 1);

  Key k[kPerThread];
  unsigned int v[kPerThread], d[kPerThread], rank[kPerThread];
  const long long wbase = base + (long long)warp * (32 * kPerThread);
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const long long idx = wbase + j * 32 + lane;
    const bool ok = idx < n;
    k[j] = ok ? keys_in[idx] : Key(0);
    v[j] = ok ? vals_in[idx] : 0u;
    d[j] = ok ? (unsigned(k[j] >> shift) & dmask) : unsigned(kRadix);
  }
  // Stable rank within the warp: item j of lane l precedes item j of lane
  // l+1 and every item j+1.
  const unsigned int lt = lanemask_lt();
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const unsigned int peers = __match_any_sync(0xffffffffu, d[j]);
    const int leader = 31 - __clz(peers);
    const unsigned int prev = (d[j] < unsigned(kRadix)) ? s_whist[warp][d[j]] : 0u;
    __syncwarp();
    if (lane == leader && d[j] < unsigned(kRadix))
      s_whist[warp][d[j]] = (unsigned short)(prev + __popc(peers));
    __syncwarp();
    rank[j] = prev + __popc(peers & lt);
  }
  // Global start of every digit: exclusive scan of this pass's histogram
  // (blocked: the digits of one thread are adjacent).
  unsigned int hsum[kDigitsPerThread], hloc = 0;
#pragma unroll
  for (int q = 0; q < kDigitsPerThread; ++q) {
    const int dg = tid * kDigitsPerThread + q;
    hsum[q] = (dg < radix) ? hist[pass * kMaxRadix + dg] : 0u;
    hloc += hsum[q];
  }
  unsigned int gtot;
  unsigned int gstart = block_exclusive_scan_256<unsigned int>(hloc, &gtot);  // syncs the block
  // Per digit: exclusive offsets across warps and the partition's count,
  // published for every digit before any look-back starts.
  unsigned int run[kDigitsPerThread];
#pragma unroll
  for (int q = 0; q < kDigitsPerThread; ++q) {
    const int dg = tid * kDigitsPerThread + q;
    unsigned int r = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const unsigned int c = s_whist[w][dg];
      s_whist[w][dg] = (unsigned short)r;
      r += c;
    }
    run[q] = r;
    if (dg < radix) st_volatile(status + (long long)dg * partitions4 + part, (part == 0 ? kRadInc : kRadAgg) | r);
  }
#pragma unroll
  for (int q = 0; q < kDigitsPerThread; ++q) {
    const int dg = tid * kDigitsPerThread + q;
    unsigned int prefix = 0;
    if (dg < radix && part > 0) {
      unsigned int* colp = status + (long long)dg * partitions4;
      prefix = radix_lookback(colp, part, &hdr->flags);
      st_volatile(colp + part, kRadInc | (prefix + run[q]));
    }
    s_gbase[dg] = gstart + prefix;
    gstart += hsum[q];
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    if (d[j] < unsigned(kRadix)) {
      const unsigned int dst = s_gbase[d[j]] + s_whist[warp][d[j]] + rank[j];
      keys_out[dst] = k[j];
      vals_out[dst] = v[j];
    }
  }
}

template <typename Key>
__global__ void __launch_bounds__(256)
k_tile_bounds(long long cap, const Header* __restrict__ hdr, const Key* __restrict__ keys,
              int2* __restrict__ ranges, int tile_shift) {
  const unsigned int f = hdr->flags;
  const long long P = hdr->pairs;
  const long long n = (f & kBadFlags) ? 0 : (P < cap ? P : cap);
  int* rg = reinterpret_cast<int*>(ranges);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const unsigned int t = unsigned(keys[i] >> tile_shift);
    if (i == 0 || unsigned(keys[i - 1] >> tile_shift) != t) rg[2 * size_t(t)] = int(i);
    if (i == n - 1 || unsigned(keys[i + 1] >> tile_shift) != t) rg[2 * size_t(t) + 1] = int(i + 1);
  }
}

template <typename Key, int kRadix, int kPerThread>
void launch_passes(const Layout& L, long long cap, Header* hdr, const unsigned int* hist,
                   unsigned int* rstatus, Key* ka, Key* kb, unsigned int* va, unsigned int* vb,
                   cudaStream_t s) {
  const int blocks = int(L.partitions);
  const size_t radix = size_t(1) << L.digit_bits;
  for (int p = 0; p < L.passes && blocks > 0; ++p) {
    const bool even = (p % 2) == 0;
    k_radix_pass<Key, kRadix, kPerThread><<<blocks, kRadixThreads, 0, s>>>(
        p, L.digit_bits, cap, L.partitions4, hdr, hist, rstatus + size_t(p) * L.partitions4 * radix,
        even ? ka : kb, even ? va : vb, even ? kb : ka, even ? vb : va);
  }
}

template <bool kComposite>
cudaError_t launch_binning_t(const gs2d_config& c, int n, const gs2d_record* rec, const int* rect,
                             const int* count, long long cap, int* tile_ranges, int* sorted_gid,
                             unsigned char* ws, cudaStream_t s) {
  using Key = KeyOf<kComposite>;
  const Layout L = layout_of(c, n, cap);
  const int T = num_tiles(c);
  Header* hdr = reinterpret_cast<Header*>(ws);
  cudaError_t e = cudaMemsetAsync(ws, 0, L.offsets, s);  // header, histograms, scan words
  if (e != cudaSuccess) return e;
  unsigned int* hist = reinterpret_cast<unsigned int*>(ws + kOffHist);
  unsigned long long* scan_status = reinterpret_cast<unsigned long long*>(ws + L.scan);
  int* offsets = reinterpret_cast<int*>(ws + L.offsets);
  unsigned int* rstatus = reinterpret_cast<unsigned int*>(ws + L.radix_status);
  const size_t radix = size_t(1) << L.digit_bits;
  const long long status_words = (long long)L.passes * L.partitions4 * (long long)radix;
  unsigned int* vals_a = (L.passes % 2 == 0) ? reinterpret_cast<unsigned int*>(sorted_gid)
                                             : reinterpret_cast<unsigned int*>(ws + L.vals_tmp);
  unsigned int* vals_b = (L.passes % 2 == 0) ? reinterpret_cast<unsigned int*>(ws + L.vals_tmp)
                                             : reinterpret_cast<unsigned int*>(sorted_gid);
  Key* ka = reinterpret_cast<Key*>(ws + L.keys_a);
  Key* kb = reinterpret_cast<Key*>(ws + L.keys_b);
  const size_t keys_final = (L.passes % 2 == 0) ? L.keys_a : L.keys_b;
  const int scan_blocks = n > 0 ? (n + kScanItems - 1) / kScanItems : 1;
  const size_t hist_smem = sizeof(unsigned int) * size_t(L.passes > 0 ? L.passes : 1) * radix;
  auto kern = k_scan_emit<kComposite>;
  if (hist_smem > 32 * 1024) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(hist_smem));
    if (e != cudaSuccess) return e;
  }
  kern<<<scan_blocks, kScanThreads, hist_smem, s>>>(
      n, tiles_x(c), L.passes, L.digit_bits, cap, reinterpret_cast<const int4*>(rect), count,
      reinterpret_cast<const float4*>(rec), hdr, scan_status, hist, offsets, ka, vals_a, rstatus,
      status_words, reinterpret_cast<unsigned int*>(tile_ranges), 2ll * T,
      (unsigned long long)keys_final);
  launch_passes<Key, kMaxRadix, 8>(L, cap, hdr, hist, rstatus, ka, kb, vals_a, vals_b, s);
  if (cap > 0) {
    long long blocks = (cap + 255) / 256;
    if (blocks > 148 * 16) blocks = 148 * 16;
    k_tile_bounds<Key><<<int(blocks), 256, 0, s>>>(
        cap, hdr, reinterpret_cast<const Key*>(ws + keys_final),
        reinterpret_cast<int2*>(tile_ranges), kComposite ? 32 : 0);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_binning(const gs2d_config& c, int n, const gs2d_record* rec, const int* rect,
                           const int* count, long long cap, int* tile_ranges, int* sorted_gid,
                           unsigned char* ws, cudaStream_t s) {
  if (c.mode == GS2D_MODE_COMPOSITE)
    return launch_binning_t<true>(c, n, rec, rect, count, cap, tile_ranges, sorted_gid, ws, s);
  return launch_binning_t<false>(c, n, rec, rect, count, cap, tile_ranges, sorted_gid, ws, s);
}

}  // namespace gs2d
