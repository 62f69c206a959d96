// Block-wide building blocks of the exact selections (top-k and the
// context-parallel merge): an exclusive scan and a radix select of the k-th
// largest 32-bit key, for CTAs of NT threads.
#pragma once

#include <stdint.h>

namespace dsa {

// Exclusive block scan of one int per thread (NT threads); *total gets the sum.
template <int NT>
__device__ __forceinline__ int block_excl_scan(int v, int* total, int* smw) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) smw[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < NW ? smw[lane] : 0;
#pragma unroll
    for (int o = 1; o < NW; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < NW) smw[lane] = s;
  }
  __syncthreads();
  const int pre = (warp ? smw[warp - 1] : 0) + x - v;
  *total = smw[NW - 1];
  __syncthreads();
  return pre;
}

// The k-th largest (1-based) of the keys held by the CTA (PER per thread; key
// 0 marks an empty slot and is never counted; 1 <= k <= number of keys).
// The bits all keys share (from the block's min and max key) are skipped; the
// rest are radix-selected 11 bits per pass with a shared histogram of 2048 bins
// (two buffers alternate, so `hist` holds 4096 ints and a buffer is cleared
// while the other fills). Per pass: histogram; per-warp sums of the bins from
// the top (each thread owns nb / NT bins); every warp scans the warp sums and
// the thread holding the k-th key finds its bin: three block barriers.
template <int NT, int PER>
__device__ uint32_t block_kth_key(const uint32_t (&keys)[PER], int k, int* hist, int* smw) {
  constexpr int NW = NT / 32;
  constexpr int kBins = 2048;
  constexpr int kMaxPer = (kBins + NT - 1) / NT;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __shared__ int s_sel[2];
  uint32_t mn = 0xFFFFFFFFu, mx = 0u;
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (keys[i]) { mn = min(mn, keys[i]); mx = max(mx, keys[i]); }
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) { smw[warp] = int(mn); smw[NW + warp] = int(mx); }
  for (int i = threadIdx.x; i < kBins; i += NT) hist[i] = 0;
  __syncthreads();
  mn = lane < NW ? uint32_t(smw[lane]) : 0xFFFFFFFFu;
  mx = lane < NW ? uint32_t(smw[NW + lane]) : 0u;
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  const uint32_t diff = mn ^ mx;
  if (diff == 0) return mx;
  int lo_bit = 32 - __clz(diff);  // bits [lo_bit, 32) are common to all keys
  uint32_t prefix = lo_bit >= 32 ? 0u : (mx >> lo_bit) << lo_bit;
  int kk = k;
  int buf = 0;
  __syncthreads();  // every warp has read smw before it is reused below
  while (lo_bit > 0) {
    const int width = min(11, lo_bit);
    const int sh = lo_bit - width;
    const int nb = 1 << width;
    int* H = hist + buf * kBins;
    int* Hn = hist + (buf ^ 1) * kBins;
    for (int i = threadIdx.x; i < kBins; i += NT) Hn[i] = 0;  // the next pass's buffer
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const uint32_t u = keys[i];
      const bool match = u != 0u && (lo_bit >= 32 || (u >> lo_bit) == (prefix >> lo_bit));
      if (match) atomicAdd(&H[(u >> sh) & uint32_t(nb - 1)], 1);
    }
    __syncthreads();
    // thread t owns bins nb-1-t*per .. nb-per-t*per (from the top)
    const int per = nb >= NT ? nb / NT : 1;
    const int top = nb - 1 - int(threadIdx.x) * per;
    int cnt[kMaxPer];
    int c = 0;
#pragma unroll
    for (int j = 0; j < kMaxPer; ++j) {
      cnt[j] = (j < per && top - j >= 0) ? H[top - j] : 0;
      c += cnt[j];
    }
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) smw[warp] = incl;
    __syncthreads();
    int wsum = lane < NW ? smw[lane] : 0;  // warp totals, scanned in every warp
    int wincl = wsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wincl, o);
      if (lane >= o) wincl += y;
    }
    const int base = __shfl_sync(0xffffffffu, wincl - wsum, warp);
    const int before = base + incl - c;
    if (before < kk && kk <= before + c) {
      int cum = before;
#pragma unroll
      for (int j = 0; j < kMaxPer; ++j) {
        if (j < per && kk <= cum + cnt[j]) {
          s_sel[0] = top - j;
          s_sel[1] = kk - cum;
          break;
        }
        cum += cnt[j];
      }
    }
    __syncthreads();
    prefix |= uint32_t(s_sel[0]) << sh;
    kk = s_sel[1];
    lo_bit = sh;
    buf ^= 1;
  }
  return prefix;
}

}  // namespace dsa

namespace dsa {

// The k-th largest (1-based) of the non-zero keys the CTA holds (PER per
// thread; 1 <= k <= their number), by histogram rounds over a key range.
// Round one's range is [lo, hi] of the keys warp 0 holds (lo no lower than
// `floor`, a key known to be at or below every key, or 0): every key is
// placed by (key - lo) >> shift into one of 2048 bins (keys outside the range
// go to the end bins), so keys that crowd into a narrow range still spread
// over many bins and the shared atomics rarely meet. Each further round
// spans the chosen bin's range. The bin holding the k-th key is found by all
// warps (two bins per thread, a warp sum each) and then warp 0 (the warp
// totals, then that warp's bins). LOWER: stop after one round and return the
// bin's lowest key (at least k keys reach it). Otherwise: stop when the bin is
// one key wide, or holds at most 32 keys (one warp ranks them), and return
// the exact k-th largest key, and in *n_gt / *n_eq (when not null) how many
// keys lie above it and how many equal it. Only each thread's first `nper`
// slots are read (a bound the whole CTA shares, so the loops stop together).
// NT = 1024; `hist` holds 4096 ints (two buffers: a round's bins are cleared
// while the other round's are read), `smw` 64, `list` 32.
template <int NT, int PER, bool LOWER>
__device__ uint32_t block_kth_range(const uint32_t (&keys)[PER], int k, uint32_t floor, int* hist, int* smw,
                                    uint32_t* list, int* n_gt = nullptr, int* n_eq = nullptr, int nper = PER) {
  static_assert(NT == 1024, "two bins per thread");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __shared__ int s_bin, s_rank, s_cnt, s_n, s_gt, s_eq;
  __shared__ uint32_t s_lo, s_hi, s_key;
  if (warp == 0) {
    uint32_t mn = 0xFFFFFFFFu, mx = 0u;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      if (i >= nper) break;
      if (keys[i]) { mn = min(mn, keys[i]); mx = max(mx, keys[i]); }
    }
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0) {
      if (mx == 0u) { mn = floor; mx = 0xFFFFFFFFu; }  // warp 0 holds no key: the widest range
      s_lo = max(mn, floor);
      s_hi = max(mx, max(mn, floor));
      s_n = 0;
      s_key = 0u;
    }
  }
  hist[threadIdx.x] = 0;
  hist[threadIdx.x + NT] = 0;
  __syncthreads();
  uint32_t lo = s_lo, hi = s_hi;
  int kk = k, buf = 0;
  bool first = true;
  while (true) {
    int* H = hist + buf * 2048;
    const uint32_t span = hi - lo;  // keys lo .. hi
    const int sh = span == 0u ? 0 : max(0, 21 - __clz(span));  // (span >> sh) < 2048
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      if (i >= nper) break;
      const uint32_t x = keys[i];
      if (x == 0u) continue;
      int b;
      if (first) {  // keys outside [lo, hi] go to the end bins
        b = x < lo ? 0 : x > hi ? 2047 : int((x - lo) >> sh);
      } else {
        if (x < lo || x > hi) continue;
        b = int((x - lo) >> sh);
      }
      atomicAdd(&H[b], 1);
    }
    __syncthreads();
    // thread t: bins 2047-2t and 2046-2t (from the top); warp w: bins 2047-64w ..
    const int c0 = H[2047 - 2 * threadIdx.x], c1 = H[2046 - 2 * threadIdx.x];
    int wsum = c0 + c1;
#pragma unroll
    for (int o = 16; o; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    if (lane == 0) smw[warp] = wsum;
    __syncthreads();
    if (warp == 0) {
      // defaults for fewer than kk keys (not expected: k <= the key count), so that no index leaves the bins
      if (lane == 0) {
        s_bin = 0;
        s_rank = 1;
        s_cnt = 0;
      }
      __syncwarp();
      const int wt = smw[lane];
      int incl = wt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, incl - wt < kk && kk <= incl);
      const int W = hit ? __ffs(hit) - 1 : 31;
      const int kr = kk - __shfl_sync(0xffffffffu, incl - wt, W);
      const int top = 2047 - 64 * W;  // warp W's bins, two per lane from the top
      const int a0 = H[top - 2 * lane], a1 = H[top - 2 * lane - 1];
      const int c2 = a0 + a1;
      int incl2 = c2;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl2, o);
        if (lane >= o) incl2 += y;
      }
      const int before = incl2 - c2;
      if (before < kr && kr <= incl2) {
        const int j = kr <= before + a0 ? 0 : 1;
        s_bin = top - 2 * lane - j;
        s_rank = kr - before - (j ? a0 : 0);
        s_cnt = j ? a1 : a0;
      }
    }
    hist[(buf ^ 1) * 2048 + threadIdx.x] = 0;  // the next round's bins (last read a round ago)
    hist[(buf ^ 1) * 2048 + threadIdx.x + NT] = 0;
    __syncthreads();
    buf ^= 1;
    const int b = s_bin;
    kk = s_rank;
    const int n = s_cnt;
    // bin b's keys: [lo + (b << sh), lo + (b << sh) + 2^sh - 1] (in 64 bits: the
    // top bin of round one may start past 2^32), widened at the ends in round one
    const uint64_t blo = uint64_t(lo) + (uint64_t(b) << sh);
    const uint64_t bhi = blo + ((uint64_t(1) << sh) - 1u);
    uint32_t nlo = uint32_t(min(blo, uint64_t(hi)));
    uint32_t nhi = uint32_t(min(bhi, uint64_t(hi)));
    const bool below = first && b == 0;  // bin 0 of round one also holds every key below lo
    if (below) nlo = floor;
    if (first && b == 2047) {  // the top bin of round one also holds every key above hi
      // (when its own range starts above hi, it holds only those: then hi < 2^32 - 1)
      nlo = blo <= uint64_t(hi) ? uint32_t(blo) : hi + 1u;
      nhi = 0xFFFFFFFFu;
    }
    first = false;
    if (LOWER) return below ? floor : nlo;
    lo = nlo;
    hi = nhi;
    if (lo == hi) {
      // the bin is one key wide: its n keys all equal the answer, and the
      // k - kk keys of the bins above it are larger
      if (n_gt) { *n_gt = k - kk; *n_eq = n; }
      return lo;
    }
    if (n <= 32) break;
  }
  // at most 32 keys lie in [lo, hi]: one warp ranks them
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    if (i >= nper) break;
    if (keys[i] && keys[i] >= lo && keys[i] <= hi) {
      const int at = atomicAdd(&s_n, 1);
      if (at < 32) list[at] = keys[i];
    }
  }
  __syncthreads();
  if (warp == 0) {
    const int n = min(s_n, 32);
    const uint32_t mine = lane < n ? list[lane] : 0u;
    int gt = 0, eq = 0;
    for (int j = 0; j < n; ++j) {
      const uint32_t x = list[j];
      gt += x > mine;
      eq += x == mine;
    }
    if (lane < n && gt < kk && kk <= gt + eq) {
      s_key = mine;
      s_gt = k - kk + gt;  // the keys of the bins above this one, and those above it in the bin
      s_eq = eq;
    }
  }
  __syncthreads();
  if (n_gt) { *n_gt = s_gt; *n_eq = s_eq; }
  return s_key;
}

template <int NT, int PER>
__device__ __forceinline__ uint32_t block_kth_fast(const uint32_t (&keys)[PER], int k, uint32_t floor, int* hist,
                                                   int* smw, uint32_t* list, int* n_gt = nullptr,
                                                   int* n_eq = nullptr, int nper = PER) {
  return block_kth_range<NT, PER, false>(keys, k, floor, hist, smw, list, n_gt, n_eq, nper);
}

// A key at or below the k-th largest such that at least k keys reach it.
template <int NT, int PER>
__device__ __forceinline__ uint32_t block_kth_lower(const uint32_t (&keys)[PER], int k, int* hist, int* smw,
                                                    uint32_t* list, int nper = PER) {
  return block_kth_range<NT, PER, true>(keys, k, 0u, hist, smw, list, nullptr, nullptr, nper);
}

}  // namespace dsa
