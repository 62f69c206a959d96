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
