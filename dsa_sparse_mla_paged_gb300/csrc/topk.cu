// Stage 2: exact top-k over fp32 indexer scores.
//
// The article ("vLLM 为 Kimi K3.1 Pro 提供 Day-0 支持", "K3.1 Pro 中的稀疏注意力")
// keeps the 2,048 best-scoring tokens; this library fixes the order as (score
// descending, token index ascending) and writes the kept tokens in ascending
// index order.
//
// Scores are compared through an order-preserving 32-bit key (larger score ->
// larger key; -0 and +0 share one key). One kernel, C CTAs per row:
//   bound   every CTA of a row finds the same threshold key g from the group
//           maxima (the key of the largest score of each 128 and each 32
//           consecutive tokens, kept by the scorer's epilogue as it stores
//           the scores, or by topk_gmax_kernel for scores handed in by the
//           caller): with groups merged to at most 8,192, g = the lowest key of
//           the histogram bin that holds the K-th largest group maximum. K
//           groups each hold a token at or above g, so at least K tokens reach
//           g and the K-th largest score tau is >= g. Rows too short for that
//           bound to be tight take a guess instead (from an evenly spaced
//           sample, aimed at ~2K tokens);
//   filter  each CTA stages its chunk of scores in shared memory (one bulk
//           copy, in flight while the bound is found) and compacts the tokens
//           with key >= g, in index order, into the row's candidate buffer
//           (one atomic reservation per CTA, recorded per chunk);
//   select  the CTA that arrives last at the row's counter reads the
//           candidates, finds the exact K-th largest key tau among them
//           (histogram rounds, then the few keys of tau's bin ranked by a
//           warp) and writes the winners in index order, ties at tau lowest
//           index first: a winner's place is the winners of the chunks before
//           its own plus those before it in its own chunk (whose candidates are
//           contiguous and ordered), so the CTAs' arrival order never matters.
// Whenever at least K tokens reach g and the buffer holds them all, the
// candidates contain every token with key >= tau, so the selection is exact.
// Otherwise (a bound or guess that was too high, or more candidates than the
// buffer holds, e.g. a row of equal scores) the last CTA runs an exact radix
// select over the whole row by itself. So the maxima steer only the speed,
// never the result. No CTA waits on another: the last one to arrive continues.
#include <algorithm>

#include "block_select.cuh"
#include "dsa_internal.cuh"
#include "sm103_ptx.cuh"

namespace dsa {

namespace {

constexpr int kTkThreads = 1024;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kBoundPer = 8;                        // bound keys per thread
constexpr int kBoundKeys = kTkThreads * kBoundPer;  // 8,192 group maxima or samples at most
constexpr int kCandPer = kCandCap / kTkThreads;     // candidates per thread in the select
constexpr int kRoundTok = kTkWarps * 1024;          // tokens a CTA filters at most (1,024 per warp)
constexpr int kGmaxThreads = 256;

// row state words
// words 2 and 3 as one 64-bit counter: the candidates reserved so far (low
// half) and the CTAs of the row done with their chunk (high half), so that the
// last CTA's arrival returns the final count with it (every CTA reserves
// before it arrives); more than kCandCap means some chunk did not fit
constexpr int kStPair = 2;

struct TopkArgs {
  const float* scores;
  int64_t stride;
  const int32_t* ctx_lens;
  const int32_t* block_table;
  uint32_t* gmax;     // [rows][gstride] key of the largest score of each 32 tokens
  uint32_t* gmax128;  // [rows][g128stride] the same per 128 tokens (cleared after use)
  int gstride, g128stride;
  int n_q, cap, K, max_pages, num_pages, max_chunks;
  int chunk;       // tokens per CTA: a multiple of 1,024, at most kRoundTok
  int* state;      // [rows][kRowState]
  int* chunkinfo;  // [rows][max_chunks][2]: (offset, count) of each CTA's candidates
  uint64_t* cand;  // [rows][kCandCap]: key << 32 | token
  int* err;
  int32_t* topk_idx;
  int32_t* phys_rows;
  // dsa_decode: the latent pool whose rows the attention reads next; each CTA
  // prefetches its candidates' rows into L2 once its part is done (or null)
  const uint8_t* lat_pool;
  int64_t lat_stride;
  int lat_row;
};

__device__ __forceinline__ uint32_t order_key(float f) { return score_order_key(f); }

struct Row {
  int r, b, L;
};

__device__ __forceinline__ Row row_of(const TopkArgs& a, int r) {
  Row w;
  w.r = r;
  w.b = r / a.n_q;
  const int t = r - w.b * a.n_q;
  const int ctx = a.ctx_lens[w.b];
  w.L = (ctx < a.n_q || ctx > a.cap) ? -1 : ctx - a.n_q + t + 1;
  if (w.L > a.stride) w.L = -1;
  return w;
}

__device__ __forceinline__ int phys_row(const TopkArgs& a, int b, int s) {
  const int pg = a.block_table[size_t(b) * a.max_pages + s / kPage];
  if (pg < 0 || pg >= a.num_pages) {
    atomicOr(a.err, DSA_DEVERR_BLOCK_TABLE);
    return -1;
  }
  return pg * kPage + (s % kPage);
}

// How a row's threshold is found (the same answer in every CTA of the row).
enum BoundKind { kAll = 0, kMaxima = 1, kSample = 2 };

struct Bound {
  BoundKind kind;
  int gshift;  // 7: the 128-token maxima, 5: the 32-token ones
  int sh;      // 2^sh of them merged per group
};

// The coarser maxima when there are enough of them for a tight bound (several
// times K groups; below ~1.1 K most of the row would pass), else the finer;
// rows too short for either take a sample.
__device__ __forceinline__ Bound bound_of(int L, int K) {
  Bound bd{kAll, 0, 0};
  if (L <= kCandCap) return bd;
  const int n128 = (L + 127) >> 7, n32 = (L + 31) >> 5;
  int n;
  if (int64_t(n128) * 8 >= int64_t(K) * 9) {
    bd.gshift = 7;
    n = n128;
  } else if (int64_t(n32) * 8 >= int64_t(K) * 9) {
    bd.gshift = 5;
    n = n32;
  } else {
    bd.kind = kSample;
    return bd;
  }
  while (((n + (1 << bd.sh) - 1) >> bd.sh) > kBoundKeys) ++bd.sh;
  bd.kind = kMaxima;
  return bd;
}

// Visit every token s < L of `row` with its key, f(s, key): thread t takes
// float4 groups t, t + NT, ..., eight of them in flight per batch.
template <typename F>
__device__ __forceinline__ void for_row_keys(const float* row, int L, F&& f) {
  const int n4 = L >> 2;
  const float4* r4 = reinterpret_cast<const float4*>(row);
  for (int i0 = threadIdx.x; i0 < n4; i0 += kTkThreads * 8) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * kTkThreads;
      v[u] = i < n4 ? __ldcg(r4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * kTkThreads;
      if (i < n4) {
        f(4 * i, order_key(v[u].x));
        f(4 * i + 1, order_key(v[u].y));
        f(4 * i + 2, order_key(v[u].z));
        f(4 * i + 3, order_key(v[u].w));
      }
    }
  }
  for (int s = (n4 << 2) + int(threadIdx.x); s < L; s += kTkThreads) f(s, order_key(__ldcg(row + s)));
}

// Keys of the contiguous token range [s0, s1) of `row` (s0 a multiple of 4),
// f(s, key) in index order; eight float4 loads in flight per batch.
template <typename F>
__device__ __forceinline__ void for_range_keys(const float* row, int s0, int s1, F&& f) {
  const int n4 = max(0, s1 - s0) >> 2;
  const float4* r4 = reinterpret_cast<const float4*>(row + s0);
  for (int i0 = 0; i0 < n4; i0 += 8) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = i0 + u < n4 ? __ldcg(r4 + i0 + u) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (i0 + u < n4) {
        const int s = s0 + 4 * (i0 + u);
        f(s, order_key(v[u].x));
        f(s + 1, order_key(v[u].y));
        f(s + 2, order_key(v[u].z));
        f(s + 3, order_key(v[u].w));
      }
    }
  }
  for (int s = s0 + 4 * n4; s < s1; ++s) f(s, order_key(__ldcg(row + s)));
}

// ---------------------------------------------------------------- exact whole-row select
// By one CTA alone (the rare path): 11 + 11 + 10 key bits, each pass a
// histogram of the keys that match the prefix so far; then each thread takes a
// contiguous range of tokens, one scan places its winners, and they are written
// in index order (ties at tau lowest index first).
__device__ void select_whole_row(const TopkArgs& a, const Row& w, int* hist, int* smw, int32_t* out,
                                 int32_t* phys) {
  __shared__ uint32_t s_prefix;
  __shared__ int s_k;
  const float* row = a.scores + size_t(w.r) * a.stride;
  if (threadIdx.x == 0) { s_prefix = 0; s_k = a.K; }
  __syncthreads();
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = pass == 0 ? 21 : pass == 1 ? 10 : 0;
    const int width = pass == 2 ? 10 : 11;
    const int nb = 1 << width;
    for (int i = threadIdx.x; i < nb; i += kTkThreads) hist[i] = 0;
    __syncthreads();
    const uint32_t pre = s_prefix;
    const uint32_t hmask = pass == 0 ? 0u : (0xFFFFFFFFu << (sh + width));
    for_row_keys(row, w.L, [&](int, uint32_t u) {
      if ((u & hmask) == pre) {
        // lanes with the same bin add once (degenerate rows put every key in one bin)
        const uint32_t bin = (u >> sh) & uint32_t(nb - 1);
        const unsigned peers = __match_any_sync(__activemask(), bin);
        if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
      }
    });
    __syncthreads();
    // bins from the top; thread t owns bins nb-1-t*per .. nb-per-t*per
    const int per = nb / kTkThreads;
    int cnt = 0;
    for (int j = 0; j < per; ++j) cnt += hist[nb - 1 - threadIdx.x * per - j];
    int tot;
    const int before = block_excl_scan<kTkThreads>(cnt, &tot, smw);
    const int kk = s_k;
    __syncthreads();
    if (before < kk && kk <= before + cnt) {
      int cum = before;
      for (int j = 0; j < per; ++j) {
        const int bin = nb - 1 - threadIdx.x * per - j;
        if (kk <= cum + hist[bin]) {
          s_prefix = pre | (uint32_t(bin) << sh);
          s_k = kk - cum;
          break;
        }
        cum += hist[bin];
      }
    }
    __syncthreads();
  }
  const uint32_t tau = s_prefix;
  const int need = s_k;
  // thread t: tokens [t * P, t * P + P)
  const int P = ((w.L + kTkThreads - 1) / kTkThreads + 3) & ~3;
  const int s0 = min(w.L, int(threadIdx.x) * P), s1 = min(w.L, s0 + P);
  int gt = 0, eq = 0;
  for_range_keys(row, s0, s1, [&](int, uint32_t u) {
    gt += u > tau;
    eq += u == tau;
  });
  int tg, te;
  const int pg = block_excl_scan<kTkThreads>(gt, &tg, smw);
  int e = block_excl_scan<kTkThreads>(eq, &te, smw);
  if (gt + eq > 0) {
    int p = pg + min(e, need);
    for_range_keys(row, s0, s1, [&](int s, uint32_t u) {
      const bool sel = u > tau || (u == tau && e++ < need);
      if (sel) {
        if (p < a.K) {
          out[p] = s;
          if (phys) phys[p] = phys_row(a, w.b, s);
        }
        ++p;
      }
    });
  }
}

// ---------------------------------------------------------------- group maxima
// For scores handed in by the caller: the keys of the largest score of each
// 32 and each 128 consecutive tokens of every row that the bound will use, and
// the row's selection state cleared. A warp reads 1,024-token blocks (lane l:
// float4s 4 l + 128 i, eight in flight); a group of 32 is eight lanes'
// float4s, a group of 128 the warp's i-th load.
__global__ void __launch_bounds__(kGmaxThreads) topk_gmax_kernel(TopkArgs a) {
  pdl_wait();
  const Row w = row_of(a, blockIdx.y);
  int* st = a.state + size_t(w.r) * kRowState;
  if (blockIdx.x == 0 && threadIdx.x < 2) st[kStPair + threadIdx.x] = 0;
  if (w.L <= a.K || bound_of(w.L, a.K).kind != kMaxima) return;
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * (kGmaxThreads / 32);
  const float* row = a.scores + size_t(w.r) * a.stride;
  uint32_t* gm = a.gmax + size_t(w.r) * a.gstride;
  uint32_t* gm128 = a.gmax128 + size_t(w.r) * a.g128stride;
  for (int blk = blockIdx.x * (kGmaxThreads / 32) + (threadIdx.x >> 5); blk * 1024 < w.L; blk += nw) {
    float4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int s = blk * 1024 + 128 * i + 4 * lane;
      // a float4 that starts below L lies inside the row's stride (a multiple of 4)
      v[i] = s < w.L ? __ldcg(reinterpret_cast<const float4*>(row + s)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int s = blk * 1024 + 128 * i + 4 * lane;
      uint32_t m = 0u;
      if (s < w.L) m = order_key(v[i].x);
      if (s + 1 < w.L) m = max(m, order_key(v[i].y));
      if (s + 2 < w.L) m = max(m, order_key(v[i].z));
      if (s + 3 < w.L) m = max(m, order_key(v[i].w));
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 4));
      if ((lane & 7) == 0 && s < w.L) gm[s >> 5] = m;
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 8));
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 16));
      if (lane == 0 && s < w.L) gm128[s >> 7] = m;
    }
  }
}

// ---------------------------------------------------------------- the selection
// Dynamic shared memory: the CTA's chunk of scores (staged by one bulk copy
// while the bound is computed), later reused by the last CTA for the winner
// counts of the ordered write.
__global__ void __launch_bounds__(kTkThreads, 1) topk_kernel(TopkArgs a) {
  __shared__ int hw[4096];  // histograms of the selections
  __shared__ int smw[64];
  __shared__ uint32_t s_list[32];
  __shared__ int s_base, s_last, s_run, s_total;
  __shared__ int s_wt[kTkWarps];  // per warp: candidates, then their offset
  __shared__ __align__(8) uint64_t s_bar;
  extern __shared__ __align__(16) float stage[];
  const int tid = threadIdx.x;
  if (tid == 0) {
    ptx::mbar_init(&s_bar, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  // the attention's CTAs may take the SMs this grid leaves (they wait for its completion)
  pdl_trigger();
  const Row w = row_of(a, blockIdx.y);
  const int c = blockIdx.x, C = gridDim.x;
  int32_t* out = a.topk_idx + size_t(w.r) * a.K;
  int32_t* phys = a.phys_rows ? a.phys_rows + size_t(w.r) * a.K : nullptr;
  uint32_t* gm128 = a.gmax128 + size_t(w.r) * a.g128stride;
  if (w.L <= a.K) {
    // every visible token is kept (an invalid row keeps none)
    if (c != 0) return;
    if (w.L < 0 && tid == 0) atomicOr(a.err, DSA_DEVERR_CTX);
    for (int i = tid; i < a.K; i += kTkThreads) {
      const bool keep = i < w.L;
      out[i] = keep ? i : -1;
      if (phys) phys[i] = keep ? phys_row(a, w.b, i) : -1;
    }
    for (int i = tid; i < (w.L + 127) >> 7; i += kTkThreads) gm128[i] = 0u;  // for the scorer's next maxima
    return;
  }
  const float* row = a.scores + size_t(w.r) * a.stride;
  int* st = a.state + size_t(w.r) * kRowState;
  // CTA c filters tokens [rb, re); its scores go to shared memory by one bulk
  // copy (rounded up to 16 B: still inside the row, whose stride is a multiple of 4)
  const int rb = c * a.chunk;
  const int re = min(w.L, rb + a.chunk);
  const uint32_t nbytes = re > rb ? uint32_t((re - rb) * 4 + 15) & ~15u : 0u;
  if (tid == 0 && nbytes) {
    ptx::mbar_arrive_expect_tx(&s_bar, nbytes);
    for (uint32_t o = 0; o < nbytes; o += 32768)
      ptx::bulk_load(reinterpret_cast<uint8_t*>(stage) + o, reinterpret_cast<const uint8_t*>(row + rb) + o,
                     min(32768u, nbytes - o), &s_bar);
  }

  // ---------------------------------------------------------------- bound
  const Bound bd = bound_of(w.L, a.K);
  uint32_t g = 0u;
  if (bd.kind == kMaxima) {
    // group i: maxima [i << sh, (i + 1) << sh) of the chosen size, merged
    const int n = (w.L + (1 << bd.gshift) - 1) >> bd.gshift;
    const int ng = (n + (1 << bd.sh) - 1) >> bd.sh;
    const uint32_t* gm = bd.gshift == 7 ? gm128 : a.gmax + size_t(w.r) * a.gstride;
    uint32_t mk[kBoundPer];
#pragma unroll
    for (int u = 0; u < kBoundPer; ++u) {
      const int gi = u * kTkThreads + tid;
      mk[u] = (bd.sh == 0 && gi < ng) ? __ldcg(gm + gi) : 0u;
    }
    if (bd.sh > 0) {
#pragma unroll
      for (int u = 0; u < kBoundPer; ++u) {
        const int gi = u * kTkThreads + tid;
        if (gi < ng) {
          const int j0 = gi << bd.sh, j1 = min(n, j0 + (1 << bd.sh));
          for (int j = j0; j < j1; ++j) mk[u] = max(mk[u], __ldcg(gm + j));
        }
      }
    }
    // group gi sits in slot gi / threads: only the first ceil(ng / threads) slots hold any
    g = block_kth_lower<kTkThreads, kBoundPer>(mk, a.K, hw, smw, s_list, (ng + kTkThreads - 1) / kTkThreads);
  } else if (bd.kind == kSample) {
    // sample i at position floor(i * L / ns); the r-th largest, r for ~2K tokens
    const int ns = min(w.L, kBoundKeys);
    uint32_t sk[kBoundPer];
#pragma unroll
    for (int u = 0; u < kBoundPer; ++u) {
      const int i = u * kTkThreads + tid;
      sk[u] = i < ns ? order_key(__ldcg(row + int(int64_t(i) * w.L / ns))) : 0u;
    }
    const int r = int(min(int64_t(ns), (int64_t(2) * a.K * ns + w.L - 1) / w.L));
    g = block_kth_lower<kTkThreads, kBoundPer>(sk, r, hw, smw, s_list, (ns + kTkThreads - 1) / kTkThreads);
  }
  if (nbytes && !ptx::mbar_wait(&s_bar, 0)) {
    if (tid == 0) atomicOr(a.err, DSA_DEVERR_TIMEOUT);
    ptx::mbar_wait(&s_bar, 0);  // the copy still owns the buffer: one more bounded wait
  }

  // ---------------------------------------------------------------- filter
  // Warp w reads the block [rb + 1024 w, + 1024) from shared memory, lane l
  // its float4s l + 32 j (j < 8): (warp, j, lane, element) is index order.
  // One atomic reserves the CTA's place in the row's candidate buffer.
  const int lane = tid & 31, warp = tid >> 5;
  const unsigned lt = (1u << lane) - 1u;
  const int wb = rb + warp * 1024;
  uint32_t pass = 0u;  // bit 4 j + e: token wb + 4 (lane + 32 j) + e is a candidate
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int s = wb + 4 * (lane + 32 * j);
    if (s < re) {
      const float4 v = *reinterpret_cast<const float4*>(stage + (s - rb));
      pass |= uint32_t(order_key(v.x) >= g) << (4 * j);
      pass |= uint32_t(s + 1 < re && order_key(v.y) >= g) << (4 * j + 1);
      pass |= uint32_t(s + 2 < re && order_key(v.z) >= g) << (4 * j + 2);
      pass |= uint32_t(s + 3 < re && order_key(v.w) >= g) << (4 * j + 3);
    }
  }
  const int wcnt = __reduce_add_sync(0xffffffffu, __popc(pass));
  if (lane == 0) s_wt[warp] = wcnt;
  __syncthreads();
  if (warp == 0) {
    const int x = s_wt[lane];
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    s_wt[lane] = incl - x;
    const int run = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) {
      int base = 0;
      if (run > 0) {
        // (the low half never carries into the high one: at most cap tokens)
        base = int(uint32_t(atomicAdd(reinterpret_cast<unsigned long long*>(st + kStPair),
                                      static_cast<unsigned long long>(run))));
      }
      s_base = base;
      s_run = run;
      *reinterpret_cast<int2*>(a.chunkinfo + (size_t(w.r) * a.max_chunks + c) * 2) = make_int2(base, run);
    }
  }
  __syncthreads();
  if (wcnt > 0 && s_base + s_run <= kCandCap) {
    uint64_t* o = a.cand + size_t(w.r) * kCandCap + s_base + s_wt[warp];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      // this float4's candidates (0..4 per lane) placed by three bit-plane ballots
      const uint32_t ci = (pass >> (4 * j)) & 15u;
      const int nn = __popc(ci);
      const unsigned b0 = __ballot_sync(0xffffffffu, nn & 1), b1 = __ballot_sync(0xffffffffu, nn & 2),
                     b2 = __ballot_sync(0xffffffffu, nn & 4);
      const int ti = __popc(b0) + 2 * __popc(b1) + 4 * __popc(b2);
      if (ti == 0) continue;
      int p = __popc(b0 & lt) + 2 * __popc(b1 & lt) + 4 * __popc(b2 & lt);
      const int s = wb + 4 * (lane + 32 * j);
      if (ci) {
        const float4 v = *reinterpret_cast<const float4*>(stage + (s - rb));
        const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if ((ci >> e) & 1u) o[p++] = (uint64_t(order_key(vv[e])) << 32) | uint32_t(s + e);
      }
      o += ti;
    }
  }

  // the last CTA of the row to get here selects; every thread's candidate
  // writes are made visible device-wide before the CTA's arrival
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned long long old = atomicAdd(reinterpret_cast<unsigned long long*>(st + kStPair), 1ull << 32);
    s_last = int(old >> 32) == C - 1;
    s_total = int(uint32_t(old));
  }
  __syncthreads();
  if (!s_last) {
    // the attention gathers the winners' latent rows next: start pulling this
    // chunk's candidates (a superset of its winners) into L2
    // (Only where the bound filters: a row short enough that every token is a
    // candidate has few latent rows, and an SM works through bulk prefetches
    // at ~25 ns each, which would hold the grid, and the attention waiting on
    // it, for tens of microseconds. Likewise a CTA with many candidates.)
    if (a.lat_pool && bd.kind != kAll && s_run <= 512) {
      // the block-table entries of eight candidates at a time are loaded
      // together, not one dependent load per candidate
      const int32_t* bt = a.block_table + size_t(w.b) * a.max_pages;
      for (uint32_t m = pass; m;) {
        int ts[8], pg[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          ts[q] = -1;
          if (m) {
            const int j = __ffs(m) - 1;
            m &= m - 1u;
            ts[q] = wb + 4 * (lane + 32 * (j >> 2)) + (j & 3);
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) pg[q] = ts[q] >= 0 ? __ldg(bt + ts[q] / kPage) : -1;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (pg[q] >= 0 && pg[q] < a.num_pages)
            ptx::prefetch_l2_bulk(a.lat_pool + size_t(pg[q]) * a.lat_stride + size_t(ts[q] % kPage) * a.lat_row,
                                  a.lat_row);
      }
    }
    return;
  }
  __threadfence();
  const int total = s_total;
  if (total > kCandCap || total < a.K) {
    select_whole_row(a, w, hw, smw, out, phys);
  } else {
    // candidates in reservation order: each CTA's are contiguous and in index
    // order, the CTAs in any order. tau and the winners need no order; a
    // winner's output place is (winners of the chunks before its own) +
    // (winners of its chunk before it), its chunk being token / chunk. The
    // chunk records load with the candidates.
    // Thread t holds candidates t * per .. t * per + per - 1, per = ceil(total /
    // threads) (at most kCandPer): every loop over a thread's slots stops after
    // `per` of them. (This CTA's phases are bound by instruction issue, eight
    // warps per scheduler, so slots that would hold nothing still cost time.)
    const int per = (total + kTkThreads - 1) / kTkThreads;
    const uint64_t* cand = a.cand + size_t(w.r) * kCandCap;
    uint64_t cv[kCandPer];
#pragma unroll
    for (int u = 0; u < kCandPer; ++u) {
      const int p = tid * per + u;
      cv[u] = (u < per && p < total) ? __ldcg(cand + p) : 0ull;
    }
    const int* recs = a.chunkinfo + size_t(w.r) * a.max_chunks * 2;
    int2 rec = tid < C ? __ldcg(reinterpret_cast<const int2*>(recs) + tid) : make_int2(0, 0);
    uint32_t mk[kCandPer];
#pragma unroll
    for (int u = 0; u < kCandPer; ++u) mk[u] = uint32_t(cv[u] >> 32);
    // tau, and how many candidates lie above it (n_gt) and equal it (n_eq)
    int n_gt, n_eq;
    const uint32_t tau = block_kth_fast<kTkThreads, kCandPer>(mk, a.K, g, hw, smw, s_list, &n_gt, &n_eq, per);
    const int need = a.K - n_gt;
    // ties at tau: the `need` lowest tokens (the need-th largest of ~token)
    uint32_t tie_max = 0xFFFFFFFFu;
    if (n_eq > need) {
      uint32_t tk[kCandPer];
#pragma unroll
      for (int u = 0; u < kCandPer; ++u) tk[u] = mk[u] == tau ? 0xFFFFFFFFu - uint32_t(cv[u]) : 0u;
      tie_max = 0xFFFFFFFFu - block_kth_fast<kTkThreads, kCandPer>(tk, need, 0u, hw, smw, s_list, nullptr, nullptr, per);
    }
    unsigned win = 0;
#pragma unroll
    for (int u = 0; u < kCandPer; ++u) {
      if (u >= per) break;
      if (mk[u] > tau || (mk[u] == tau && uint32_t(cv[u]) <= tie_max)) win |= 1u << u;
    }
    int tw;
    const int wbase = block_excl_scan<kTkThreads>(__popc(win), &tw, smw);  // winners before mine
    // winners before reservation position p: s_wb[p / per] + those of its thread below p % per
    int* s_wb = reinterpret_cast<int*>(stage);    // [kTkThreads + 1]
    int* s_wm = s_wb + kTkThreads + 1;            // [kTkThreads] winner bits per thread
    int* s_first = s_wm + kTkThreads;             // [C] winners before the chunk's first candidate
    int* s_pre = s_first + C;                     // [C] winners of the chunks before
    s_wb[tid] = wbase;
    s_wm[tid] = int(win);
    if (tid == 0) s_wb[kTkThreads] = tw;
    __syncthreads();
    auto wbefore = [&](int p) {
      const int t = p / per;
      return t >= kTkThreads ? s_wb[kTkThreads]
                             : s_wb[t] + __popc(unsigned(s_wm[t]) & ((1u << (p - t * per)) - 1u));
    };
    int carry = 0;
    for (int c0 = 0; c0 < C; c0 += kTkThreads) {
      const int ch = c0 + tid;
      if (c0 > 0) rec = ch < C ? __ldcg(reinterpret_cast<const int2*>(recs) + ch) : make_int2(0, 0);
      int wch = 0, first = 0;
      if (ch < C && rec.y > 0) {
        first = wbefore(rec.x);
        wch = wbefore(rec.x + rec.y) - first;
      }
      int t;
      const int pre = block_excl_scan<kTkThreads>(wch, &t, smw) + carry;
      if (ch < C) {
        s_first[ch] = first;
        s_pre[ch] = pre;
      }
      carry += t;
    }
    __syncthreads();
    int wb = wbase;
    // a token's chunk, s / chunk, through the reciprocal: for any s < 2^31 and
    // chunk >= 1,024 the rounded product is within one of the quotient, and the
    // two comparisons correct it
    const float inv_chunk = 1.0f / float(a.chunk);
#pragma unroll
    for (int u = 0; u < kCandPer; ++u) {
      if (u >= per) break;
      if ((win >> u) & 1u) {
        const int s = int(uint32_t(cv[u]));
        int ch = int(float(s) * inv_chunk);
        if (ch * a.chunk > s) --ch;
        else if ((ch + 1) * a.chunk <= s) ++ch;
        const int pos = s_pre[ch] + (wb - s_first[ch]);
        if (pos < a.K) {
          out[pos] = s;
          if (phys) phys[pos] = phys_row(a, w.b, s);
        }
        ++wb;
      }
    }
  }
  // the row's 128-token maxima and state start from zero at the next call
  for (int i = tid; i < (w.L + 127) >> 7; i += kTkThreads) gm128[i] = 0u;
  __syncthreads();
  if (tid == 0) *reinterpret_cast<unsigned long long*>(st + kStPair) = 0ull;
}

}  // namespace

// CTAs per row: about one wave over all rows, each filtering a chunk of a
// multiple of 1,024 tokens, at most kRoundTok (so at most 8,192 CTAs per row
// at the largest cap).
struct TopkGrid {
  int ctas, chunk;
};

TopkGrid topk_grid(const WsLayout& L) {
  const int target = std::max(1, sm_count() / std::max(1, L.rows));
  TopkGrid g;
  g.chunk = std::min(kRoundTok, std::max(1024, (L.cap + target - 1) / target));
  g.chunk = (g.chunk + 1023) / 1024 * 1024;
  g.ctas = (L.cap + g.chunk - 1) / g.chunk;
  return g;
}

cudaError_t launch_topk(const dsa_params_t& p, const WsLayout& L, char* ws, const float* scores,
                        int64_t score_stride, const int32_t* ctx_lens, const int32_t* block_table,
                        int32_t* topk_idx, int32_t* phys_rows, cudaStream_t st, bool have_gmax,
                        const void* lat_pool) {
  TopkArgs a;
  a.scores = scores;
  a.stride = score_stride;
  a.ctx_lens = ctx_lens;
  a.block_table = block_table;
  a.gmax = reinterpret_cast<uint32_t*>(ws + L.gmax);
  a.gmax128 = reinterpret_cast<uint32_t*>(ws + L.gmax128);
  a.gstride = L.gstride;
  a.g128stride = L.g128stride;
  a.n_q = p.n_q;
  a.cap = L.cap;
  a.K = p.topk;
  a.max_pages = p.max_pages_per_req;
  a.num_pages = p.num_pages;
  a.max_chunks = L.max_chunks;
  a.state = reinterpret_cast<int*>(ws + L.state);
  a.chunkinfo = reinterpret_cast<int*>(ws + L.chunkinfo);
  a.cand = reinterpret_cast<uint64_t*>(ws + L.cand);
  a.err = reinterpret_cast<int*>(ws + L.err);
  a.topk_idx = topk_idx;
  a.phys_rows = phys_rows;
  a.lat_pool = static_cast<const uint8_t*>(lat_pool);
  a.lat_stride = p.lat_page_stride;
  a.lat_row = p.lat_fmt == DSA_LAT_NVFP4_352 ? kDNope / 2 + kDNope / 16 + kDRope : kLatRowFp8;
  cudaError_t e = cudaSuccess;
  if (!have_gmax) {
    const int gx = std::max(1, (L.cap + 16383) / 16384);  // two 1,024-token blocks per warp
    e = launch_pdl(topk_gmax_kernel, dim3(gx, L.rows), dim3(kGmaxThreads), 0, st, a);
  }
  const TopkGrid tg = topk_grid(L);
  a.chunk = tg.chunk;
  const size_t smem = std::max(size_t(tg.chunk) * 4, size_t(2 * kTkThreads + 1 + 2 * tg.ctas) * 4);
  // the kernel also has static shared memory: its dynamic part needs the
  // opt-in whenever the two together pass the default 48 KB
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e == cudaSuccess)
    e = launch_pdl(topk_kernel, dim3(tg.ctas, L.rows), dim3(kTkThreads), smem, st, a);
  return e;
}

}  // namespace dsa
