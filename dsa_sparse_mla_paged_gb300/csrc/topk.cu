// Stage 2: exact top-k over fp32 indexer scores.
//
// The article ("vLLM 为 Kimi K3.1 Pro 提供 Day-0 支持", "K3.1 Pro 中的稀疏注意力")
// keeps the 2,048 best-scoring tokens; this library fixes the order as (score
// descending, token index ascending) and writes the kept tokens in ascending
// index order.
//
// Scores are compared through an order-preserving 32-bit key (larger score ->
// larger key; -0 and +0 share one key). One kernel, C CTAs per row:
//   bound   every CTA of a row finds the same threshold key g:
//           - from the group maxima (the largest key of each 32 consecutive
//             tokens, written by the scorer's epilogue as it stores the scores,
//             or by topk_gmax_kernel for scores handed in by the caller): with
//             groups merged to at most 8,192, g = the K-th largest group
//             maximum. K groups each hold a token at or above g, so at least K
//             tokens reach g and the K-th largest score tau is >= g: a bound,
//             not a guess;
//           - for rows too short for that bound to be tight, g is a guess (the
//             r-th largest of an evenly spaced sample, r set for ~2K tokens);
//   filter  each CTA compacts the tokens of its chunk with key >= g, in index
//           order, into the row's candidate buffer (one atomic reservation per
//           CTA, its place recorded per chunk);
//   select  the CTA that arrives last at the row's counter gathers the
//           candidates chunk by chunk (in index order again), radix-selects the
//           exact K-th largest key tau among them and writes the winners in
//           order, ties at tau lowest index first.
// Whenever at least K tokens reach g and the buffer holds them all, the
// candidates contain every token with key >= tau, so the selection is exact.
// Otherwise (a guess that was too high, or more candidates than the buffer
// holds, e.g. a row of equal scores) the last CTA runs an exact radix select
// over the whole row by itself. No CTA waits on another: the last one to
// arrive continues, and the result does not depend on the order of arrival.
#include <algorithm>

#include "block_select.cuh"
#include "dsa_internal.cuh"
#include "sm103_ptx.cuh"

namespace dsa {

namespace {

constexpr int kTkThreads = 1024;
constexpr int kBoundPer = 8;                        // bound keys per thread
constexpr int kBoundKeys = kTkThreads * kBoundPer;  // 8,192 group maxima or samples at most
constexpr int kCandPer = kCandCap / kTkThreads;     // candidates per thread in the select
constexpr int kRoundTok = 32 * 1024;                // tokens a CTA filters at most (1,024 per warp)
constexpr int kGmaxThreads = 256;

// row state words
constexpr int kStCursor = 1;   // candidates reserved so far
constexpr int kStOverflow = 2; // a chunk did not fit the buffer
constexpr int kStArrived = 3;  // CTAs of the row done with their chunk

struct TopkArgs {
  const float* scores;
  int64_t stride;
  const int32_t* ctx_lens;
  const int32_t* block_table;
  const uint32_t* gmax;  // [rows][gstride] key of the largest score of each 32 tokens
  int gstride;
  int n_q, cap, K, max_pages, num_pages, max_chunks;
  int chunk;       // tokens per CTA: a multiple of 1,024, at most kRoundTok
  int* state;      // [rows][kRowState]
  int* chunkinfo;  // [rows][max_chunks][2]: (offset, count) in the candidate buffer, per CTA
  uint64_t* cand;  // [rows][kCandCap]: key << 32 | token
  int* err;
  int32_t* topk_idx;
  int32_t* phys_rows;
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

// Group maxima are merged 2^sh at a time so that at most kBoundKeys remain.
// The bound is tight once there are several times K groups; below ~1.1 K it
// would let most of the row through, and a sample serves better.
__device__ __forceinline__ BoundKind bound_kind(int L, int K, int* sh) {
  if (L <= kCandCap) return kAll;
  const int n32 = (L + 31) >> 5;
  if (int64_t(n32) * 8 < int64_t(K) * 9) return kSample;
  int s = 0;
  while (((n32 + (1 << s) - 1) >> s) > kBoundKeys) ++s;
  *sh = s;
  return kMaxima;
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
// For scores handed in by the caller: the key of the largest score of each 32
// consecutive tokens of every row that the bound will use, and the row's
// selection state cleared. A warp reads 1,024-token blocks (lane l: float4s
// 4 l + 128 i, eight in flight); each group of 32 is eight lanes' float4s.
__global__ void __launch_bounds__(kGmaxThreads) topk_gmax_kernel(TopkArgs a, uint32_t* gmax) {
  pdl_wait();
  const Row w = row_of(a, blockIdx.y);
  int* st = a.state + size_t(w.r) * kRowState;
  if (blockIdx.x == 0 && threadIdx.x < 3) st[kStCursor + threadIdx.x] = 0;
  int sh = 0;
  if (w.L <= a.K || bound_kind(w.L, a.K, &sh) != kMaxima) return;
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * (kGmaxThreads / 32);
  const float* row = a.scores + size_t(w.r) * a.stride;
  uint32_t* gm = gmax + size_t(w.r) * a.gstride;
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
    }
  }
}

// ---------------------------------------------------------------- the selection
__global__ void __launch_bounds__(kTkThreads, 1) topk_kernel(TopkArgs a) {
  __shared__ int hist[4096];
  __shared__ int smw[64];
  __shared__ int s_base, s_last, s_run;
  __shared__ int s_wt[32];
  extern __shared__ int rec_smem[];  // the last CTA: [nrec + 1] prefix of counts, [nrec] offsets
  pdl_wait();
  const int tid = threadIdx.x;
  const Row w = row_of(a, blockIdx.y);
  const int c = blockIdx.x, C = gridDim.x;
  int32_t* out = a.topk_idx + size_t(w.r) * a.K;
  int32_t* phys = a.phys_rows ? a.phys_rows + size_t(w.r) * a.K : nullptr;
  if (w.L <= a.K) {
    // every visible token is kept (an invalid row keeps none)
    if (c != 0) return;
    if (w.L < 0 && tid == 0) atomicOr(a.err, DSA_DEVERR_CTX);
    for (int i = tid; i < a.K; i += kTkThreads) {
      const bool keep = i < w.L;
      out[i] = keep ? i : -1;
      if (phys) phys[i] = keep ? phys_row(a, w.b, i) : -1;
    }
    return;
  }
  const float* row = a.scores + size_t(w.r) * a.stride;
  int* st = a.state + size_t(w.r) * kRowState;

  // ---------------------------------------------------------------- bound
  int sh = 0;
  const BoundKind kind = bound_kind(w.L, a.K, &sh);
  uint32_t g = 0u;
  if (kind == kMaxima) {
    // group i: 32-token maxima [i << sh, (i + 1) << sh) merged
    const int n32 = (w.L + 31) >> 5;
    const int ng = (n32 + (1 << sh) - 1) >> sh;
    const uint32_t* gm = a.gmax + size_t(w.r) * a.gstride;
    uint32_t mk[kBoundPer];
    if (sh >= 2) {
#pragma unroll
      for (int u = 0; u < kBoundPer; ++u) mk[u] = 0u;
      // uint4 words; a group's words are [i << sh, min(n32, (i + 1) << sh))
      const int nq = 1 << (sh - 2);
      for (int q = 0; q < nq; ++q) {
        uint4 v[kBoundPer];
#pragma unroll
        for (int u = 0; u < kBoundPer; ++u) {
          const int gi = u * kTkThreads + tid;
          const int j = (gi << sh) + 4 * q;
          v[u] = (gi < ng && j < n32) ? __ldcg(reinterpret_cast<const uint4*>(gm + j)) : make_uint4(0, 0, 0, 0);
          if (gi < ng && j < n32 && j + 4 > n32) {  // the row's last words: only those below n32
            if (j + 1 >= n32) v[u].y = 0u;
            if (j + 2 >= n32) v[u].z = 0u;
            v[u].w = 0u;
          }
        }
#pragma unroll
        for (int u = 0; u < kBoundPer; ++u) mk[u] = max(mk[u], max(max(v[u].x, v[u].y), max(v[u].z, v[u].w)));
      }
    } else {
#pragma unroll
      for (int u = 0; u < kBoundPer; ++u) {
        const int gi = u * kTkThreads + tid;
        uint32_t m = 0u;
        if (gi < ng) {
          const int j0 = gi << sh, j1 = min(n32, j0 + (1 << sh));
          for (int j = j0; j < j1; ++j) m = max(m, __ldcg(gm + j));
        }
        mk[u] = m;
      }
    }
    g = block_kth_key<kTkThreads, kBoundPer>(mk, a.K, hist, smw);
  } else if (kind == kSample) {
    // sample i at position floor(i * L / ns); the r-th largest, r for ~2K tokens
    const int ns = min(w.L, kBoundKeys);
    uint32_t sk[kBoundPer];
#pragma unroll
    for (int u = 0; u < kBoundPer; ++u) {
      const int i = u * kTkThreads + tid;
      sk[u] = i < ns ? order_key(__ldcg(row + int(int64_t(i) * w.L / ns))) : 0u;
    }
    const int r = int(min(int64_t(ns), (int64_t(2) * a.K * ns + w.L - 1) / w.L));
    g = block_kth_key<kTkThreads, kBoundPer>(sk, r, hist, smw);
  }

  // ---------------------------------------------------------------- filter
  // CTA c: tokens [c * chunk, (c + 1) * chunk); warp w reads [base + 1024 w,
  // + 1024), lane l the float4s l + 32 i (i < 8): coalesced, and (warp, i, lane,
  // element) is index order. The CTA reserves its place with one atomic and
  // records it at index c.
  const int lane = tid & 31, warp = tid >> 5;
  const unsigned lt = (1u << lane) - 1u;
  {
    const int rb = c * a.chunk;
    const int re = min(w.L, rb + a.chunk);
    const int wb = rb + warp * 1024;
    float4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int s = wb + 4 * (lane + 32 * i);
      // a float4 that starts below re lies inside the row's stride (a multiple of 4)
      v[i] = s < re ? __ldcg(reinterpret_cast<const float4*>(row + s)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    uint32_t pass = 0;  // bit 4i + j: token wb + 4 (lane + 32 i) + j is a candidate
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int s = wb + 4 * (lane + 32 * i);
      pass |= uint32_t(s < re && order_key(v[i].x) >= g) << (4 * i);
      pass |= uint32_t(s + 1 < re && order_key(v[i].y) >= g) << (4 * i + 1);
      pass |= uint32_t(s + 2 < re && order_key(v[i].z) >= g) << (4 * i + 2);
      pass |= uint32_t(s + 3 < re && order_key(v[i].w) >= g) << (4 * i + 3);
    }
    const int wtot = __reduce_add_sync(0xffffffffu, __popc(pass));
    if (lane == 0) s_wt[warp] = wtot;
    __syncthreads();
    if (tid == 0) {
      int run = 0;
      for (int i = 0; i < 32; ++i) {
        const int x = s_wt[i];
        s_wt[i] = run;
        run += x;
      }
      int base = 0;
      if (run > 0) {
        base = atomicAdd(st + kStCursor, run);
        if (base + run > kCandCap) atomicOr(st + kStOverflow, 1);
      }
      s_base = base;
      s_run = run;
      *reinterpret_cast<int2*>(a.chunkinfo + (size_t(w.r) * a.max_chunks + c) * 2) = make_int2(base, run);
    }
    __syncthreads();
    if (wtot > 0 && s_base + s_run <= kCandCap) {
      uint64_t* o = a.cand + size_t(w.r) * kCandCap + s_base + s_wt[warp];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        // this float4's candidates (0..4 per lane) placed by three bit-plane ballots
        const uint32_t ci = (pass >> (4 * i)) & 15u;
        const int n = __popc(ci);
        const unsigned b0 = __ballot_sync(0xffffffffu, n & 1), b1 = __ballot_sync(0xffffffffu, n & 2),
                       b2 = __ballot_sync(0xffffffffu, n & 4);
        const int ti = __popc(b0) + 2 * __popc(b1) + 4 * __popc(b2);
        if (ti == 0) continue;
        int p = __popc(b0 & lt) + 2 * __popc(b1 & lt) + 4 * __popc(b2 & lt);
        const int s = wb + 4 * (lane + 32 * i);
        const float vv[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if ((ci >> j) & 1u) o[p++] = (uint64_t(order_key(vv[j])) << 32) | uint32_t(s + j);
        o += ti;
      }
    }
  }
  // the last CTA of the row to get here selects
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(st + kStArrived, 1) == C - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int total = __ldcg(st + kStCursor);
  const int ovf = __ldcg(st + kStOverflow);
  if (ovf != 0 || total < a.K) {
    select_whole_row(a, w, hist, smw, out, phys);
  } else {
    // chunk records -> exclusive prefix of counts (record order = index order)
    const int nrec = C;
    int* s_pre = rec_smem;
    int* s_off = rec_smem + nrec + 1;
    int carry = 0;
    for (int r0 = 0; r0 < nrec; r0 += kTkThreads) {
      const int ri = r0 + tid;
      const int2 rec = ri < nrec
                           ? __ldcg(reinterpret_cast<const int2*>(a.chunkinfo + (size_t(w.r) * a.max_chunks + ri) * 2))
                           : make_int2(0, 0);
      int tot;
      const int cp = block_excl_scan<kTkThreads>(rec.y, &tot, smw) + carry;
      if (ri < nrec) {
        s_pre[ri] = cp;
        s_off[ri] = rec.x;
      }
      carry += tot;
    }
    if (tid == 0) s_pre[nrec] = carry;
    __syncthreads();
    // thread t: candidates t * 8 .. t * 8 + 7 of the ordered list
    const uint64_t* cand = a.cand + size_t(w.r) * kCandCap;
    const int p0 = tid * kCandPer;
    int ch = 0;
    if (p0 < total) {
      int lo = 0, hi = nrec - 1;  // last record with s_pre <= p0
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_pre[mid] <= p0) lo = mid; else hi = mid - 1;
      }
      ch = lo;
    }
    int src[kCandPer];
#pragma unroll
    for (int u = 0; u < kCandPer; ++u) {
      const int p = p0 + u;
      src[u] = -1;
      if (p < total) {
        while (s_pre[ch + 1] <= p) ++ch;
        src[u] = s_off[ch] + (p - s_pre[ch]);
      }
    }
    uint64_t cv[kCandPer];
#pragma unroll
    for (int u = 0; u < kCandPer; ++u) cv[u] = src[u] >= 0 ? __ldcg(cand + src[u]) : 0ull;
    uint32_t mk[kCandPer];
#pragma unroll
    for (int u = 0; u < kCandPer; ++u) mk[u] = uint32_t(cv[u] >> 32);
    const uint32_t tau = block_kth_key<kTkThreads, kCandPer>(mk, a.K, hist, smw);
    // one scan of (keys > tau, keys == tau) packed 16 | 16 bits: the tokens
    // selected before this thread are those above tau plus the first `need`
    // ties in index order
    int gt = 0, ne = 0;
#pragma unroll
    for (int u = 0; u < kCandPer; ++u) {
      gt += src[u] >= 0 && mk[u] > tau;
      ne += src[u] >= 0 && mk[u] == tau;
    }
    int t2;
    const int pk = block_excl_scan<kTkThreads>((gt << 16) | ne, &t2, smw);
    const int need = a.K - (t2 >> 16);
    int e = pk & 0xFFFF;
    int p = (pk >> 16) + min(e, need);
#pragma unroll
    for (int u = 0; u < kCandPer; ++u) {
      if (src[u] < 0) break;
      const bool sel = mk[u] > tau || (mk[u] == tau && e++ < need);
      if (sel) {
        const int s = int(uint32_t(cv[u]));
        if (p < a.K) {
          out[p] = s;
          if (phys) phys[p] = phys_row(a, w.b, s);
        }
        ++p;
      }
    }
  }
  // the row's state starts from zero at the next call
  __syncthreads();
  if (tid == 0) {
    st[kStCursor] = 0;
    st[kStOverflow] = 0;
    st[kStArrived] = 0;
  }
}

}  // namespace

// CTAs per row: about one wave over all rows, each filtering a chunk of a
// multiple of 1,024 tokens, at most kRoundTok (so at most cap / 1,024 = the
// row's max_chunks records, and at most 8,192 CTAs per row at the largest cap).
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
                        int32_t* topk_idx, int32_t* phys_rows, cudaStream_t st, bool have_gmax) {
  TopkArgs a;
  a.scores = scores;
  a.stride = score_stride;
  a.ctx_lens = ctx_lens;
  a.block_table = block_table;
  a.gmax = reinterpret_cast<const uint32_t*>(ws + L.gmax);
  a.gstride = L.gstride;
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
  cudaError_t e = cudaSuccess;
  if (!have_gmax) {
    const int gx = std::max(1, (L.cap + 16383) / 16384);  // two 1,024-token blocks per warp
    e = launch_pdl(topk_gmax_kernel, dim3(gx, L.rows), dim3(kGmaxThreads), 0, st, a,
                   reinterpret_cast<uint32_t*>(ws + L.gmax));
  }
  const TopkGrid tg = topk_grid(L);
  a.chunk = tg.chunk;
  const size_t smem = size_t(2 * tg.ctas + 1) * 4;
  if (e == cudaSuccess && smem > 48 * 1024)
    e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e == cudaSuccess)
    e = launch_pdl(topk_kernel, dim3(tg.ctas, L.rows), dim3(kTkThreads), smem, st, a);
  return e;
}

}  // namespace dsa
