// Stage 2: exact top-k over fp32 indexer scores.
//
// The article ("vLLM 为 Kimi K3.1 Pro 提供 Day-0 支持", "K3.1 Pro 中的稀疏注意力")
// keeps the 2,048 best-scoring tokens; this library fixes the order as (score
// descending, token index ascending) and writes the kept tokens in ascending
// index order.
//
// Scores are compared through an order-preserving 32-bit key (larger score ->
// larger key; -0 and +0 share one key). Three kernels:
//   sample  one cluster of 8 CTAs per row: the 8,192 threads read <= 8,192
//           evenly spaced scores (one each, so no SM issues more than 1,024
//           scattered reads) into the first CTA's shared memory, which picks a
//           key g that about 2K tokens of the row are expected to reach
//   filter  one CTA per 4,096-token chunk: compact the chunk's tokens with
//           key >= g, in index order, into the row's candidate buffer (a
//           region reserved with one atomic; its place recorded per chunk)
//   select  one CTA per row: gather the candidates chunk by chunk (so they are
//           in index order again), radix-select the exact K-th largest key tau
//           among them and write the winners in order, ties at tau lowest
//           index first.
// Whenever at least K tokens reach g, the candidates contain every token with
// key >= tau, so the selection is exact. Otherwise (g too high, or more
// candidates than the buffer holds, e.g. a row of equal scores) the select CTA
// runs an exact radix select over the whole row by itself. No CTA ever waits
// on another; the result does not depend on the order of the atomics.
#include "block_select.cuh"
#include "dsa_internal.cuh"
#include "sm103_ptx.cuh"

namespace dsa {

namespace {

constexpr int kFiltThreads = 256;
constexpr int kSelThreads = 1024;
constexpr int kSampleMax = 8192;

struct TopkArgs {
  const float* scores;
  int64_t stride;
  const int32_t* ctx_lens;
  const int32_t* block_table;
  int n_q, cap, K, max_pages, num_pages, max_chunks;
  int* state;      // [rows][kRowState]: 0 g, 1 cursor, 2 overflow
  int* chunkinfo;  // [rows][max_chunks][2]: (offset, count) in the candidate buffer
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

// ---------------------------------------------------------------- sample
constexpr int kSampleThreads = 1024;
constexpr int kSampleCluster = 8;
constexpr int kSamplePer = kSampleMax / kSampleThreads;  // 8 samples per thread of the first CTA
constexpr size_t kSampleSmem = size_t(kSampleMax) * 4 + 4096 * 4;

__global__ void __cluster_dims__(kSampleCluster, 1, 1) __launch_bounds__(kSampleThreads, 1)
    topk_sample_kernel(TopkArgs a) {
  extern __shared__ uint32_t sample_smem[];
  uint32_t* sk = sample_smem;                                  // [8192] sample keys (first CTA)
  int* hist = reinterpret_cast<int*>(sample_smem + kSampleMax);  // [4096]
  __shared__ int smw[64];
  pdl_wait();
  ptx::cluster_sync();  // every CTA of the cluster runs before any remote store
  const uint32_t rank = ptx::cluster_ctarank();
  const Row w = row_of(a, blockIdx.y);
  if (w.L <= a.K) return;  // the whole cluster (one row) returns
  const int ns = min(w.L, kSampleMax);
  // sample i = rank * 1024 + t at evenly spaced positions (any fixed spread
  // serves: g only has to be a good guess)
  {
    const int i = int(rank) * kSampleThreads + threadIdx.x;
    const float step = float(w.L) / float(ns);
    const float* row = a.scores + size_t(w.r) * a.stride;
    const uint32_t key = i < ns ? order_key(__ldcg(row + min(w.L - 1, int(float(i) * step)))) : 0u;
    ptx::st_cluster_u32(ptx::mapa_shared(ptx::smem_u32(sk + i), 0), key);
  }
  ptx::cluster_sync();  // the first CTA holds every sample
  if (rank != 0) return;
  uint32_t keys[kSamplePer];
#pragma unroll
  for (int u = 0; u < kSamplePer; ++u) keys[u] = sk[threadIdx.x * kSamplePer + u];
  // the r-th largest sample: about 2K tokens of the row are expected at or above it.
  // For small r the r-th largest of the threads' maxima (8 samples each) serves:
  // the top r samples almost always sit in r different threads, and a slightly
  // lower g only adds candidates.
  const int r = int((int64_t(2) * a.K * ns + w.L - 1) / w.L);
  uint32_t g = 0u;
  if (r <= 64) {
    uint32_t m[1] = {0u};
#pragma unroll
    for (int u = 0; u < kSamplePer; ++u) m[0] = max(m[0], keys[u]);
    g = block_kth_key<kSampleThreads, 1>(m, r, hist, smw);
  } else if (r < ns) {
    g = block_kth_key<kSampleThreads, kSamplePer>(keys, r, hist, smw);
  }
  int* st = a.state + size_t(w.r) * kRowState;
  if (threadIdx.x == 0) {
    st[0] = int(g);
    st[1] = 0;  // candidate cursor
    st[2] = 0;  // overflow
  }
}

// ---------------------------------------------------------------- filter
__global__ void __launch_bounds__(kFiltThreads) topk_filter_kernel(TopkArgs a) {
  pdl_wait();
  __shared__ int smw[8];
  __shared__ int s_base;
  const Row w = row_of(a, blockIdx.y);
  if (w.L <= a.K) return;
  const int nch = (w.L + kTopkChunk - 1) / kTopkChunk;
  const int c = blockIdx.x;
  if (c >= nch) return;
  int* st = a.state + size_t(w.r) * kRowState;
  const uint32_t g = uint32_t(st[0]);
  const float* row = a.scores + size_t(w.r) * a.stride;
  // thread t holds tokens s0 + 16t .. s0 + 16t + 15 (all loads issued first)
  const int s = c * kTopkChunk + threadIdx.x * 16;
  const int n = min(16, max(0, w.L - s));
  float v[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (4 * i + 4 <= n) {
      const float4 f = __ldcg(reinterpret_cast<const float4*>(row + s + 4 * i));
      v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) v[4 * i + e] = 4 * i + e < n ? row[s + 4 * i + e] : 0.f;
    }
  }
  uint32_t keep = 0;
  int m = 0;
#pragma unroll
  for (int e = 0; e < 16; ++e)
    if (e < n && order_key(v[e]) >= g) { keep |= 1u << e; ++m; }
  int run;
  const int pre = block_excl_scan<kFiltThreads>(m, &run, smw);
  if (threadIdx.x == 0) {
    const int base = atomicAdd(st + 1, run);
    if (base + run > kCandCap) atomicOr(st + 2, 1);
    s_base = base;
    int* ci = a.chunkinfo + (size_t(w.r) * a.max_chunks + c) * 2;
    ci[0] = base;
    ci[1] = run;
  }
  __syncthreads();
  const int base = s_base;
  if (base + run > kCandCap) return;
  uint64_t* out = a.cand + size_t(w.r) * kCandCap + base + pre;
  int p = 0;
#pragma unroll
  for (int e = 0; e < 16; ++e)
    if (keep & (1u << e)) out[p++] = (uint64_t(order_key(v[e])) << 32) | uint32_t(s + e);
}

// ---------------------------------------------------------------- select
// Exact radix select over the whole row by this CTA alone (the rare path):
// 11 + 11 + 10 key bits, then an ordered write in tiles of kSelThreads tokens.
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
    for (int i = threadIdx.x; i < nb; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    const uint32_t pre = s_prefix;
    const uint32_t hmask = pass == 0 ? 0u : (0xFFFFFFFFu << (sh + width));
    for (int s = threadIdx.x; s < w.L; s += kSelThreads) {
      const uint32_t u = order_key(__ldcg(row + s));
      if ((u & hmask) == pre) atomicAdd(&hist[(u >> sh) & uint32_t(nb - 1)], 1);
    }
    __syncthreads();
    // bins from the top; thread t owns bins nb-1-t*per .. nb-per-t*per
    const int per = nb / kSelThreads;
    int cnt = 0;
    for (int j = 0; j < per; ++j) cnt += hist[nb - 1 - threadIdx.x * per - j];
    int tot;
    const int before = block_excl_scan<kSelThreads>(cnt, &tot, smw);
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
  int pos = 0, eq_run = 0;
  for (int base = 0; base < w.L; base += kSelThreads) {
    const int s = base + threadIdx.x;
    const uint32_t u = s < w.L ? order_key(__ldcg(row + s)) : 0u;
    const int is_eq = (s < w.L && u == tau) ? 1 : 0;
    int te;
    const int eq_pre = block_excl_scan<kSelThreads>(is_eq, &te, smw) + eq_run;
    const int sel = (s < w.L && (u > tau || (is_eq && eq_pre < need))) ? 1 : 0;
    int ts;
    const int p = block_excl_scan<kSelThreads>(sel, &ts, smw) + pos;
    if (sel && p < a.K) {
      out[p] = s;
      if (phys) phys[p] = phys_row(a, w.b, s);
    }
    pos += ts;
    eq_run += te;
  }
}

constexpr size_t kSelSmem = size_t(kCandCap) * 8 + 4096 * 4;

__global__ void __launch_bounds__(kSelThreads, 1) topk_select_kernel(TopkArgs a) {
  pdl_wait();
  extern __shared__ uint32_t sel_smem[];
  uint32_t* ckey = sel_smem;                                  // [kCandCap]
  int* cidx = reinterpret_cast<int*>(sel_smem + kCandCap);    // [kCandCap]
  int* hist = cidx + kCandCap;                                // [4096]
  __shared__ int smw[64];
  const Row w = row_of(a, blockIdx.x);
  int32_t* out = a.topk_idx + size_t(w.r) * a.K;
  int32_t* phys = a.phys_rows ? a.phys_rows + size_t(w.r) * a.K : nullptr;
  if (w.L <= a.K) {
    // every visible token is kept (an invalid row keeps none)
    if (w.L < 0 && threadIdx.x == 0) atomicOr(a.err, DSA_DEVERR_CTX);
    for (int i = threadIdx.x; i < a.K; i += kSelThreads) {
      const bool keep = i < w.L;
      out[i] = keep ? i : -1;
      if (phys) phys[i] = keep ? phys_row(a, w.b, i) : -1;
    }
    return;
  }
  // the row state and the first window of chunk records are loaded together
  const int nch = (w.L + kTopkChunk - 1) / kTopkChunk;
  const int* ci = a.chunkinfo + size_t(w.r) * a.max_chunks * 2;
  const int2 rec0 = int(threadIdx.x) < nch ? *reinterpret_cast<const int2*>(ci + 2 * threadIdx.x) : make_int2(0, 0);
  const int* st = a.state + size_t(w.r) * kRowState;
  const int total = st[1];
  if (st[2] != 0 || total < a.K) {
    select_whole_row(a, w, hist, smw, out, phys);
    return;
  }
  // gather the candidates chunk by chunk (index order again): chunks in
  // windows of 1024; positions spread over all threads, each finds its chunk
  // by binary search over the window's offsets
  const uint64_t* cand = a.cand + size_t(w.r) * kCandCap;
  int* wpre = hist;          // [1024] window prefix of counts
  int* wsrc = hist + 1024;   // [1024] source offsets
  int done = 0;
  for (int c0 = 0; c0 < nch; c0 += kSelThreads) {
    const int c = c0 + threadIdx.x;
    const int2 rec = c0 == 0 ? rec0 : (c < nch ? *reinterpret_cast<const int2*>(ci + 2 * c) : make_int2(0, 0));
    int tot;
    const int pre = block_excl_scan<kSelThreads>(rec.y, &tot, smw);
    wpre[threadIdx.x] = pre;
    wsrc[threadIdx.x] = rec.x;
    __syncthreads();
    const int nw = min(kSelThreads, nch - c0);
    // every position's source first, then all loads in flight at once
    // (tot <= kCandCap: at most kCandCap / kSelThreads positions per thread)
    constexpr int kPos = kCandCap / kSelThreads;
    int srcs[kPos];
#pragma unroll
    for (int u = 0; u < kPos; ++u) {
      const int pos = threadIdx.x + u * kSelThreads;
      srcs[u] = -1;
      if (pos < tot) {
        int lo = 0, hi = nw - 1;  // last chunk with wpre <= pos
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (wpre[mid] <= pos) lo = mid; else hi = mid - 1;
        }
        srcs[u] = wsrc[lo] + (pos - wpre[lo]);
      }
    }
    uint64_t vals[kPos];
#pragma unroll
    for (int u = 0; u < kPos; ++u) vals[u] = srcs[u] >= 0 ? cand[srcs[u]] : 0ull;
#pragma unroll
    for (int u = 0; u < kPos; ++u) {
      const int pos = threadIdx.x + u * kSelThreads;
      if (srcs[u] >= 0) {
        ckey[done + pos] = uint32_t(vals[u] >> 32);
        cidx[done + pos] = int(uint32_t(vals[u]));
      }
    }
    done += tot;
    __syncthreads();
  }
  // exact K-th largest candidate key and the ties at it to take
  constexpr int kSelPer = kCandCap / kSelThreads;  // 8
  uint32_t mk[kSelPer];
#pragma unroll
  for (int u = 0; u < kSelPer; ++u) {
    const int i = threadIdx.x * kSelPer + u;
    mk[u] = i < total ? ckey[i] : 0u;
  }
  const uint32_t tau = block_kth_key<kSelThreads, kSelPer>(mk, a.K, hist, smw);
  // one scan of (keys > tau, keys == tau) packed 16 | 16 bits: the tokens
  // selected before this thread are those above tau plus the first `need`
  // ties in index order
  int gt = 0, ne = 0;
#pragma unroll
  for (int u = 0; u < kSelPer; ++u) {
    const bool valid = threadIdx.x * kSelPer + u < total;
    gt += valid && mk[u] > tau;
    ne += valid && mk[u] == tau;
  }
  int tot;
  const int pre = block_excl_scan<kSelThreads>((gt << 16) | ne, &tot, smw);
  const int need = a.K - (tot >> 16);
  int e = pre & 0xFFFF;
  int p = (pre >> 16) + min(e, need);
  // ordered write: thread t takes candidates t*8 .. t*8+7
#pragma unroll
  for (int u = 0; u < kSelPer; ++u) {
    const int i = threadIdx.x * kSelPer + u;
    if (i >= total) break;
    const bool sel = mk[u] > tau || (mk[u] == tau && e++ < need);
    if (sel) {
      if (p < a.K) {
        out[p] = cidx[i];
        if (phys) phys[p] = phys_row(a, w.b, cidx[i]);
      }
      ++p;
    }
  }
}

}  // namespace

cudaError_t launch_topk(const dsa_params_t& p, const WsLayout& L, char* ws, const float* scores,
                        int64_t score_stride, const int32_t* ctx_lens, const int32_t* block_table,
                        int32_t* topk_idx, int32_t* phys_rows, cudaStream_t st) {
  TopkArgs a;
  a.scores = scores;
  a.stride = score_stride;
  a.ctx_lens = ctx_lens;
  a.block_table = block_table;
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
  cudaError_t e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSelSmem));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(topk_sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSampleSmem));
  if (e == cudaSuccess)
    e = launch_pdl(topk_sample_kernel, dim3(kSampleCluster, L.rows), dim3(kSampleThreads), kSampleSmem, st, a);
  if (e == cudaSuccess)
    e = launch_pdl(topk_filter_kernel, dim3(L.max_chunks, L.rows), dim3(kFiltThreads), 0, st, a);
  if (e == cudaSuccess) e = launch_pdl(topk_select_kernel, dim3(L.rows), dim3(kSelThreads), kSelSmem, st, a);
  return e;
}

}  // namespace dsa
