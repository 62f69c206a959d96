// Stage 2: exact top-k over fp32 indexer scores.
//
// The article ("vLLM 为 Kimi K3.1 Pro 提供 Day-0 支持", "K3.1 Pro 中的稀疏注意力")
// keeps the 2,048 best-scoring tokens; this library fixes the order as (score
// descending, token index ascending) and writes the kept tokens in ascending
// index order.
//
// Method: radix select on the order-preserving 32-bit image of each score
// (11 + 11 + 10 bits), split over the context in chunks of kTopkChunk tokens.
//   pass 0..2  every chunk CTA histograms its tokens' next digit (among the
//              tokens that still match the prefix) into smem, then adds the
//              non-zero bins to the row's global histogram; the last CTA of the
//              row to finish (atomic ticket, no waiting) walks the histogram and
//              fixes the next digit of the threshold tau.
//   count      every chunk counts tokens above tau and equal to tau; the last
//              CTA turns the counts into per-chunk output offsets.
//   write      every chunk writes its selected tokens in index order (block
//              scans), ties at tau taken lowest index first.
// Counts do not depend on the order of atomics, so the result is deterministic.
#include "dsa_internal.cuh"

namespace dsa {

namespace {

constexpr int kThreads = 256;

struct TopkArgs {
  const float* scores;
  int64_t stride;
  const int32_t* ctx_lens;
  const int32_t* block_table;
  int n_q, cap, K, max_pages, num_pages, max_chunks;
  int* hist;      // [rows][5120]
  int* state;     // [rows][kRowState]
  int* ticket;    // [rows][4]
  int* chunkcnt;  // [rows][max_chunks][2]
  int* chunkoff;  // [rows][max_chunks][2]
  int* err;
  int32_t* topk_idx;
  int32_t* phys_rows;
};

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block scan (256 threads) of one int per thread; *total gets the sum.
__device__ __forceinline__ int block_excl_scan(int v, int* total, int* sm8) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm8[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < 8 ? sm8[lane] : 0;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < 8) sm8[lane] = s;
  }
  __syncthreads();
  const int pre = (warp ? sm8[warp - 1] : 0) + x - v;
  *total = sm8[7];
  __syncthreads();
  return pre;
}

// Find bin d (scanning from the top) holding the k-th largest (1-based) entry.
// Writes d and the count strictly above it to out[0], out[1] (shared memory).
__device__ void resolve_bin(const int* hist, int nbins, int k, int* out, int* sm8) {
  const int per = nbins / kThreads;
  const int hi = nbins - 1 - threadIdx.x * per;
  int s = 0;
  for (int j = 0; j < per; ++j) s += __ldcg(hist + hi - j);
  int tot;
  const int pre = block_excl_scan(s, &tot, sm8);
  if (pre < k && k <= pre + s) {
    int c = pre;
    for (int j = 0; j < per; ++j) {
      const int h = __ldcg(hist + hi - j);
      if (k <= c + h) {
        out[0] = hi - j;
        out[1] = c;
        break;
      }
      c += h;
    }
  }
  __syncthreads();
}

struct RowInfo {
  int r, b, L, nch, c;
};

__device__ __forceinline__ RowInfo row_info(const TopkArgs& a) {
  RowInfo ri;
  ri.r = blockIdx.y;
  ri.b = ri.r / a.n_q;
  const int t = ri.r - ri.b * a.n_q;
  const int ctx = a.ctx_lens[ri.b];
  ri.L = (ctx < a.n_q || ctx > a.cap) ? -1 : ctx - a.n_q + t + 1;
  if (ri.L > a.stride) ri.L = -1;
  ri.nch = ri.L > 0 ? (ri.L + kTopkChunk - 1) / kTopkChunk : 0;
  ri.c = blockIdx.x;
  return ri;
}

// The chunk's scores for this thread: 4 float4 loads (all issued before any
// use), element i*1024 + 4*tid + e of the chunk; `n[i]` valid lanes per load.
struct ChunkVals {
  float v[4][4];
  int n[4];
};

__device__ __forceinline__ void load_chunk(const float* row, int s0, int s1, ChunkVals& c) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int s = s0 + i * kThreads * 4 + threadIdx.x * 4;
    c.n[i] = min(4, max(0, s1 - s));
    if (c.n[i] == 4) {
      const float4 f = __ldcg(reinterpret_cast<const float4*>(row + s));
      c.v[i][0] = f.x; c.v[i][1] = f.y; c.v[i][2] = f.z; c.v[i][3] = f.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) c.v[i][e] = e < c.n[i] ? row[s + e] : 0.f;
    }
  }
}

// Histogram pass `pass` (0, 1, 2) of one chunk.
template <int PASS>
__global__ void __launch_bounds__(kThreads) topk_hist_kernel(TopkArgs a) {
  constexpr int NB = PASS == 2 ? kHist2Bins : 2048;
  __shared__ int sh[NB];
  __shared__ int sm8[8];
  __shared__ int res[2];
  __shared__ int last;
  const RowInfo ri = row_info(a);
  if (ri.L <= a.K || ri.c >= ri.nch) return;
  int* st = a.state + size_t(ri.r) * kRowState;
  uint32_t prefix = 0;
  if (PASS == 1) prefix = uint32_t(st[0]);
  if (PASS == 2) prefix = (uint32_t(st[0]) << 11) | uint32_t(st[2]);
  for (int i = threadIdx.x; i < NB; i += kThreads) sh[i] = 0;
  __syncthreads();
  const float* row = a.scores + size_t(ri.r) * a.stride;
  const int s0 = ri.c * kTopkChunk;
  const int s1 = min(ri.L, s0 + kTopkChunk);
  ChunkVals cv;
  load_chunk(row, s0, s1, cv);
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (e >= cv.n[i]) break;
      const uint32_t u = order_key(cv.v[i][e]);
      if (PASS == 0) atomicAdd(&sh[u >> 21], 1);
      if (PASS == 1 && (u >> 21) == prefix) atomicAdd(&sh[(u >> 10) & 2047u], 1);
      if (PASS == 2 && (u >> 10) == prefix) atomicAdd(&sh[u & 1023u], 1);
    }
  __syncthreads();
  int* gh = a.hist + size_t(ri.r) * (kHist0Bins + kHist1Bins + kHist2Bins) +
            (PASS == 0 ? 0 : PASS == 1 ? kHist0Bins : kHist0Bins + kHist1Bins);
  for (int i = threadIdx.x; i < NB; i += kThreads)
    if (sh[i]) atomicAdd(gh + i, sh[i]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(a.ticket + ri.r * 4 + PASS, 1) == ri.nch - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  const int k = PASS == 0 ? a.K : PASS == 1 ? st[1] : st[3];
  resolve_bin(gh, NB, k, res, sm8);
  if (threadIdx.x == 0) {
    if (PASS == 0) { st[0] = res[0]; st[1] = k - res[1]; }
    if (PASS == 1) { st[2] = res[0]; st[3] = k - res[1]; }
    if (PASS == 2) {
      st[4] = int((prefix << 10) | uint32_t(res[0]));  // tau (order key)
      st[5] = k - res[1];                               // ties at tau to take
    }
    a.ticket[ri.r * 4 + PASS] = 0;
  }
}

// Count tokens above / equal to tau per chunk; the last CTA scans the counts.
__global__ void __launch_bounds__(kThreads) topk_count_kernel(TopkArgs a) {
  __shared__ int sm8[8];
  __shared__ int last;
  const RowInfo ri = row_info(a);
  if (ri.L <= a.K || ri.c >= ri.nch) return;
  int* st = a.state + size_t(ri.r) * kRowState;
  const uint32_t tau = uint32_t(st[4]);
  const float* row = a.scores + size_t(ri.r) * a.stride;
  const int s0 = ri.c * kTopkChunk;
  const int s1 = min(ri.L, s0 + kTopkChunk);
  int gt = 0, eq = 0;
  ChunkVals cv;
  load_chunk(row, s0, s1, cv);
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (e >= cv.n[i]) break;
      const uint32_t u = order_key(cv.v[i][e]);
      gt += u > tau;
      eq += u == tau;
    }
  int tg, te;
  block_excl_scan(gt, &tg, sm8);
  block_excl_scan(eq, &te, sm8);
  int* cc = a.chunkcnt + (size_t(ri.r) * a.max_chunks + ri.c) * 2;
  if (threadIdx.x == 0) { cc[0] = tg; cc[1] = te; }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(a.ticket + ri.r * 4 + 3, 1) == ri.nch - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  const int need = st[5];
  int run_gt = 0, run_eq = 0;
  const int* ccr = a.chunkcnt + size_t(ri.r) * a.max_chunks * 2;
  int* cor = a.chunkoff + size_t(ri.r) * a.max_chunks * 2;
  for (int c0 = 0; c0 < ri.nch; c0 += kThreads) {
    const int c = c0 + threadIdx.x;
    const int g = c < ri.nch ? __ldcg(ccr + 2 * c) : 0;
    const int e = c < ri.nch ? __ldcg(ccr + 2 * c + 1) : 0;
    int sg, se;
    const int pg = block_excl_scan(g, &sg, sm8) + run_gt;
    const int pe = block_excl_scan(e, &se, sm8) + run_eq;
    if (c < ri.nch) {
      cor[2 * c] = pg + min(pe, need);  // selected tokens before chunk c
      cor[2 * c + 1] = pe;              // ties before chunk c
    }
    run_gt += sg;
    run_eq += se;
  }
  if (threadIdx.x == 0) a.ticket[ri.r * 4 + 3] = 0;
}

__device__ __forceinline__ int phys_row(const TopkArgs& a, int b, int s) {
  const int pg = a.block_table[size_t(b) * a.max_pages + s / kPage];
  if (pg < 0 || pg >= a.num_pages) {
    atomicOr(a.err, DSA_DEVERR_BLOCK_TABLE);
    return -1;
  }
  return pg * kPage + (s % kPage);
}

// Write the selected tokens of one chunk in index order.
__global__ void __launch_bounds__(kThreads) topk_write_kernel(TopkArgs a) {
  __shared__ int sm8[8];
  const RowInfo ri = row_info(a);
  int32_t* out = a.topk_idx + size_t(ri.r) * a.K;
  int32_t* phys = a.phys_rows ? a.phys_rows + size_t(ri.r) * a.K : nullptr;
  if (ri.L <= a.K) {
    // every visible token is kept (an invalid row keeps none)
    if (ri.c != 0) return;
    if (ri.L < 0 && threadIdx.x == 0) atomicOr(a.err, DSA_DEVERR_CTX);
    for (int i = threadIdx.x; i < a.K; i += kThreads) {
      const bool keep = i < ri.L;
      out[i] = keep ? i : -1;
      if (phys) phys[i] = keep ? phys_row(a, ri.b, i) : -1;
    }
    return;
  }
  if (ri.c >= ri.nch) return;
  const int* st = a.state + size_t(ri.r) * kRowState;
  const uint32_t tau = uint32_t(st[4]);
  const int need = st[5];
  const int* co = a.chunkoff + (size_t(ri.r) * a.max_chunks + ri.c) * 2;
  int pos = co[0];
  int eq_run = co[1];
  const float* row = a.scores + size_t(ri.r) * a.stride;
  const int s0 = ri.c * kTopkChunk;
  const int s1 = min(ri.L, s0 + kTopkChunk);
  ChunkVals cv;
  load_chunk(row, s0, s1, cv);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int s = s0 + i * kThreads * 4 + threadIdx.x * 4;
    const int n = cv.n[i];
    uint32_t u[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) u[e] = order_key(cv.v[i][e]);
    int ne = 0;
    for (int e = 0; e < n; ++e) ne += u[e] == tau;
    int te;
    int eq_pre = block_excl_scan(ne, &te, sm8) + eq_run;
    bool sel[4];
    int ns = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      sel[e] = false;
      if (e < n) {
        if (u[e] > tau) sel[e] = true;
        else if (u[e] == tau) sel[e] = (eq_pre++) < need;
      }
      ns += sel[e];
    }
    int ts;
    int p = block_excl_scan(ns, &ts, sm8) + pos;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (sel[e]) {
        if (p < a.K) {
          out[p] = s + e;
          if (phys) phys[p] = phys_row(a, ri.b, s + e);
        }
        ++p;
      }
    pos += ts;
    eq_run += te;
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
  a.hist = reinterpret_cast<int*>(ws + L.hist);
  a.state = reinterpret_cast<int*>(ws + L.state);
  a.ticket = reinterpret_cast<int*>(ws + L.ticket);
  a.chunkcnt = reinterpret_cast<int*>(ws + L.chunkcnt);
  a.chunkoff = reinterpret_cast<int*>(ws + L.chunkoff);
  a.err = reinterpret_cast<int*>(ws + L.err);
  a.topk_idx = topk_idx;
  a.phys_rows = phys_rows;
  // histograms and tickets start at zero for every call
  cudaError_t e = cudaMemsetAsync(ws + L.hist, 0, L.ticket + size_t(L.rows) * 16 - L.hist, st);
  if (e != cudaSuccess) return e;
  dim3 grid(L.max_chunks, L.rows);
  topk_hist_kernel<0><<<grid, kThreads, 0, st>>>(a);
  topk_hist_kernel<1><<<grid, kThreads, 0, st>>>(a);
  topk_hist_kernel<2><<<grid, kThreads, 0, st>>>(a);
  topk_count_kernel<<<grid, kThreads, 0, st>>>(a);
  topk_write_kernel<<<grid, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace dsa
