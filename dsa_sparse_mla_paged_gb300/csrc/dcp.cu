// Decode context parallelism, emulated on one GPU: the exact top-k merge of W
// token shards ("vLLM 为 Kimi K3.1 Pro 提供 Day-0 支持", section "长上下文：带稀疏
// indexer 的 decode 上下文并行", "流量减少 10× 的精确 top-k 合并").
//
// Shard r of a row holds tokens s with s mod W == r. Three kernels:
//   keys   the bf16 keys of every shard's tokens, gathered shard by shard
//   shard  one CTA per (shard, row): the shard's first min(K, L_r) tokens in
//          the shard's order (bf16 score key desc, token asc), as the lists a
//          GPU would keep (key, token) by position
//   merge  one CTA per row: the first exchange packs each shard's first m = ceil(1.5 K / W)
//          candidates (at most K) into 32-bit words (key16 << 16 |
//          (4095 - position) << 4 | (15 - shard)), radix-selects the K largest,
//          and finds the shards whose m candidates were all selected while they
//          hold more among their first K; those send their first K and a second
//          exchange selects again. The winners are written in ascending token order,
//          with the re-sent shard mask and the words exchanged.
// Then a fourth kernel, the cross-shard LSE combine of the shards' partial
// attention outputs (same section: each GPU attends over its own winners,
// then the partials are merged by their log-sum-exp).
#include <cuda_bf16.h>

#include "block_select.cuh"
#include "dsa_internal.cuh"
#include "sm103_ptx.cuh"

namespace dsa {

namespace {

constexpr int kDcpThreads = 1024;
constexpr int kTieCap = 4096;  // ties at the shard threshold gathered and sorted in shared memory

struct DcpArgs {
  const float* scores;
  int64_t stride;
  const int32_t* ctx_lens;
  int n_q, cap, K, W, m;
  int64_t S;        // shard row of keys16, in keys (multiple of 8)
  uint16_t* keys16; // [rows][W][S] key16 by shard position
  uint32_t* lkey;   // [rows][kDcpMaxWorld][K] key16 by position
  int32_t* ltok;    // [rows][kDcpMaxWorld][K] token by position
  int32_t* lcount;  // [rows][kDcpMaxWorld]
  int32_t* topk_idx;
  int32_t* stats;   // [rows][2] or null: re-sent shard mask, words exchanged
  int* err;
};

// Visible length of a row, or 0 (and the error bit) for an invalid context.
__device__ __forceinline__ int dcp_row_len(const DcpArgs& a, int row, bool report) {
  const int b = row / a.n_q, t = row - b * a.n_q;
  const int ctx = a.ctx_lens[b];
  if (ctx < a.n_q || ctx > a.cap || ctx - a.n_q + t + 1 > a.stride) {
    if (report && threadIdx.x == 0) atomicOr(a.err, DSA_DEVERR_CTX);
    return 0;
  }
  return ctx - a.n_q + t + 1;
}

// 16-bit order key of the bf16 rounding (nearest even) of an fp32 score.
__device__ __forceinline__ uint32_t bf16_order_key(float f) {
  const uint64_t u = __float_as_uint(f);
  uint32_t b = uint32_t((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16) & 0xFFFFu;
  if (b == 0x8000u) b = 0u;
  return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
}

// Ascending bitonic sort of the 2048 keys v[0 .. 2048) (32- or 64-bit) by
// the CTA's 1024 threads, the network unrolled at compile time. Thread t holds
// elements 2t and 2t + 1 in registers; a partner in the same warp (stride < 64)
// is read by shuffle, any other through shared memory (15 of the 66 steps).
// v must be written and synchronised before the call; it holds the sorted keys
// after.
template <typename T>
__device__ __forceinline__ void sort2048(T* v) {
  static_assert(kDcpThreads == 1024, "two keys per thread");
  const int e0 = 2 * int(threadIdx.x);
  T x0 = v[e0], x1 = v[e0 + 1];
#pragma unroll
  for (int size = 2; size <= 2048; size <<= 1) {
    const bool up = (e0 & size) == 0;
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride == 1) {
        const T lo = x0 < x1 ? x0 : x1, hi = x0 < x1 ? x1 : x0;
        x0 = up ? lo : hi;
        x1 = up ? hi : lo;
      } else {
        T y0, y1;
        if (stride < 64) {
          y0 = __shfl_xor_sync(0xffffffffu, x0, stride >> 1);
          y1 = __shfl_xor_sync(0xffffffffu, x1, stride >> 1);
        } else {
          __syncthreads();  // the previous exchange has been read
          v[e0] = x0;
          v[e0 + 1] = x1;
          __syncthreads();
          y0 = v[e0 ^ stride];
          y1 = v[(e0 ^ stride) + 1];
        }
        const bool keep_min = ((e0 & stride) == 0) == up;
        x0 = keep_min ? (x0 < y0 ? x0 : y0) : (x0 < y0 ? y0 : x0);
        x1 = keep_min ? (x1 < y1 ? x1 : y1) : (x1 < y1 ? y1 : x1);
      }
    }
  }
  __syncthreads();
  v[e0] = x0;
  v[e0 + 1] = x1;
  __syncthreads();
}

__device__ __forceinline__ int pow2_at_least(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

// ---------------------------------------------------------------- shard keys
// What each shard's GPU would hold: the 16-bit keys of its tokens, contiguous
// (keys16[row][r][i] = key of token r + i * W). One coalesced pass over the
// scores, so the shard kernels below read their own tokens densely.
constexpr int kKeysThreads = 256;

__global__ void __launch_bounds__(kKeysThreads) dcp_keys_kernel(DcpArgs a) {
  pdl_wait();
  const int row = blockIdx.y;
  const int L = dcp_row_len(a, row, false);
  const int t0 = (blockIdx.x * kKeysThreads + int(threadIdx.x)) * 4;
  if (t0 >= L) return;
  // t0 + 3 < score_stride: t0 < L <= stride, both t0 and stride multiples of 4
  const float4 f = __ldcg(reinterpret_cast<const float4*>(a.scores + size_t(row) * a.stride + t0));
  const float v[4] = {f.x, f.y, f.z, f.w};
  uint16_t* base = a.keys16 + size_t(row) * a.W * a.S;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int t = t0 + e;
    if (t < L) base[size_t(t % a.W) * a.S + t / a.W] = uint16_t(bf16_order_key(v[e]));
  }
}

// ---------------------------------------------------------------- shard lists
constexpr uint32_t kNoKey = 0x10000u;  // a position past the shard's end

// Keys of shard positions [8v, 8v + 8); positions >= Lr read as kNoKey. The
// 16-byte load stays inside the shard's row: S is a multiple of 8 and 8v < Lr <= S.
__device__ __forceinline__ void keys8(const uint16_t* src, int v, int Lr, uint32_t (&k)[8]) {
  uint4 q = make_uint4(0u, 0u, 0u, 0u);
  if (8 * v < Lr) q = __ldcg(reinterpret_cast<const uint4*>(src) + v);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int e = 0; e < 8; ++e) k[e] = (8 * v + e < Lr) ? ((w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu) : kNoKey;
}

// The bin of a kHiBins-bin histogram that holds the kk-th largest key, and the
// number of keys in the bins above it (1 <= kk <= keys counted). Thread t owns
// the two bins 2047 - 2t and 2046 - 2t; one scan of the per-thread sums finds
// the owner, which walks its bins.
constexpr int kHiBits = 11, kHiBins = 1 << kHiBits, kLoBits = 16 - kHiBits;
static_assert(kHiBins == 2 * kDcpThreads, "two bins per thread");

__device__ __forceinline__ int2 top_bin(const int* H, int kk, int* smw, int* s_out) {
  const int top = kHiBins - 1 - 2 * int(threadIdx.x);
  const int c0 = H[top], c1 = H[top - 1];
  int tot;
  const int before = block_excl_scan<kDcpThreads>(c0 + c1, &tot, smw);
  if (before < kk && kk <= before + c0 + c1) {
    if (kk <= before + c0) { s_out[0] = top; s_out[1] = before; }
    else { s_out[0] = top - 1; s_out[1] = before + c0; }
  }
  __syncthreads();
  return make_int2(s_out[0], s_out[1]);
}

// Distributed shared memory of the shard cluster (addresses from mapa).
__device__ __forceinline__ uint32_t dsm_ld_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void dsm_st_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void dsm_st_u64(uint32_t addr, uint64_t v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ uint32_t dsm_atom_add(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void dsm_red_add(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

constexpr int kShardCluster = 4;  // CTAs per (row, shard)

// The n-th largest key16 of the shard (an 11-bit and a 5-bit histogram pass:
// 11 bits spread the keys over enough bins that the shared atomics rarely
// collide), then the tokens above it and the lowest-token ties at it, sorted
// into the shard order. A cluster of kShardCluster CTAs shares the shard's
// positions: each counts its quarter into its own histogram and adds it into
// the first CTA's, which picks the bins; the tokens found go to the first
// CTA's list, which sorts and writes it.
__global__ void __cluster_dims__(kShardCluster, 1, 1) __launch_bounds__(kDcpThreads, 1)
    dcp_shard_kernel(DcpArgs a) {
  pdl_wait();
  __shared__ int hist[kHiBins];     // this CTA's counts
  __shared__ int hsum[kHiBins];     // first CTA: the cluster's pass-1 counts
  __shared__ int hsum2[1 << kLoBits];  // first CTA: the cluster's pass-2 counts
  __shared__ int s_sel[4];          // first CTA: high bin, count above it, threshold key, ties wanted
  __shared__ int s_n[3];            // first CTA: list fill, tie fill, ties at the threshold
  __shared__ int smw[64];
  extern __shared__ uint64_t dcp_smem[];
  uint64_t* list = dcp_smem;                                   // first CTA: [2048] (0xFFFF - key) << 32 | token
  uint32_t* ties = reinterpret_cast<uint32_t*>(list + kMaxTopK);  // first CTA: [kTieCap] tokens at the threshold
  const uint32_t q = ptx::cluster_ctarank();
  const int r = blockIdx.x / kShardCluster, row = blockIdx.y;
  const int L = dcp_row_len(a, row, false);
  const int Lr = L > r ? (L - 1 - r) / a.W + 1 : 0;
  const int n = min(a.K, Lr);
  int32_t* cnt_out = a.lcount + size_t(row) * kDcpMaxWorld + r;
  if (n == 0) {  // the whole cluster
    if (q == 0 && threadIdx.x == 0) *cnt_out = 0;
    return;
  }
  const uint16_t* src = a.keys16 + (size_t(row) * a.W + r) * a.S;
  const int nv = (Lr + 7) / 8;
  const int per = (nv + kShardCluster - 1) / kShardCluster;
  const int v0 = int(q) * per, v1 = min(nv, v0 + per);  // this CTA's vectors of 8 positions
  const auto first = [](const void* p) { return ptx::mapa_shared(ptx::smem_u32(p), 0); };
  uint32_t k[8];
  for (int i = threadIdx.x; i < kHiBins; i += kDcpThreads) {
    hist[i] = 0;
    hsum[i] = 0;
  }
  if (threadIdx.x < (1 << kLoBits)) hsum2[threadIdx.x] = 0;
  ptx::cluster_sync();  // every CTA runs and the first CTA's sums are zero
  // pass 1: the high 11 bits
  for (int v = v0 + int(threadIdx.x); v < v1; v += kDcpThreads) {
    keys8(src, v, Lr, k);
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (k[e] != kNoKey) atomicAdd(&hist[k[e] >> kLoBits], 1);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kHiBins; i += kDcpThreads) {
    if (hist[i]) dsm_red_add(first(&hsum[i]), uint32_t(hist[i]));
    hist[i] = 0;
  }
  ptx::cluster_sync();  // the first CTA holds the cluster's counts
  if (q == 0) top_bin(hsum, n, smw, s_sel);
  ptx::cluster_sync();
  const uint32_t hb = dsm_ld_u32(first(&s_sel[0]));
  const int above_hb = int(dsm_ld_u32(first(&s_sel[1])));
  // pass 2: the low 5 bits within that bin
  for (int v = v0 + int(threadIdx.x); v < v1; v += kDcpThreads) {
    keys8(src, v, Lr, k);
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (k[e] != kNoKey && (k[e] >> kLoBits) == hb) atomicAdd(&hist[k[e] & ((1u << kLoBits) - 1)], 1);
  }
  __syncthreads();
  if (threadIdx.x < (1 << kLoBits) && hist[threadIdx.x])
    dsm_red_add(first(&hsum2[threadIdx.x]), uint32_t(hist[threadIdx.x]));
  ptx::cluster_sync();
  if (q == 0 && threadIdx.x == 0) {
    int above = above_hb, l = (1 << kLoBits) - 1;
    for (; l > 0; --l) {
      if (above + hsum2[l] >= n) break;
      above += hsum2[l];
    }
    s_sel[2] = int((hb << kLoBits) | uint32_t(l));
    s_sel[3] = n - above;  // ties at the threshold to take (lowest tokens first)
    s_n[0] = 0;
    s_n[1] = 0;
    s_n[2] = hsum2[l];
  }
  ptx::cluster_sync();
  const uint32_t tau = dsm_ld_u32(first(&s_sel[2]));
  const int n_ties = int(dsm_ld_u32(first(&s_n[2])));
  // pass 3: tokens above the threshold, and the ties (all of them when they fit), into the first CTA
  {
    const uint32_t list0 = first(list), ties0 = first(ties), nl0 = first(&s_n[0]), nt0 = first(&s_n[1]);
    for (int v = v0 + int(threadIdx.x); v < v1; v += kDcpThreads) {
      keys8(src, v, Lr, k);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t tok = uint32_t(r + (8 * v + e) * a.W);
        if (k[e] != kNoKey && k[e] > tau) {
          const uint32_t at = dsm_atom_add(nl0, 1u);
          dsm_st_u64(list0 + 8u * at, (uint64_t(0xFFFFu - k[e]) << 32) | tok);
        } else if (k[e] == tau && n_ties <= kTieCap) {
          const uint32_t at = dsm_atom_add(nt0, 1u);
          dsm_st_u32(ties0 + 4u * at, tok);
        }
      }
    }
  }
  ptx::cluster_sync();  // the first CTA holds every token found
  if (q != 0) return;
  const int need = s_sel[3];
  const int n_gt = s_n[0];
  if (n_ties <= kTieCap) {
    // lowest `need` tokens among the ties
    const int p = pow2_at_least(n_ties);
    for (int i = n_ties + threadIdx.x; i < p; i += kDcpThreads) ties[i] = 0xFFFFFFFFu;
    __syncthreads();
    // ascending 32-bit bitonic sort of the tie tokens in place
    for (int size = 2; size <= p; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = threadIdx.x; i < (p >> 1); i += kDcpThreads) {
          const int lo = 2 * i - (i & (stride - 1));
          const int hi = lo + stride;
          const bool up = (lo & size) == 0;
          const uint32_t x = ties[lo], y = ties[hi];
          if ((x > y) == up) { ties[lo] = y; ties[hi] = x; }
        }
        __syncthreads();
      }
    }
    for (int i = threadIdx.x; i < need; i += kDcpThreads)
      list[n_gt + i] = (uint64_t(0xFFFFu - tau) << 32) | ties[i];
  } else {
    // many equal keys: the ties in position (= token) order, 8 positions per
    // thread, chunk by chunk
    int taken = 0;
    for (int v0 = 0; v0 < nv && taken < need; v0 += kDcpThreads) {
      const int v = v0 + int(threadIdx.x);
      keys8(src, v, Lr, k);
      int mine = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) mine += k[e] == tau ? 1 : 0;
      int tot;
      int at = taken + block_excl_scan<kDcpThreads>(mine, &tot, smw);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (k[e] == tau) {
          if (at < need) list[n_gt + at] = (uint64_t(0xFFFFu - tau) << 32) | uint32_t(r + (8 * v + e) * a.W);
          ++at;
        }
      taken += tot;
    }
  }
  __syncthreads();
  // the shard order: key desc, token asc
  for (int i = n + threadIdx.x; i < kMaxTopK; i += kDcpThreads) list[i] = ~0ull;
  __syncthreads();
  sort2048<uint64_t>(list);
  uint32_t* kout = a.lkey + (size_t(row) * kDcpMaxWorld + r) * a.K;
  int32_t* tout = a.ltok + (size_t(row) * kDcpMaxWorld + r) * a.K;
  for (int j = threadIdx.x; j < n; j += kDcpThreads) {
    kout[j] = 0xFFFFu - uint32_t(list[j] >> 32);
    tout[j] = int32_t(uint32_t(list[j]));
  }
  if (threadIdx.x == 0) *cnt_out = n;
}

// ---------------------------------------------------------------- merge
// Candidate c of an exchange (shard lists laid end to end, `cnt` per shard) -> word.
template <int PER>
__device__ __forceinline__ void exchange_words(const DcpArgs& a, int row, const int* cnt, const int* off, int total,
                                            uint32_t (&words)[PER]) {
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int c = threadIdx.x + u * kDcpThreads;
    words[u] = 0u;
    if (c < total) {
      int r = 0;
      while (r + 1 < a.W && off[r + 1] <= c) ++r;
      const int j = c - off[r];
      const uint32_t key = a.lkey[(size_t(row) * kDcpMaxWorld + r) * a.K + j];
      words[u] = (key << 16) | (uint32_t(4095 - j) << 4) | uint32_t(15 - r);
    }
  }
}

// One exchange's selection bookkeeping. The selected words are the ones >= tau.
// A shard's words fall with its position, so its selected words are a prefix
// of its candidates; sel[r] is that prefix's length, found by the one selected
// candidate whose successor (same shard) is not selected. The winners' tokens
// go to win[] in candidate order (block scan, no contended atomics).
template <int PER>
__device__ __forceinline__ void take_exchange(const DcpArgs& a, int row, const uint32_t (&wd)[PER], uint32_t tau,
                                           const int* off, uint32_t* selbits, int* sel, uint32_t* win, int* smw,
                                           bool collect) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int mine = 0;
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const bool s_ = wd[u] != 0u && wd[u] >= tau;
    const unsigned b = __ballot_sync(0xffffffffu, s_);
    if (lane == 0) selbits[u * (kDcpThreads / 32) + warp] = b;
    mine += s_ ? 1 : 0;
  }
  __syncthreads();
  int tot;
  int at = block_excl_scan<kDcpThreads>(mine, &tot, smw);
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    if (wd[u] != 0u && wd[u] >= tau) {
      const int c = int(threadIdx.x) + u * kDcpThreads;
      const int r = 15 - int(wd[u] & 15u), j = 4095 - int((wd[u] >> 4) & 4095u);
      const int nx = c + 1;
      if (nx >= off[r + 1] || !((selbits[nx >> 5] >> (nx & 31)) & 1u)) sel[r] = j + 1;
      if (collect) win[at++] = uint32_t(a.ltok[(size_t(row) * kDcpMaxWorld + r) * a.K + j]);
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kDcpThreads, 1) dcp_merge_kernel(DcpArgs a) {
  pdl_wait();
  extern __shared__ uint64_t dcp_smem[];
  int* hist = reinterpret_cast<int*>(dcp_smem);                   // [4096] radix select
  uint32_t* win = reinterpret_cast<uint32_t*>(dcp_smem + 2048);  // [2048] winners (token)
  __shared__ int smw[64];
  __shared__ uint32_t selbits[32 * kDcpThreads / 32];             // one bit per candidate (32 per thread)
  __shared__ int cnt[kDcpMaxWorld], off[kDcpMaxWorld + 1], held[kDcpMaxWorld], sel[kDcpMaxWorld];
  __shared__ int s_resend, s_words;
  const int row = blockIdx.x;
  const int L = dcp_row_len(a, row, true);
  int32_t* out = a.topk_idx + size_t(row) * a.K;
  if (L <= a.K) {
    // every visible token is kept, as in the single-GPU top-k
    for (int i = threadIdx.x; i < a.K; i += kDcpThreads) out[i] = i < L ? i : -1;
    if (a.stats && threadIdx.x == 0) {
      a.stats[2 * row] = 0;
      a.stats[2 * row + 1] = L;
    }
    return;
  }
  if (threadIdx.x < a.W) {
    held[threadIdx.x] = a.lcount[size_t(row) * kDcpMaxWorld + threadIdx.x];
    sel[threadIdx.x] = 0;
  }
  if (threadIdx.x == 0) s_resend = 0;
  __syncthreads();
  for (int ex = 0; ex < 2; ++ex) {
    if (threadIdx.x == 0) {
      int o = 0, words = ex == 0 ? 0 : s_words;
      for (int r = 0; r < a.W; ++r) {
        const bool full = (s_resend >> r) & 1;
        cnt[r] = min(full ? a.K : a.m, held[r]);
        off[r] = o;
        o += cnt[r];
        if (ex == 0 || full) words += cnt[r];
      }
      off[a.W] = o;
      s_words = words;
    }
    __syncthreads();
    const int total = off[a.W];
    // the K largest words (all distinct); the second exchange holds at most ~W/1.5 full lists
    if (ex == 0) {
      uint32_t wd[4];
      exchange_words<4>(a, row, cnt, off, total, wd);
      const uint32_t tau = block_kth_key<kDcpThreads, 4>(wd, a.K, hist, smw);
      take_exchange<4>(a, row, wd, tau, off, selbits, sel, win, smw, true);
      if (threadIdx.x == 0) {
        int mask = 0;
        for (int r = 0; r < a.W; ++r)
          if (held[r] > a.m && sel[r] == a.m) mask |= 1 << r;
        s_resend = mask;
      }
      __syncthreads();
      if (s_resend == 0) break;  // the first exchange's winners stand
    } else {
      uint32_t wd[32];
      exchange_words<32>(a, row, cnt, off, total, wd);
      const uint32_t tau = block_kth_key<kDcpThreads, 32>(wd, a.K, hist, smw);
      take_exchange<32>(a, row, wd, tau, off, selbits, sel, win, smw, true);
    }
  }
  // winners in ascending token order (exactly K of them: the words are distinct)
  for (int i = a.K + threadIdx.x; i < kMaxTopK; i += kDcpThreads) win[i] = 0xFFFFFFFFu;
  __syncthreads();
  sort2048<uint32_t>(win);
  for (int i = threadIdx.x; i < a.K; i += kDcpThreads) out[i] = int32_t(win[i]);
  if (a.stats && threadIdx.x == 0) {
    a.stats[2 * row] = s_resend;
    a.stats[2 * row + 1] = s_words;
  }
}

// ---------------------------------------------------------------- LSE combine
// out = sum_i e^{lse_i - lse} O_i, lse = ln sum_i e^{lse_i} over the parts; a
// part with lse_i = -inf (no tokens) adds nothing; all parts empty -> 0, -inf.
// 64 threads per (row, head), 8 dims (16 B of bf16) per thread per part.
constexpr int kCombPairs = 4;

__global__ void __launch_bounds__(64 * kCombPairs) dcp_lse_combine_kernel(const __nv_bfloat16* __restrict__ part_out,
                                                                         const float* __restrict__ part_lse,
                                                                         int parts, int pairs,
                                                                         __nv_bfloat16* __restrict__ out,
                                                                         float* __restrict__ lse) {
  pdl_wait();
  const int pair = blockIdx.x * kCombPairs + int(threadIdx.x >> 6);
  if (pair >= pairs) return;
  const int d0 = int(threadIdx.x & 63) * 8;
  float li[kDcpMaxWorld];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < kDcpMaxWorld; ++i) {
    li[i] = i < parts ? __ldg(part_lse + size_t(i) * pairs + pair) : -INFINITY;
    m = fmaxf(m, li[i]);
  }
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float total = -INFINITY;
  if (m != -INFINITY) {
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < kDcpMaxWorld; ++i) sum += (li[i] == -INFINITY) ? 0.f : expf(li[i] - m);
    total = m + logf(sum);
#pragma unroll
    for (int i = 0; i < kDcpMaxWorld; ++i) {
      if (i < parts && li[i] != -INFINITY) {
        const float wi = expf(li[i] - total);
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(part_out + (size_t(i) * pairs + pair) * kDNope + d0));
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 f = __bfloat1622float2(h[u]);
          acc[2 * u] = fmaf(wi, f.x, acc[2 * u]);
          acc[2 * u + 1] = fmaf(wi, f.y, acc[2 * u + 1]);
        }
      }
    }
  }
  uint4 o;
  __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
  for (int u = 0; u < 4; ++u) oh[u] = __floats2bfloat162_rn(acc[2 * u], acc[2 * u + 1]);
  *reinterpret_cast<uint4*>(out + size_t(pair) * kDNope + d0) = o;
  if (lse && d0 == 0) lse[pair] = total;
}

}  // namespace

cudaError_t launch_dcp_lse_combine(int rows, int parts, const void* part_out, const float* part_lse, void* out,
                                   float* lse, cudaStream_t st) {
  const int pairs = rows * kHeads;
  return launch_pdl(dcp_lse_combine_kernel, dim3((pairs + kCombPairs - 1) / kCombPairs), dim3(64 * kCombPairs), 0,
                    st, static_cast<const __nv_bfloat16*>(part_out), part_lse, parts, pairs,
                    static_cast<__nv_bfloat16*>(out), lse);
}

cudaError_t launch_dcp_merge(const dsa_params_t& p, const WsLayout& L, char* ws, const float* scores,
                             int64_t score_stride, const int32_t* ctx_lens, int world, int32_t* topk_idx,
                             int32_t* stats, cudaStream_t st) {
  DcpArgs a;
  a.scores = scores;
  a.stride = score_stride;
  a.ctx_lens = ctx_lens;
  a.n_q = p.n_q;
  a.cap = L.cap;
  a.K = p.topk;
  a.W = world;
  a.m = (3 * p.topk + 2 * world - 1) / (2 * world);  // ceil(1.5 K / W)
  a.S = ((int64_t(L.cap) + world - 1) / world + 7) / 8 * 8;
  a.keys16 = reinterpret_cast<uint16_t*>(ws + L.dcp_keys16);
  a.lkey = reinterpret_cast<uint32_t*>(ws + L.dcp_key);
  a.ltok = reinterpret_cast<int32_t*>(ws + L.dcp_tok);
  a.lcount = reinterpret_cast<int32_t*>(ws + L.dcp_cnt);
  a.topk_idx = topk_idx;
  a.stats = stats;
  a.err = reinterpret_cast<int*>(ws + L.err);
  const size_t shard_smem = size_t(kMaxTopK) * 8 + size_t(kTieCap) * 4;
  const size_t merge_smem = size_t(2048) * 8 + size_t(kMaxTopK) * 8;
  cudaError_t e = cudaFuncSetAttribute(dcp_shard_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(shard_smem));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dcp_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(merge_smem));
  if (e == cudaSuccess)
    e = launch_pdl(dcp_keys_kernel, dim3((L.cap + 4 * kKeysThreads - 1) / (4 * kKeysThreads), L.rows),
                   dim3(kKeysThreads), 0, st, a);
  if (e == cudaSuccess)
    e = launch_pdl(dcp_shard_kernel, dim3(world * kShardCluster, L.rows), dim3(kDcpThreads), shard_smem, st, a);
  if (e == cudaSuccess) e = launch_pdl(dcp_merge_kernel, dim3(L.rows), dim3(kDcpThreads), merge_smem, st, a);
  return e;
}

}  // namespace dsa
