// Stage 3: exact absorbed-MLA attention over the selected latents, split over
// the K selected slots, then an LSE merge of the splits.
//
// ("vLLM 为 Kimi K3.1 Pro 提供 Day-0 支持", "K3.1 Pro 中的稀疏注意力": attention runs
// exactly over the kept tokens' 576-B FP8 latents, one latent shared by all 96
// heads; "长上下文：带稀疏 indexer 的 decode 上下文并行": partial outputs merge by
// log-sum-exp.)
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "dsa_internal.cuh"

namespace dsa {

namespace {

__device__ __forceinline__ float e4m3f(uint8_t c) {
  __half_raw hr = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c), __NV_E4M3);
  return __half2float(__half(hr));
}

constexpr int kHG = 16;   // heads per CTA
constexpr int kTT = 32;   // tokens per tile
constexpr int kCS = kDQK + 1;

struct MlaArgs {
  const __nv_bfloat16* q;
  const uint8_t* lat_pool;
  int64_t lat_stride;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  const int32_t* topk_idx;
  int max_pages, num_pages, n_q, cap, K, splits, per_split;
  float sm_scale, lat_scale;
  float* opart;  // [rows][splits][96][512]
  float* lpart;  // [rows][splits][96]
  int* err;
};

// One CTA per (split, row, group of 16 heads); O for 16 heads x 512 dims in registers.
__global__ void __launch_bounds__(256) sparse_mla_simt_kernel(MlaArgs a) {
  extern __shared__ float sm[];
  float* qs = sm;                      // [16][576]
  float* cs = qs + kHG * kDQK;         // [32][577]
  float* ps = cs + kTT * kCS;          // [16][32]
  __shared__ float s_m[kHG], s_l[kHG], s_alpha[kHG];
  __shared__ const uint8_t* s_row[kTT];

  const int split = blockIdx.x, r = blockIdx.y, hg = blockIdx.z;
  const int b = r / a.n_q, t = r - b * a.n_q;
  const int ctx = a.ctx_lens[b];
  const int L = (ctx < a.n_q || ctx > a.cap) ? 0 : ctx - a.n_q + t + 1;
  const int tid = threadIdx.x;

  for (int i = tid; i < kHG * kDQK; i += 256) {
    const int h = i / kDQK, d = i - h * kDQK;
    qs[i] = __bfloat162float(a.q[(size_t(r) * kHeads + hg * kHG + h) * kDQK + d]);
  }
  if (tid < kHG) { s_m[tid] = -INFINITY; s_l[tid] = 0.f; }
  float o[kHG][2];
#pragma unroll
  for (int h = 0; h < kHG; ++h) o[h][0] = o[h][1] = 0.f;

  const int j0 = split * a.per_split;
  const int j1 = min(a.K, j0 + a.per_split);
  for (int jt = j0; jt < j1; jt += kTT) {
    __syncthreads();
    if (tid < kTT) {
      const uint8_t* rowp = nullptr;
      const int j = jt + tid;
      if (j < j1) {
        const int s = a.topk_idx[size_t(r) * a.K + j];
        if (s >= 0 && s < L) {
          const int pg = a.block_table[size_t(b) * a.max_pages + s / kPage];
          if (pg >= 0 && pg < a.num_pages)
            rowp = a.lat_pool + size_t(pg) * a.lat_stride + size_t(s % kPage) * kLatRowFp8;
          else
            atomicOr(a.err, DSA_DEVERR_BLOCK_TABLE);
        } else if (s != -1) {
          atomicOr(a.err, DSA_DEVERR_TOPK_INDEX);
        }
      }
      s_row[tid] = rowp;
    }
    __syncthreads();
    for (int i = tid; i < kTT * (kDQK / 16); i += 256) {
      const int j = i / (kDQK / 16), c = i - j * (kDQK / 16);
      const uint8_t* rp = s_row[j];
      float* dst = cs + j * kCS + c * 16;
      if (rp) {
        const uint4 v = *reinterpret_cast<const uint4*>(rp + c * 16);
        const uint8_t* by = reinterpret_cast<const uint8_t*>(&v);
#pragma unroll
        for (int e = 0; e < 16; ++e) dst[e] = e4m3f(by[e]) * a.lat_scale;
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) dst[e] = 0.f;
      }
    }
    __syncthreads();
    {
      const int h = tid >> 4, jj = tid & 15;
#pragma unroll
      for (int k2 = 0; k2 < 2; ++k2) {
        const int j = jj + 16 * k2;
        float d = 0.f;
        const float* qv = qs + h * kDQK;
        const float* cv = cs + j * kCS;
        for (int i = 0; i < kDQK; ++i) d = fmaf(qv[i], cv[i], d);
        ps[h * kTT + j] = s_row[j] ? d * a.sm_scale : -INFINITY;
      }
    }
    __syncthreads();
    if (tid < kHG) {
      const int h = tid;
      float mt = -INFINITY;
      for (int j = 0; j < kTT; ++j) mt = fmaxf(mt, ps[h * kTT + j]);
      const float mo = s_m[h];
      const float mn = fmaxf(mo, mt);
      float alpha = 1.f, lsum = 0.f;
      if (mn == -INFINITY) {
        for (int j = 0; j < kTT; ++j) ps[h * kTT + j] = 0.f;
      } else {
        alpha = (mo == -INFINITY) ? 0.f : expf(mo - mn);
        for (int j = 0; j < kTT; ++j) {
          const float pj = expf(ps[h * kTT + j] - mn);
          ps[h * kTT + j] = pj;
          lsum += pj;
        }
      }
      s_m[h] = mn;
      s_l[h] = s_l[h] * alpha + lsum;
      s_alpha[h] = alpha;
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < kHG; ++h) {
      const float al = s_alpha[h];
      float a0 = o[h][0] * al, a1 = o[h][1] * al;
      for (int j = 0; j < kTT; ++j) {
        const float pj = ps[h * kTT + j];
        a0 = fmaf(pj, cs[j * kCS + tid], a0);
        a1 = fmaf(pj, cs[j * kCS + tid + 256], a1);
      }
      o[h][0] = a0;
      o[h][1] = a1;
    }
  }
  __syncthreads();
  float* op = a.opart + ((size_t(r) * a.splits + split) * kHeads + hg * kHG) * kDNope;
#pragma unroll
  for (int h = 0; h < kHG; ++h) {
    const float l = s_l[h];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    op[h * kDNope + tid] = o[h][0] * inv;
    op[h * kDNope + tid + 256] = o[h][1] * inv;
  }
  if (tid < kHG) {
    const float l = s_l[tid];
    a.lpart[(size_t(r) * a.splits + split) * kHeads + hg * kHG + tid] = l > 0.f ? s_m[tid] + logf(l) : -INFINITY;
  }
}

// LSE merge of the splits of one row: out = sum_i e^{lse_i - lse} O_i, lse = ln sum_i e^{lse_i}.
__global__ void __launch_bounds__(256) mla_combine_kernel(const float* __restrict__ opart,
                                                          const float* __restrict__ lpart, int splits,
                                                          __nv_bfloat16* __restrict__ out,
                                                          float* __restrict__ lse) {
  const int r = blockIdx.x;
  const int h = blockIdx.y;
  __shared__ float wts[kMaxSplits];
  __shared__ float s_lse;
  if (threadIdx.x == 0) {
    float m = -INFINITY;
    for (int i = 0; i < splits; ++i) m = fmaxf(m, lpart[(size_t(r) * splits + i) * kHeads + h]);
    float tot = 0.f;
    if (m != -INFINITY)
      for (int i = 0; i < splits; ++i) tot += expf(lpart[(size_t(r) * splits + i) * kHeads + h] - m);
    const float L = m == -INFINITY ? -INFINITY : m + logf(tot);
    for (int i = 0; i < splits; ++i)
      wts[i] = m == -INFINITY ? 0.f : expf(lpart[(size_t(r) * splits + i) * kHeads + h] - L);
    s_lse = L;
  }
  __syncthreads();
  for (int d = threadIdx.x; d < kDNope; d += 256) {
    float acc = 0.f;
    for (int i = 0; i < splits; ++i) acc = fmaf(wts[i], opart[((size_t(r) * splits + i) * kHeads + h) * kDNope + d], acc);
    out[(size_t(r) * kHeads + h) * kDNope + d] = __float2bfloat16_rn(acc);
  }
  if (lse && threadIdx.x == 0) lse[size_t(r) * kHeads + h] = s_lse;
}

}  // namespace

cudaError_t launch_sparse_mla(const dsa_params_t& p, const WsLayout& L, char* ws, const void* q,
                              const void* lat_pool, const int32_t* block_table, const int32_t* ctx_lens,
                              const int32_t* topk_idx, void* out, float* lse, cudaStream_t st) {
  MlaArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.lat_pool = static_cast<const uint8_t*>(lat_pool);
  a.lat_stride = p.lat_page_stride;
  a.block_table = block_table;
  a.ctx_lens = ctx_lens;
  a.topk_idx = topk_idx;
  a.max_pages = p.max_pages_per_req;
  a.num_pages = p.num_pages;
  a.n_q = p.n_q;
  a.cap = L.cap;
  a.K = p.topk;
  a.splits = L.splits;
  a.per_split = ((p.topk + L.splits - 1) / L.splits + kTT - 1) / kTT * kTT;
  a.sm_scale = p.softmax_scale;
  a.lat_scale = p.latent_scale;
  a.opart = reinterpret_cast<float*>(ws + L.opart);
  a.lpart = reinterpret_cast<float*>(ws + L.lpart);
  a.err = reinterpret_cast<int*>(ws + L.err);
  const size_t smem = (size_t(kHG) * kDQK + size_t(kTT) * kCS + kHG * kTT) * sizeof(float);
  cudaFuncSetAttribute(sparse_mla_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  dim3 grid(L.splits, L.rows, kHeads / kHG);
  sparse_mla_simt_kernel<<<grid, 256, smem, st>>>(a);
  dim3 g2(L.rows, kHeads);
  mla_combine_kernel<<<g2, 256, 0, st>>>(a.opart, a.lpart, L.splits, static_cast<__nv_bfloat16*>(out), lse);
  return cudaGetLastError();
}

}  // namespace dsa
