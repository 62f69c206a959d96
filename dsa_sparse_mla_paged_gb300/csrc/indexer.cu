// Stage 1: the lightning indexer over the paged FP8 index-key cache.
//
// score(t, s) = sum_h w'_h * max(0, scale_s * (q8_h . k_s)), with the indexer
// query quantised to E4M3 per head and its scale folded into the head weights
// (vLLM, "vLLM 为 Kimi K3.1 Pro 提供 Day-0 支持": sections "K3.1 Pro 中的稀疏注意力"
// and "低延迟解码：融合的 DSA 解码路径").
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "dsa_internal.cuh"

namespace dsa {

// ---------------------------------------------------------------------------
// FP8 query quantisation: one warp per 8 heads of one row.
//   amax_h = max |q_h|, q8 = E4M3_rne_sat(q * (448 / amax_h)), w' = w * (amax_h / 448)
// Every step is an IEEE fp32 operation with round-to-nearest (explicit _rn
// intrinsics, so no contraction or fast-math rewrite changes a bit).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) idx_q_quant_kernel(const __nv_bfloat16* __restrict__ q_idx,
                                                          const float* __restrict__ w,
                                                          uint8_t* __restrict__ q8,
                                                          float* __restrict__ wq) {
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int hh = 0; hh < 8; ++hh) {
    const int h = warp * 8 + hh;
    const size_t base = (size_t(row) * kIdxHeads + h) * kIdxDim + lane * 4;
    const uint2 raw = *reinterpret_cast<const uint2*>(q_idx + base);
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
    float v[4] = {__low2float(a), __high2float(a), __low2float(b), __high2float(b)};
    float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float inv = m > 0.f ? __fdiv_rn(448.0f, m) : 1.0f;
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(__fmul_rn(v[i], inv), __NV_SATFINITE, __NV_E4M3);
      packed |= uint32_t(c) << (8 * i);
    }
    *reinterpret_cast<uint32_t*>(q8 + base) = packed;
    if (lane == 0) wq[size_t(row) * kIdxHeads + h] = __fmul_rn(w[size_t(row) * kIdxHeads + h], __fdiv_rn(m, 448.0f));
  }
}

cudaError_t launch_idx_q_quant(const dsa_params_t& p, const void* q_idx, const float* w, uint8_t* q8,
                               float* wq, cudaStream_t st) {
  const int rows = p.batch * p.n_q;
  idx_q_quant_kernel<<<rows, 128, 0, st>>>(static_cast<const __nv_bfloat16*>(q_idx), w, q8, wq);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Reference-shaped SIMT scorer: one CTA per (page, request), all n_q rows.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float e4m3_to_float(uint8_t c) {
  __half_raw hr = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c), __NV_E4M3);
  return __half2float(__half(hr));
}

__global__ void __launch_bounds__(256) indexer_simt_kernel(
    const uint8_t* __restrict__ q8, const float* __restrict__ wq, const uint8_t* __restrict__ key_pool,
    int64_t key_page_stride, const int32_t* __restrict__ block_table, int max_pages,
    const int32_t* __restrict__ ctx_lens, int num_pages, int n_q, float* __restrict__ scores,
    int64_t score_stride, int* err) {
  extern __shared__ float sm[];
  float* kf = sm;                              // [64][129]
  float* qf = kf + 64 * 129;                   // [n_q*32][128]
  float* part = qf + n_q * kIdxHeads * kIdxDim;  // [4][64]
  __shared__ float ssc[64];

  const int lp = blockIdx.x, b = blockIdx.y;
  const int cap = max_pages * kPage;
  const int ctx = ctx_lens[b];
  if (ctx < n_q || ctx > cap) {
    if (lp == 0 && threadIdx.x == 0) atomicOr(err, DSA_DEVERR_CTX);
    return;
  }
  if (lp * kPage >= ctx) return;
  int page = block_table[size_t(b) * max_pages + lp];
  if (page < 0 || page >= num_pages) {
    if (threadIdx.x == 0) atomicOr(err, DSA_DEVERR_BLOCK_TABLE);
    page = 0;
  }
  const uint8_t* pg = key_pool + size_t(page) * key_page_stride;
  for (int i = threadIdx.x; i < 64 * 128; i += 256) kf[(i >> 7) * 129 + (i & 127)] = e4m3_to_float(pg[i]);
  if (threadIdx.x < 64) ssc[threadIdx.x] = reinterpret_cast<const float*>(pg + 64 * 128)[threadIdx.x];
  const uint8_t* qrow = q8 + size_t(b) * n_q * kIdxHeads * kIdxDim;
  for (int i = threadIdx.x; i < n_q * kIdxHeads * kIdxDim; i += 256) qf[i] = e4m3_to_float(qrow[i]);
  __syncthreads();

  const int j = threadIdx.x & 63, g = threadIdx.x >> 6;
  const float sc = ssc[j];
  for (int t = 0; t < n_q; ++t) {
    float acc = 0.f;
    for (int hh = 0; hh < 8; ++hh) {
      const int h = g * 8 + hh;
      const float* qv = qf + (t * kIdxHeads + h) * kIdxDim;
      const float* kv = kf + j * 129;
      float d = 0.f;
#pragma unroll 8
      for (int i = 0; i < kIdxDim; ++i) d = fmaf(qv[i], kv[i], d);
      acc += wq[(size_t(b) * n_q + t) * kIdxHeads + h] * fmaxf(sc * d, 0.f);
    }
    part[g * 64 + j] = acc;
    __syncthreads();
    if (threadIdx.x < 64) {
      const int s = lp * kPage + threadIdx.x;
      const int L = ctx - n_q + t + 1;
      const float v = (part[threadIdx.x] + part[64 + threadIdx.x]) + (part[128 + threadIdx.x] + part[192 + threadIdx.x]);
      if (s < L && s < score_stride) scores[(size_t(b) * n_q + t) * score_stride + s] = v;
    }
    __syncthreads();
  }
}

cudaError_t launch_indexer(const dsa_params_t& p, const uint8_t* q8, const float* wq, const void* key_pool,
                           const int32_t* block_table, const int32_t* ctx_lens, float* scores,
                           int64_t score_stride, int* err, cudaStream_t st) {
  const size_t smem = (64 * 129 + size_t(p.n_q) * kIdxHeads * kIdxDim + 4 * 64) * sizeof(float);
  cudaFuncSetAttribute(indexer_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  dim3 grid(p.max_pages_per_req, p.batch);
  indexer_simt_kernel<<<grid, 256, smem, st>>>(q8, wq, static_cast<const uint8_t*>(key_pool), p.key_page_stride,
                                              block_table, p.max_pages_per_req, ctx_lens, p.num_pages, p.n_q,
                                              scores, score_stride, err);
  return cudaGetLastError();
}

}  // namespace dsa
