// The fused indexer front end of a decode step ("vLLM 为 Kimi K3.1 Pro 提供 Day-0
// 支持", section "低延迟解码：融合的 DSA 解码路径": a single kernel normalises the
// query latent, projects it onto the indexer heads, makes it FP8 with the scale
// moved into the head weights, and produces the new token's index key).
// For query row (b, t):
//   n  = bf16(c_q / sqrt(mean(c_q^2) + eps) * gamma)       query RMS norm
//   q  = bf16(n @ W_q^T)                                    32 heads x 128
//   q8 = E4M3(q * 448 / amax_h), w' = w * (amax_h / 448)    the scorer's inputs
//   k  = bf16(x @ W_k^T)                                    the new token's key
// and k goes, FP8 (E4M3 + fp32 scale) or MXFP4 (E2M1 + E8M0 per 32), into the
// cache slot of token ctx_b - n_q + t.
//
// Grid: 8 x 37 CTAs. Row j < 32 computes head j, rows 32..35 a quarter of
// the key's hidden width each, and the first CTA of row 36 writes the
// scorer's tile plan. A CTA owns 16 of the 128 outputs of its head (or key
// quarter): it prefetches those 16 weight rows into L2 at launch, then streams
// them (once per group of R = 4 or 8 query rows) against the group's inputs,
// staged as fp32 in shared memory 2,048 columns at a time (two CTAs fit an SM,
// so the 296 CTAs run in one wave). Each CTA leaves its outputs in the
// workspace; the last CTA of a head (or of the key) to finish a pass, found by
// an arrival counter, reads them back, rounds and quantises the rows and
// writes them (the key's quarters are added in order). A decode step is bound
// by the weight bytes.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "dsa_internal.cuh"
#include "sm103_ptx.cuh"

namespace dsa {

namespace {

constexpr int kFeSplit = 8;      // CTAs per 128 outputs (16 outputs each)
constexpr int kFeThreads = 256;  // 8 warps x 2 outputs
constexpr int kFeKeyParts = 4;   // the key's hidden width is split in quarters
constexpr int kFeJobs = kIdxHeads + kFeKeyParts + 1;  // heads, key quarters, the plan
constexpr int kFeOut = kIdxDim / kFeSplit;
constexpr int kFeBlk = 8;        // 16-byte chunks per lane per staged block: 2,048 inputs per row
static_assert(kFeMaxRows % 8 == 0, "whole passes");
static_assert(kFeOut == 2 * (kFeThreads / 32), "two outputs per warp");

struct FeArgs {
  const __nv_bfloat16* c_q;
  const __nv_bfloat16* gamma;
  const __nv_bfloat16* w_q;
  const float* w;
  const __nv_bfloat16* x;
  const __nv_bfloat16* w_k;
  uint8_t* key_pool;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  uint8_t* q8;
  float* wq;
  uint8_t* q8_out;
  float* w_out;
  int* tile_prefix;
  int* err;
  float* fe_part;  // [kFeKeyParts][rows][128] the key's partial sums
  float* fe_q;     // [rows][32][128] the heads' bf16-rounded outputs
  int* fe_cnt;     // [33][kFeMaxPasses] arrivals per (head or key, pass); 0 between calls
  int64_t key_page_stride;
  int rows, batch, n_q, d_c, d_model, max_pages, num_pages, cap, mx;
  float eps;
};

__device__ __forceinline__ void bf16x8(const uint4& v, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ float warp_max(float m) {
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  return m;
}

// E2M1 code of y: nearest of {0, .5, 1, 1.5, 2, 3, 4, 6} with ties to the even
// code, magnitudes past 6 saturating, the sign bit kept.
__device__ __forceinline__ uint32_t e2m1_code(float y) {
  const float a = fabsf(y);
  const uint32_t mag = a <= 0.25f ? 0u : a < 0.75f ? 1u : a <= 1.25f ? 2u : a < 1.75f ? 3u
                     : a <= 2.5f ? 4u : a < 3.5f ? 5u : a <= 5.0f ? 6u : 7u;
  return mag | (signbit(y) ? 8u : 0u);
}

// 2^-e for e in [-127, 127] (2^-127 is the subnormal 0x00400000).
__device__ __forceinline__ float exp2_neg(int e) {
  return e <= 126 ? __uint_as_float(uint32_t(127 - e) << 23) : __uint_as_float(0x00400000u);
}

// Rank-0 epilogue of one row: the 128 bf16 outputs of the row (4 per lane).
__device__ __forceinline__ void head_out(const FeArgs& a, int row, int h, int lane, const float (&v)[4]) {
  const float m = warp_max(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
  const float inv = m > 0.f ? __fdiv_rn(448.0f, m) : 1.0f;
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    packed |= uint32_t(__nv_cvt_float_to_fp8(__fmul_rn(v[i], inv), __NV_SATFINITE, __NV_E4M3)) << (8 * i);
  const size_t off = (size_t(row) * kIdxHeads + h) * kIdxDim + lane * 4;
  *reinterpret_cast<uint32_t*>(a.q8 + off) = packed;
  if (a.q8_out) *reinterpret_cast<uint32_t*>(a.q8_out + off) = packed;
  if (lane == 0) {
    const float wp = __fmul_rn(a.w[size_t(row) * kIdxHeads + h], __fdiv_rn(m, 448.0f));
    a.wq[size_t(row) * kIdxHeads + h] = wp;
    if (a.w_out) a.w_out[size_t(row) * kIdxHeads + h] = wp;
  }
}

__device__ __forceinline__ void key_out(const FeArgs& a, int row, int lane, const float (&v)[4]) {
  const int b = row / a.n_q, t = row - b * a.n_q;
  const int ctx = a.ctx_lens[b];
  if (ctx < a.n_q || ctx > a.cap) {
    if (lane == 0) atomicOr(a.err, DSA_DEVERR_CTX);
    return;
  }
  const int pos = ctx - a.n_q + t;
  const int pg = a.block_table[size_t(b) * a.max_pages + pos / kPage];
  if (pg < 0 || pg >= a.num_pages) {
    if (lane == 0) atomicOr(a.err, DSA_DEVERR_BLOCK_TABLE);
    return;
  }
  uint8_t* page = a.key_pool + size_t(pg) * a.key_page_stride;
  const int slot = pos % kPage;
  if (!a.mx) {
    const float m = warp_max(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
    const float inv = m > 0.f ? __fdiv_rn(448.0f, m) : 1.0f;
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      packed |= uint32_t(__nv_cvt_float_to_fp8(__fmul_rn(v[i], inv), __NV_SATFINITE, __NV_E4M3)) << (8 * i);
    *reinterpret_cast<uint32_t*>(page + slot * kIdxDim + lane * 4) = packed;
    if (lane == 0) *reinterpret_cast<float*>(page + kPage * kIdxDim + slot * 4) = __fdiv_rn(m, 448.0f);
  } else {
    // lanes 8g .. 8g + 7 hold block g (values 32g .. 32g + 31)
    float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 4; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    int e = 0;
    if (m > 0.f) {
      const int ex = int((__float_as_uint(m) >> 23) & 0xFFu);  // floor(log2 m) + 127 for a normal m
      e = max(-127, min(127, ex - 127 - 2));
    }
    const float s = exp2_neg(e);
    const uint32_t c0 = e2m1_code(__fmul_rn(v[0], s)), c1 = e2m1_code(__fmul_rn(v[1], s));
    const uint32_t c2 = e2m1_code(__fmul_rn(v[2], s)), c3 = e2m1_code(__fmul_rn(v[3], s));
    *reinterpret_cast<uint16_t*>(page + slot * 64 + lane * 2) = uint16_t(c0 | c1 << 4 | c2 << 8 | c3 << 12);
    if ((lane & 7) == 0) page[kPage * 64 + slot * 4 + (lane >> 3)] = uint8_t(e + 127);
  }
}

template <int R>
__global__ void __launch_bounds__(kFeThreads, 2)
    idx_frontend_kernel(FeArgs a) {
  pdl_trigger();
  extern __shared__ __align__(16) float fe_in[];           // [R][kFeBlk * 256] staged inputs (fp32)
  __shared__ float s_rstd[R];
  __shared__ int s_last;
  const int job = blockIdx.y;
  if (job == kFeJobs - 1) {  // the tile plan
    if (blockIdx.x == 0)  // decode rows (n_q <= 8): one unit per request
      build_tile_plan<kFeThreads>(a.ctx_lens, a.batch, unit_map(a.n_q, 1, 0), a.cap, a.tile_prefix, a.err);
    return;
  }
  const int rank = blockIdx.x;  // which 16 outputs
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool is_key = job >= kIdxHeads;
  const int part = job - kIdxHeads;  // key: which quarter of the hidden width
  const int d = is_key ? a.d_model : a.d_c;
  const int nch = d / 256;           // 16-byte chunks per lane per row
  const int cj0 = is_key ? part * nch / kFeKeyParts : 0;
  const int cj1 = is_key ? (part + 1) * nch / kFeKeyParts : nch;
  const int o0 = rank * kFeOut + 2 * warp;  // this warp's outputs o0, o0 + 1
  const __nv_bfloat16* w0 = is_key ? a.w_k + size_t(o0) * d : a.w_q + (size_t(job) * kIdxDim + o0) * d;
  const __nv_bfloat16* w1 = w0 + d;
  // The weights are constants of the model, not outputs of the previous
  // kernel: start pulling this CTA's 16 row segments into L2 before waiting.
  if (threadIdx.x < kFeOut) {
    const __nv_bfloat16* row = w0 + (int(threadIdx.x) - 2 * warp) * size_t(d) + size_t(cj0) * 256;
    ptx::prefetch_l2_bulk(row, uint32_t(cj1 - cj0) * 512u);
  }
  pdl_wait();
  for (int r0 = 0, pass = 0; r0 < a.rows; r0 += R, ++pass) {
    const int nr = min(R, a.rows - r0);
    // ---- the query rows' 1 / RMS (warp w: row r0 + w); the first block's raw
    // values stay in shared memory for the staging below
    __syncthreads();  // the previous pass's inputs are consumed
    if (!is_key && warp < nr) {
      const uint4* src = reinterpret_cast<const uint4*>(a.c_q + size_t(r0 + warp) * d);
      float4* raw = reinterpret_cast<float4*>(fe_in) + size_t(warp) * kFeBlk * 64;
      float ss = 0.f;
      for (int j = 0; j < nch; ++j) {
        float f[8];
        bf16x8(__ldg(src + j * 32 + lane), f);
        if (j < kFeBlk) {
          raw[(j * 32 + lane) * 2] = make_float4(f[0], f[1], f[2], f[3]);
          raw[(j * 32 + lane) * 2 + 1] = make_float4(f[4], f[5], f[6], f[7]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) s_rstd[warp] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, float(d)), a.eps)));
      __syncwarp();  // the warp's staging reads it
    }
    float acc0[R], acc1[R];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) acc0[rr] = acc1[rr] = 0.f;
    for (int jb = cj0; jb < cj1; jb += kFeBlk) {
      const int nj = min(kFeBlk, cj1 - jb);
      const uint4* pw0 = reinterpret_cast<const uint4*>(w0) + jb * 32;
      const uint4* pw1 = reinterpret_cast<const uint4*>(w1) + jb * 32;
      // the block's first four weight chunks, loaded before the staging so
      // that their latency overlaps it
      uint4 wa[4], wb[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (u < nj) {
          wa[u] = __ldg(pw0 + u * 32 + lane);
          wb[u] = __ldg(pw1 + u * 32 + lane);
        }
      if (jb != cj0) __syncthreads();  // the previous block's inputs are consumed
      // ---- stage the block's inputs as fp32: warp w prepares row r0 + w
      if (warp < nr) {
        const int row = r0 + warp;
        float4* dst = reinterpret_cast<float4*>(fe_in) + size_t(warp) * kFeBlk * 64;
        if (is_key) {
          const uint4* src = reinterpret_cast<const uint4*>(a.x + size_t(row) * d) + jb * 32;
          for (int j = 0; j < nj; ++j) {
            float f[8];
            bf16x8(__ldg(src + j * 32 + lane), f);
            dst[(j * 32 + lane) * 2] = make_float4(f[0], f[1], f[2], f[3]);
            dst[(j * 32 + lane) * 2 + 1] = make_float4(f[4], f[5], f[6], f[7]);
          }
        } else {
          const uint4* src = reinterpret_cast<const uint4*>(a.c_q + size_t(row) * d) + jb * 32;
          const uint4* g = reinterpret_cast<const uint4*>(a.gamma) + jb * 32;
          const float rstd = s_rstd[warp];  // written by this warp's lane 0
          for (int j = 0; j < nj; ++j) {
            float f[8], gg[8], n[8];
            if (jb == 0) {  // the raw values are already here (this lane wrote them)
              const float4 ra = dst[(j * 32 + lane) * 2], rb = dst[(j * 32 + lane) * 2 + 1];
              f[0] = ra.x; f[1] = ra.y; f[2] = ra.z; f[3] = ra.w;
              f[4] = rb.x; f[5] = rb.y; f[6] = rb.z; f[7] = rb.w;
            } else {
              bf16x8(__ldg(src + j * 32 + lane), f);
            }
            bf16x8(__ldg(g + j * 32 + lane), gg);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              n[i] = __bfloat162float(__float2bfloat16_rn(__fmul_rn(__fmul_rn(f[i], rstd), gg[i])));
            dst[(j * 32 + lane) * 2] = make_float4(n[0], n[1], n[2], n[3]);
            dst[(j * 32 + lane) * 2 + 1] = make_float4(n[4], n[5], n[6], n[7]);
          }
        }
      }
      __syncthreads();
      // ---- the warp's two weight rows against the block's rows, four chunks at a time
      for (int jg = 0; jg < nj; jg += 4) {
        if (jg > 0) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (jg + u < nj) {
              wa[u] = __ldg(pw0 + (jg + u) * 32 + lane);
              wb[u] = __ldg(pw1 + (jg + u) * 32 + lane);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (jg + u >= nj) break;
          float f0[8], f1[8];
          bf16x8(wa[u], f0);
          bf16x8(wb[u], f1);
#pragma unroll
          for (int rr = 0; rr < R; ++rr) {
            const float4* xr =
                reinterpret_cast<const float4*>(fe_in) + (size_t(rr) * kFeBlk * 32 + (jg + u) * 32 + lane) * 2;
            const float4 xa = xr[0], xb = xr[1];
            const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              acc0[rr] = fmaf(f0[i], xv[i], acc0[rr]);
              acc1[rr] = fmaf(f1[i], xv[i], acc1[rr]);
            }
          }
        }
      }
    }
    // lane 8i + rr (rr < R) keeps output o0 + i of row rr
    float mine = 0.f;
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
      float s0 = acc0[rr], s1 = acc1[rr];
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        s0 += __shfl_xor_sync(0xffffffffu, s0, o);
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
      }
      if (lane == rr) mine = s0;
      if (lane == 8 + rr) mine = s1;
    }
    // Every CTA leaves its outputs in the workspace (a head's bf16-rounded
    // values; the key's fp32 partial sums); the last CTA of the group to finish
    // the pass (a ticket) reads them back, finishes and quantises the rows.
    if (lane < 16 && (lane & 7) < nr) {
      const int hr = lane & 7, ho = o0 + (lane >> 3);
      if (is_key) a.fe_part[(size_t(part) * a.rows + r0 + hr) * kIdxDim + ho] = mine;
      else a.fe_q[(size_t(r0 + hr) * kIdxHeads + job) * kIdxDim + ho] = __bfloat162float(__float2bfloat16_rn(mine));
    }
    __threadfence();
    __syncthreads();
    const int group = is_key ? kIdxHeads : job;
    int* cnt = a.fe_cnt + size_t(group) * kFeMaxPasses + pass;
    if (threadIdx.x == 0) s_last = atomicAdd(cnt, 1) == (is_key ? kFeKeyParts : 1) * kFeSplit - 1;
    __syncthreads();
    if (s_last) {
      __threadfence();
      if (warp < nr) {
        const int row = r0 + warp;
        float v[4];
        if (is_key) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float t = 0.f;
#pragma unroll
            for (int q = 0; q < kFeKeyParts; ++q)
              t = __fadd_rn(t, __ldcg(a.fe_part + (size_t(q) * a.rows + row) * kIdxDim + lane * 4 + i));
            v[i] = __bfloat162float(__float2bfloat16_rn(t));
          }
          key_out(a, row, lane, v);
        } else {
          const float4 g4 = __ldcg(reinterpret_cast<const float4*>(a.fe_q + (size_t(row) * kIdxHeads + job) * kIdxDim) + lane);
          v[0] = g4.x; v[1] = g4.y; v[2] = g4.z; v[3] = g4.w;
          head_out(a, row, job, lane, v);
        }
      }
      if (threadIdx.x == 0) *cnt = 0;  // ready for the next call
    }
  }
}

}  // namespace

cudaError_t launch_idx_frontend(const dsa_params_t& p, const WsLayout& L, char* ws, const FrontendIn& in,
                                cudaStream_t st) {
  FeArgs a;
  a.c_q = static_cast<const __nv_bfloat16*>(in.c_q);
  a.gamma = static_cast<const __nv_bfloat16*>(in.gamma);
  a.w_q = static_cast<const __nv_bfloat16*>(in.w_q);
  a.w = in.w;
  a.x = static_cast<const __nv_bfloat16*>(in.x);
  a.w_k = static_cast<const __nv_bfloat16*>(in.w_k);
  a.key_pool = static_cast<uint8_t*>(in.key_pool);
  a.block_table = in.block_table;
  a.ctx_lens = in.ctx_lens;
  a.q8 = reinterpret_cast<uint8_t*>(ws + L.q8);
  a.wq = reinterpret_cast<float*>(ws + L.wq);
  a.q8_out = static_cast<uint8_t*>(in.q8_out);
  a.w_out = in.w_out;
  a.tile_prefix = reinterpret_cast<int*>(ws + L.tiles);
  a.err = reinterpret_cast<int*>(ws + L.err);
  a.key_page_stride = p.key_page_stride;
  a.rows = L.rows;
  a.batch = p.batch;
  a.n_q = p.n_q;
  a.d_c = in.d_c;
  a.d_model = in.d_model;
  a.max_pages = p.max_pages_per_req;
  a.num_pages = p.num_pages;
  a.cap = L.cap;
  a.mx = p.key_fmt == DSA_KEY_MXFP4_68;
  a.eps = in.eps;
  a.fe_part = reinterpret_cast<float*>(ws + L.fe_part);
  a.fe_cnt = reinterpret_cast<int*>(ws + L.fe_cnt);
  a.fe_q = reinterpret_cast<float*>(ws + L.fe_q);
  // four query rows per pass when the batch has at most four, else eight
  const bool small = L.rows <= 4;
  const size_t smem = size_t(small ? 4 : 8) * kFeBlk * 256 * 4;
  auto kern = small ? idx_frontend_kernel<4> : idx_frontend_kernel<8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e == cudaSuccess) e = launch_pdl(kern, dim3(kFeSplit, kFeJobs), dim3(kFeThreads), smem, st, a);
  return e;
}

}  // namespace dsa
