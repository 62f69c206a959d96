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
#include "sm103_ptx.cuh"

namespace dsa {

namespace {

// ---------------------------------------------------------------------------
// Tensor-core split-KV attention (sm_103a).
//
// A 96-head x 512-dim fp32 output needs all 512 TMEM columns, so each (row,
// split) runs as two CTAs: CTA half hv accumulates output dims [256hv,
// 256hv+256) in TMEM columns [0, 256) and keeps the 64-token score tile in
// columns [256, 320). Both halves compute the same scores (QK^T over all 576
// dims), hence the same softmax; the 96 heads are the M=128 rows (rows 96..127
// are padding that is never read back).
//   warps 0..2  softmax / epilogue: one head row per thread (thread-local
//               online softmax in base 2, lazy rescale of O by more than 2^8)
//   warps 4..7  converters: gather the split's selected latent rows (paged,
//               16-B loads, one tile ahead in registers) and expand E4M3 ->
//               bf16 exactly into the 128-B swizzled K-major tile
//   warp  3     (its TMEM lanes are padding rows) TMEM owner, Q by TMA, MMA issuer:
//               S[128 x 64]  = Q[128 x 576] . C^T           (36 x K=16)
//               O[128 x 256] += P[128 x 64] . V[64 x 256]    (4 x K=16, V MN-major)
// ---------------------------------------------------------------------------
constexpr int kNT = 64;                    // tokens per tile
constexpr int kKB = kDQK / 64;             // 9 K-blocks of 64 dims (128 B of bf16)
constexpr int kQBlk = kHeads * 128;        // 12,288 B per Q K-block (96 rows)
constexpr int kLBlk = kNT * 128;           // 8,192 B per latent K-block (64 rows)
constexpr int kQBytes = kKB * kQBlk;       // 110,592
constexpr int kLatBytes = kKB * kLBlk;     // 73,728
constexpr int kPBytes = 128 * 128;         // 16,384
constexpr int kTcMlaThreads = 256;
constexpr uint32_t kSCol = 256;
constexpr int kSplitTiles = kSplitTok / kNT;  // tiles per split
constexpr size_t kTcMlaSmem = 1024 + kQBytes + kLatBytes + kPBytes + kSplitTok * 8 + kSplitTiles * 8 + 8 * 8 + 16;

struct MlaTc {
  const int32_t* block_table;
  const int32_t* ctx_lens;
  const int32_t* topk_idx;
  const uint8_t* lat_pool;
  int64_t lat_stride;
  int max_pages, num_pages, n_q, cap, K, splits, per_split;
  float sm_scale_log2, lat_scale;
  float* opart;
  float* lpart;
  int* err;
};

__device__ __forceinline__ uint32_t bf16x2_from_e4m3x2(uint16_t two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
  const __nv_bfloat162 b = __float22bfloat162_rn(f);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// 16 E4M3 bytes -> 16 bf16 (exact when scale == 1), as two 16-B chunks.
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t v, float scale) {
  const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
  const __nv_bfloat162 o = __floats2bfloat162_rn(f.x * scale, f.y * scale);
  return *reinterpret_cast<const uint32_t*>(&o);
}

__device__ __forceinline__ void expand_e4m3x16(const uint4 w, float scale, uint4& lo, uint4& hi) {
  lo.x = bf16x2_from_e4m3x2(uint16_t(w.x)); lo.y = bf16x2_from_e4m3x2(uint16_t(w.x >> 16));
  lo.z = bf16x2_from_e4m3x2(uint16_t(w.y)); lo.w = bf16x2_from_e4m3x2(uint16_t(w.y >> 16));
  hi.x = bf16x2_from_e4m3x2(uint16_t(w.z)); hi.y = bf16x2_from_e4m3x2(uint16_t(w.z >> 16));
  hi.z = bf16x2_from_e4m3x2(uint16_t(w.w)); hi.w = bf16x2_from_e4m3x2(uint16_t(w.w >> 16));
  if (scale != 1.0f) {
    lo.x = scale_bf16x2(lo.x, scale); lo.y = scale_bf16x2(lo.y, scale);
    lo.z = scale_bf16x2(lo.z, scale); lo.w = scale_bf16x2(lo.w, scale);
    hi.x = scale_bf16x2(hi.x, scale); hi.y = scale_bf16x2(hi.y, scale);
    hi.z = scale_bf16x2(hi.z, scale); hi.w = scale_bf16x2(hi.w, scale);
  }
}

__global__ void __launch_bounds__(kTcMlaThreads, 1) sparse_mla_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                                                                         MlaTc a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Qs = sm;
  uint8_t* LAT = Qs + kQBytes;
  uint8_t* Ps = LAT + kLatBytes;
  const uint8_t** rowptr = reinterpret_cast<const uint8_t**>(Ps + kPBytes);            // [kSplitTok]
  unsigned long long* vmask = reinterpret_cast<unsigned long long*>(rowptr + kSplitTok);  // [kSplitTiles]
  uint64_t* bars = reinterpret_cast<uint64_t*>(vmask + kSplitTiles);
  uint64_t* q_full = bars + 0;
  uint64_t* lat_full = bars + 1;
  uint64_t* lat_free = bars + 2;
  uint64_t* s_full = bars + 3;
  uint64_t* p_full = bars + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 8);

  const int half = blockIdx.x & 1, split = blockIdx.x >> 1, r = blockIdx.y;
  const int b = r / a.n_q, t = r - b * a.n_q;
  const int ctx = a.ctx_lens[b];
  const int L = (ctx < a.n_q || ctx > a.cap) ? 0 : ctx - a.n_q + t + 1;
  const int j0 = split * a.per_split;
  const int j1 = min(a.K, j0 + a.per_split);
  const int nt = j1 > j0 ? (j1 - j0 + kNT - 1) / kNT : 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* op = a.opart + (size_t(r) * a.splits + split) * kHeads * kDNope + half * 256;
  float* lp = a.lpart + (size_t(r) * a.splits + split) * kHeads;

  if (nt == 0) {  // a split past the top-k list: empty partial
    for (int i = threadIdx.x; i < kHeads * 256; i += blockDim.x) op[(i >> 8) * kDNope + (i & 255)] = 0.f;
    if (half == 0)
      for (int i = threadIdx.x; i < kHeads; i += blockDim.x) lp[i] = -INFINITY;
    return;
  }

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    ptx::mbar_init(lat_full, 4);
    ptx::mbar_init(lat_free, 1);
    ptx::mbar_init(s_full, 1);
    ptx::mbar_init(p_full, 3);
    ptx::fence_mbar_init();
  }
  if (warp == 3) {
    ptx::tmem_alloc(tmem_slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 3) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      ptx::mbar_arrive_expect_tx(q_full, kQBytes);
      for (int kb = 0; kb < kKB; ++kb) ptx::tma_load_2d(Qs + kb * kQBlk, &qmap, q_full, kb * 64, r * kHeads);
      if (!ptx::mbar_wait(q_full, 0)) ok = false;
      const uint32_t id_qk = ptx::idesc(1, 1, 128, kNT);
      const uint32_t id_pv = ptx::idesc(1, 1, 128, 256, 0, 1);
      const uint32_t q0 = ptx::smem_u32(Qs), l0 = ptx::smem_u32(LAT), p0 = ptx::smem_u32(Ps);
      for (int k = 0; k < nt && ok; ++k) {
        if (!ptx::mbar_wait(lat_full, uint32_t(k) & 1u)) { ok = false; break; }
        ptx::tc_fence_after();
        for (int kb = 0; kb < kKB; ++kb)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            ptx::mma_f16(tmem + kSCol, ptx::sdesc_sw128(q0 + kb * kQBlk + kk * 32),
                         ptx::sdesc_sw128(l0 + kb * kLBlk + kk * 32), id_qk, (kb | kk) ? 1u : 0u);
        ptx::mma_commit(s_full);
        if (!ptx::mbar_wait(p_full, uint32_t(k) & 1u)) { ok = false; break; }
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kNT / 16; ++kk)
          ptx::mma_f16(tmem, ptx::sdesc_sw128(p0 + kk * 32),
                       ptx::sdesc_sw128_mn(l0 + 4 * half * kLBlk + kk * 16 * 128, kLBlk, 1024), id_pv,
                       (k > 0 || kk > 0) ? 1u : 0u);
        ptx::mma_commit(lat_free);
      }
      if (!ok) atomicOr(a.err, DSA_DEVERR_TIMEOUT);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ converters
    const int ct = threadIdx.x - 128;
    // Resolve every selected slot of the split once (slot -> page -> row address);
    // the loads are independent, so their latency overlaps the Q copy.
    for (int jj = ct; jj < nt * kNT; jj += 128) {
      const int j = j0 + jj;
      const uint8_t* rp = nullptr;
      if (j < j1) {
        const int sidx = a.topk_idx[size_t(r) * a.K + j];
        if (sidx >= 0 && sidx < L) {
          const int pg = a.block_table[size_t(b) * a.max_pages + sidx / kPage];
          if (pg >= 0 && pg < a.num_pages)
            rp = a.lat_pool + size_t(pg) * a.lat_stride + size_t(sidx % kPage) * kLatRowFp8;
          else
            atomicOr(a.err, DSA_DEVERR_BLOCK_TABLE);
        } else if (sidx != -1) {
          atomicOr(a.err, DSA_DEVERR_TOPK_INDEX);
        }
      }
      rowptr[jj] = rp;
      const unsigned m = __ballot_sync(0xffffffffu, rp != nullptr);
      if (lane == 0) reinterpret_cast<uint32_t*>(vmask)[jj >> 5] = m;
    }
    ptx::named_bar_sync(1, 128);
    uint4 buf[18];
    bool ok = true;
    for (int k = -1; k < nt; ++k) {
      if (k >= 0) {
        if (k > 0 && !ptx::mbar_wait(lat_free, uint32_t(k - 1) & 1u)) ok = false;
        if (ok) {
#pragma unroll
          for (int u = 0; u < 18; ++u) {
            const int pc = ct + 128 * u;
            const int jj = pc / 36, c16 = pc % 36;
            const int kb = c16 >> 2, c = (c16 & 3) * 2;
            uint4 lo, hi;
            expand_e4m3x16(buf[u], a.lat_scale, lo, hi);
            uint8_t* rowb = LAT + kb * kLBlk + jj * 128;
            *reinterpret_cast<uint4*>(rowb + ((c ^ (jj & 7)) << 4)) = lo;
            *reinterpret_cast<uint4*>(rowb + (((c + 1) ^ (jj & 7)) << 4)) = hi;
          }
          ptx::fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(lat_full);
        if (!ok) break;
      }
      if (k + 1 < nt) {
        // start tile k+1's loads; they land while tile k is multiplied
        const uint8_t* const* rp = rowptr + (k + 1) * kNT;
#pragma unroll
        for (int u = 0; u < 18; ++u) {
          const int pc = ct + 128 * u;
          const uint8_t* p = rp[pc / 36];
          buf[u] = p ? __ldg(reinterpret_cast<const uint4*>(p + (pc % 36) * 16)) : make_uint4(0, 0, 0, 0);
        }
      }
    }
    if (!ok) atomicOr(a.err, DSA_DEVERR_TIMEOUT);
  } else if (warp < 3) {
    // ------------------------------------------------------------ softmax / epilogue
    const int h = warp * 32 + lane;
    const uint32_t lane_base = uint32_t(warp * 32) << 16;
    float m_use = -INFINITY, l = 0.f;
    bool ok = true;
    for (int k = 0; k < nt; ++k) {
      // lat_full orders the converters' validity mask before this read (they
      // cannot refill the tile before this row's P has been consumed)
      if (!ptx::mbar_wait(lat_full, uint32_t(k) & 1u)) { ok = false; break; }
      if (!ptx::mbar_wait(s_full, uint32_t(k) & 1u)) { ok = false; break; }
      ptx::tc_fence_after();
      float sv[64];
      ptx::tmem_ld32(tmem + lane_base + kSCol, *reinterpret_cast<float(*)[32]>(&sv[0]));
      ptx::tmem_ld32(tmem + lane_base + kSCol + 32, *reinterpret_cast<float(*)[32]>(&sv[32]));
      const unsigned long long vm = vmask[k];
      float tmax = -INFINITY;
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        sv[i] = ((vm >> i) & 1ull) ? sv[i] * a.sm_scale_log2 : -INFINITY;
        tmax = fmaxf(tmax, sv[i]);
      }
      bool need = false;
      float alpha = 1.f;
      if (m_use == -INFINITY) {
        m_use = tmax;
      } else if (tmax > m_use + 8.f) {
        need = true;
        alpha = exp2f(m_use - tmax);
        m_use = tmax;
      }
      if (__any_sync(0xffffffffu, need)) {
        // O (this warp's 32 rows, 256 columns) *= alpha; the previous PV is complete
        // because this tile's latents were written only after it finished.
        l *= alpha;
#pragma unroll 1
        for (int c = 0; c < 256; c += 32) {
          float o[32];
          ptx::tmem_ld32(tmem + lane_base + c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          ptx::tmem_st32(tmem + lane_base + c, o);
        }
      }
      float psum = 0.f;
      uint8_t* prow = Ps + h * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = 8 * c + 2 * e;
          const float p0 = m_use == -INFINITY ? 0.f : exp2f(sv[i] - m_use);
          const float p1 = m_use == -INFINITY ? 0.f : exp2f(sv[i + 1] - m_use);
          psum += p0 + p1;
          const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
          pk[e] = *reinterpret_cast<const uint32_t*>(&pb);
        }
        *reinterpret_cast<uint4*>(prow + ((c ^ (h & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      l += psum;
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(p_full);
    }
    if (ok && !ptx::mbar_wait(lat_free, uint32_t(nt - 1) & 1u)) ok = false;
    if (!ok) {
      if (lane == 0) atomicOr(a.err, DSA_DEVERR_TIMEOUT);
    } else {
      ptx::tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      float* orow = op + size_t(h) * kDNope;
#pragma unroll 1
      for (int c = 0; c < 256; c += 32) {
        float o[32];
        ptx::tmem_ld32(tmem + lane_base + c, o);
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(orow + c + i) = make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
      }
      if (half == 0) lp[h] = l > 0.f ? (m_use + log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 3) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
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
  CUtensorMap qmap;
  {
    const uint64_t dims[2] = {uint64_t(kDQK), uint64_t(L.rows) * kHeads};
    const uint64_t strides[1] = {uint64_t(kDQK) * 2};
    const uint32_t box[2] = {64, uint32_t(kHeads)};
    if (!encode_map(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, 2, dims, strides, box, true))
      return cudaErrorInvalidValue;
  }
  MlaTc t;
  t.block_table = block_table;
  t.ctx_lens = ctx_lens;
  t.topk_idx = topk_idx;
  t.lat_pool = static_cast<const uint8_t*>(lat_pool);
  t.lat_stride = p.lat_page_stride;
  t.max_pages = p.max_pages_per_req;
  t.num_pages = p.num_pages;
  t.n_q = p.n_q;
  t.cap = L.cap;
  t.K = p.topk;
  t.splits = L.splits;
  t.per_split = kSplitTok;
  t.sm_scale_log2 = p.softmax_scale * 1.4426950408889634f;
  t.lat_scale = p.latent_scale;
  t.opart = reinterpret_cast<float*>(ws + L.opart);
  t.lpart = reinterpret_cast<float*>(ws + L.lpart);
  t.err = reinterpret_cast<int*>(ws + L.err);
  cudaError_t e = cudaFuncSetAttribute(sparse_mla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(kTcMlaSmem));
  if (e != cudaSuccess) return e;
  dim3 grid(2 * L.splits, L.rows);
  sparse_mla_tc_kernel<<<grid, kTcMlaThreads, kTcMlaSmem, st>>>(qmap, t);
  dim3 g2(L.rows, kHeads);
  mla_combine_kernel<<<g2, 256, 0, st>>>(t.opart, t.lpart, L.splits, static_cast<__nv_bfloat16*>(out), lse);
  return cudaGetLastError();
}

}  // namespace dsa
