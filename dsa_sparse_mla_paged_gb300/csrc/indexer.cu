// Stage 1: the lightning indexer over the paged FP8 index-key cache.
//
// score(t, s) = sum_h w'_h * max(0, scale_s * (q8_h . k_s)), with the indexer
// query quantised to E4M3 per head and its scale folded into the head weights
// (vLLM, "vLLM 为 Kimi K3.1 Pro 提供 Day-0 支持": sections "K3.1 Pro 中的稀疏注意力"
// and "低延迟解码：融合的 DSA 解码路径").
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <cstring>

#include "dsa_internal.cuh"
#include "sm103_ptx.cuh"

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
                                                          float* __restrict__ wq,
                                                          const int32_t* __restrict__ ctx_lens, int units,
                                                          UnitMap map, int cap, int* __restrict__ tile_prefix,
                                                          int* err) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (row == gridDim.x - 1) {
    build_tile_plan<128>(ctx_lens, units, map, cap, tile_prefix, err);
    return;
  }
  // all eight heads' loads first (independent), then the per-head reductions
  uint2 raw[8];
#pragma unroll
  for (int hh = 0; hh < 8; ++hh)
    raw[hh] = *reinterpret_cast<const uint2*>(q_idx + (size_t(row) * kIdxHeads + warp * 8 + hh) * kIdxDim + lane * 4);
  const float wl = lane < 8 ? w[size_t(row) * kIdxHeads + warp * 8 + lane] : 0.f;
#pragma unroll
  for (int hh = 0; hh < 8; ++hh) {
    const int h = warp * 8 + hh;
    const size_t base = (size_t(row) * kIdxHeads + h) * kIdxDim + lane * 4;
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&raw[hh].x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&raw[hh].y);
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
    const float wh = __shfl_sync(0xffffffffu, wl, hh);
    if (lane == 0) wq[size_t(row) * kIdxHeads + h] = __fmul_rn(wh, __fdiv_rn(m, 448.0f));
  }
}

cudaError_t launch_idx_q_quant(const dsa_params_t& p, const WsLayout& L, char* ws, const void* q_idx,
                               const float* w, const int32_t* ctx_lens, cudaStream_t st, int world, int rank) {
  const UnitMap map = unit_map(p.n_q, world, rank);
  return launch_pdl(idx_q_quant_kernel, dim3(L.rows + 1), dim3(128), 0, st,
                    static_cast<const __nv_bfloat16*>(q_idx), w, reinterpret_cast<uint8_t*>(ws + L.q8),
                    reinterpret_cast<float*>(ws + L.wq), ctx_lens, p.batch * map.groups, map, L.cap,
                    reinterpret_cast<int*>(ws + L.tiles), reinterpret_cast<int*>(ws + L.err));
}

// ---------------------------------------------------------------------------
// Tensor-core scorer (sm_103a): a persistent CTA per SM walks a contiguous
// range of the batch's 128-token tiles (two pages each), so every CTA streams
// the same number of keys whatever the context lengths ("key-balanced").
//   warp 0     : TMA producer -- key pages (128-B swizzled) and their scales,
//                lane g issuing tile g of a stage, and the request's FP8
//                query when the request changes
//   warp 1     : TMEM owner and MMA issuer -- D[128 tok x 32*n_q] =
//                keys[128 x 128] * q8^T, four K=32 FP8 MMAs per tile
//   warps 2..5 : epilogue -- one token row per thread out of TMEM,
//                score = sum_h w'_h * max(scale * D_h, 0), coalesced store
// MXFP4 keys (68 B: 128 E2M1 + one E8M0 exponent per 32) take the same MMA and
// epilogue. The producer then bulk-copies raw page pairs into a ring of their
// own, and four converter warps (after the epilogue warps) rewrite each token
// as E4M3 values k * 2^(6 + e_b - e_max) (the token's largest block lands in
// [32, 384], below E4M3's 448) plus a per-token scale 2^(e_max - 133): exact
// whenever the token's block exponents lie within 14 of one another (E4M3
// reaches 2^-9); beyond that a small block's values round to the nearest
// multiple of 2^-9, an error of at most 2^-10 x 2^(e_max - 133) per key value.
// ---------------------------------------------------------------------------
namespace {

constexpr int kTcThreads = 192;    // FP8 keys
constexpr int kMxConvThreads = 128;  // MXFP4 keys: 4 converter warps after the epilogue warps
constexpr int kMxPageBytes = kPage * (kIdxDim / 2 + kIdxDim / 32);  // 4,352
constexpr int kMxRawTile = 2 * kMxPageBytes;
constexpr int kTileTok = 128;
constexpr int kKeyTileBytes = kTileTok * kIdxDim;   // 16 KB
constexpr int kScaleTileBytes = kTileTok * 4;       // 512 B

struct IdxTc {
  const int32_t* block_table;
  const int32_t* ctx_lens;
  const int32_t* tile_prefix;
  const float* wq;
  const uint8_t* key_pool;
  float* scores;
  uint32_t* gmax;     // [rows][gstride] order key of the largest score of each 32 tokens (for the top-k bound)
  uint32_t* gmax128;  // [rows][g128stride] the same per 128 tokens, by atomic max; null: not kept
  int gstride, g128stride;
  int64_t score_stride;
  int64_t key_page_stride;
  int units, n_q, max_pages, num_pages, stages, nacc, group, ncol, tmem_cols;  // n_q: rows per unit
  int raw_slots;  // MXFP4: raw page-pair slots
  UnitMap map;
  int* err;
};

// Unit u: request, first query row (global), valid rows, and context (that of
// its last row; the rows before it see fewer tokens).
struct UnitInfo {
  int b, row0, valid, ctx;
};

__device__ __forceinline__ int unit_req(const IdxTc& a, int u) { return u / a.map.groups; }

__device__ __forceinline__ UnitInfo unit_info(const IdxTc& a, int u) {
  UnitInfo x;
  x.b = u / a.map.groups;
  const int first = unit_first_row(a.map, u - x.b * a.map.groups);
  x.row0 = x.b * a.map.rows_per_req + first;
  x.valid = min(a.map.gsz, a.map.rows_per_req - first);
  x.ctx = a.ctx_lens[x.b] - a.map.rows_per_req + first + x.valid;
  return x;
}

struct TileWalk {
  int b, j;        // request, tile within the request
  long long t;     // global tile index
  int end_b;       // global tile index where request b ends
};

__device__ __forceinline__ void walk_start(const IdxTc& a, long long t0, TileWalk& w) {
  int lo = 0, hi = a.units - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a.tile_prefix[mid] > t0) hi = mid; else lo = mid + 1;
  }
  w.b = lo;
  w.end_b = a.tile_prefix[lo];
  w.t = t0;
  w.j = int(t0 - (lo ? a.tile_prefix[lo - 1] : 0));
}

__device__ __forceinline__ void walk_next(const IdxTc& a, TileWalk& w) {
  ++w.t;
  ++w.j;
  while (w.t >= w.end_b && w.b + 1 < a.units) {
    ++w.b;
    w.j = 0;
    w.end_b = a.tile_prefix[w.b];
  }
}

// Block-table entries of one tile as loaded: range-checked only where they
// are used, so the loads of a look-ahead stay in flight.
struct TilePages {
  int b, pg0, pg1, two;  // two: the tile holds a second page
};

__device__ __forceinline__ int page_or_zero(const IdxTc& a, int pg) {
  if (pg < 0 || pg >= a.num_pages) {
    atomicOr(a.err, DSA_DEVERR_BLOCK_TABLE);
    return 0;
  }
  return pg;
}

// Move the walk `n` tiles forward; `np` tracks the pages of the walk's request.
__device__ __forceinline__ void advance_walk(const IdxTc& a, TileWalk& w, int& np, int n) {
  w.t += n;
  w.j += n;
  if (w.t >= w.end_b) {
    const int b0 = w.b;
    while (w.t >= w.end_b && w.b + 1 < a.units) {
      ++w.b;
      w.end_b = a.tile_prefix[w.b];
    }
    w.j = int(w.t - (w.b ? a.tile_prefix[w.b - 1] : 0));
    if (w.b != b0) np = (unit_info(a, w.b).ctx + kPage - 1) / kPage;
  }
}

// Lane `lane` of the producer warp: the pages of tile (w.t + lane).
__device__ __forceinline__ TilePages tile_pages(const IdxTc& a, const TileWalk& w, int np, long long t_end,
                                                int lane) {
  TilePages tp{w.b, 0, 0, 0};
  if (w.t + lane >= t_end) return tp;
  TileWalk x = w;
  int xnp = np;
  if (lane) advance_walk(a, x, xnp, lane);
  tp.b = x.b;
  const int lp0 = 2 * x.j;
  const int32_t* row = a.block_table + size_t(unit_req(a, x.b)) * a.max_pages;
  tp.pg0 = row[lp0];
  tp.two = lp0 + 1 < xnp;
  if (tp.two) tp.pg1 = row[lp0 + 1];
  return tp;
}

// Epilogue position inside a stage: tile g, query row t.
struct EpiState {
  int g, t;
};

// Step the epilogue position past one block (another warpgroup reduces it).
__device__ __forceinline__ void epi_skip(const IdxTc& a, TileWalk& w, EpiState& e) {
  if (++e.t == a.n_q) {
    e.t = 0;
    ++e.g;
    walk_next(a, w);
  }
}

__device__ __forceinline__ void epi_store(const IdxTc& a, float sum, int rowt, int lane, TileWalk& w, EpiState& e,
                                          const UnitInfo& ui) {
  const int tok = w.j * kTileTok + rowt;
  const int Lt = ui.ctx - ui.valid + e.t + 1;
  // a short last group computes padding rows past `valid`: never stored
  const bool keep = e.t < ui.valid && tok < Lt && tok < a.score_stride;
  if (keep) a.scores[(size_t(ui.row0) + e.t) * a.score_stride + tok] = sum;
  // the warp's 32 tokens are one group: the key of their largest stored score
  // (kept only for the fused step's top-k, which takes its bound from them)
  if (a.gmax) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, keep ? score_order_key(sum) : 0u);
    if (lane == 0 && m != 0u) {
      a.gmax[(size_t(ui.row0) + e.t) * a.gstride + (tok >> 5)] = m;
      atomicMax(a.gmax128 + (size_t(ui.row0) + e.t) * a.g128stride + (tok >> 7), m);
    }
  }
  epi_skip(a, w, e);
}

// Packed fp32 pairs (one instruction for two lanes of work; each half rounds
// as its scalar op would).
__device__ __forceinline__ unsigned long long f2_pack(float x, float y) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(unsigned long long r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// Several query rows with several epilogue warpgroups: the warp keeps the
// current unit's head weights in its own shared-memory copy (wme[t][h]), read
// four at a time by every lane, and reduces w'_h * max(scale * d_h, 0) in
// packed pairs (heads 4i + {0, 1} and 4i + {2, 3}, each half rounding as its
// scalar op would). (Factoring a non-negative key scale out of the head sum, as
// the one-row epilogue does, measured slower here: one code path is smaller.)
__device__ __forceinline__ void epi_block_wide(const IdxTc& a, const float (&v)[32], const float (&sc)[4], int rowt,
                                               int lane, TileWalk& w, EpiState& e, int& cur_b, UnitInfo& ui,
                                               float* wme) {
  if (w.b != cur_b) {
    cur_b = w.b;
    ui = unit_info(a, w.b);
    __syncwarp();  // every lane is done with the previous unit's weights
#pragma unroll
    for (int t = 0; t < kMaxNQ; ++t)
      wme[t * kIdxHeads + lane] = t < ui.valid ? a.wq[(size_t(ui.row0) + t) * kIdxHeads + lane] : 0.f;
    __syncwarp();
  }
  float scale = sc[0];
#pragma unroll
  for (int g = 1; g < 4; ++g)
    if (e.g == g) scale = sc[g];
  const float4* wrow = reinterpret_cast<const float4*>(wme + e.t * kIdxHeads);
  unsigned long long p01 = f2_pack(0.f, 0.f), p23 = p01;  // partial sums of heads 4i + {0, 1} and 4i + {2, 3}
  const unsigned long long s2 = f2_pack(scale, scale);
#pragma unroll
  for (int i = 0; i < kIdxHeads / 4; ++i) {
    const float4 w4 = wrow[i];
    float2 x = f2_unpack(f2_mul(s2, f2_pack(v[4 * i], v[4 * i + 1])));
    float2 y = f2_unpack(f2_mul(s2, f2_pack(v[4 * i + 2], v[4 * i + 3])));
    p01 = f2_fma(f2_pack(w4.x, w4.y), f2_pack(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)), p01);
    p23 = f2_fma(f2_pack(w4.z, w4.w), f2_pack(fmaxf(y.x, 0.f), fmaxf(y.y, 0.f)), p23);
  }
  const float2 a01 = f2_unpack(p01), a23 = f2_unpack(p23);
  const float sum = (a01.x + a01.y) + (a23.x + a23.y);
  epi_store(a, sum, rowt, lane, w, e, ui);
}

// Reduce one 32-column accumulator block (tile e.g, query row e.t) of this
// thread's token row and store the score, then step to the next block.
__device__ __forceinline__ void epi_block(const IdxTc& a, const float (&v)[32], const float (&sc)[4], int rowt,
                                          int lane, TileWalk& w, EpiState& e, int& cur_b, UnitInfo& ui,
                                          float (&wl)[kMaxNQ], float (&wr)[kIdxHeads]) {
  if (w.b != cur_b) {
    cur_b = w.b;
    ui = unit_info(a, w.b);
    if (a.n_q == 1) {
      const float4* src = reinterpret_cast<const float4*>(a.wq + size_t(ui.row0) * kIdxHeads);
#pragma unroll
      for (int i = 0; i < kIdxHeads / 4; ++i) {
        const float4 f = src[i];
        wr[4 * i] = f.x; wr[4 * i + 1] = f.y; wr[4 * i + 2] = f.z; wr[4 * i + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int t = 0; t < kMaxNQ; ++t) wl[t] = t < ui.valid ? a.wq[(size_t(ui.row0) + t) * kIdxHeads + lane] : 0.f;
    }
  }
  float scale = sc[0], wt = wl[0];
#pragma unroll
  for (int g = 1; g < 4; ++g)
    if (e.g == g) scale = sc[g];
#pragma unroll
  for (int t = 1; t < kMaxNQ; ++t)
    if (e.t == t) wt = wl[t];
  // four independent partial sums (heads h = 4i + j), added pairwise: a short
  // dependency chain per block. One query row: every thread holds all 32 head
  // weights; several rows: lane h holds w'_h of each row and shares it.
  // (a key scale >= 0 leaves the head sum: max(scale * d, 0) = scale * max(d, 0))
  float part[4] = {0.f, 0.f, 0.f, 0.f};
  const bool factor = scale >= 0.f;
  const float hs = factor ? 1.f : scale;
  if (a.n_q == 1) {
#pragma unroll
    for (int h = 0; h < kIdxHeads; ++h) part[h & 3] = fmaf(wr[h], fmaxf(hs * v[h], 0.f), part[h & 3]);
  } else {
#pragma unroll
    for (int h = 0; h < kIdxHeads; ++h)
      part[h & 3] = fmaf(__shfl_sync(0xffffffffu, wt, h), fmaxf(hs * v[h], 0.f), part[h & 3]);
  }
  const float hsum = (part[0] + part[1]) + (part[2] + part[3]);
  const float sum = factor ? scale * hsum : hsum;
  epi_store(a, sum, rowt, lane, w, e, ui);
}


// One MXFP4 token (64 B of E2M1 pairs, element 2i in the low nibble; 4 E8M0
// exponents) -> 128 E4M3 values v * 2^(6 + e_b - e_max) into its 128-B swizzled
// row, and its scale 2^(e_max - 133).
__device__ __forceinline__ void mx_convert_row(const uint8_t* vals, uint32_t e4, uint8_t* row, int r, float* scale) {
  const uint32_t e0 = e4 & 0xFFu, e1 = (e4 >> 8) & 0xFFu, e2 = (e4 >> 16) & 0xFFu, e3 = e4 >> 24;
  const uint32_t emax = max(max(e0, e1), max(e2, e3));
  // 2^(emax - 133): an fp32 normal for emax >= 7, a subnormal (bit emax + 16) below
  *scale = emax == 255u ? __uint_as_float(0x7FC00000u)
                        : emax >= 7u ? __uint_as_float((emax - 6u) << 23) : __uint_as_float(1u << (emax + 16u));
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint32_t eb = (e4 >> (8 * b)) & 0xFFu;
    const uint32_t d = emax - eb;  // 2^(6 - d) as f16 (normal to d = 20, subnormal to d = 30, zero below)
    const unsigned short mbits = d <= 20u ? (unsigned short)((21u - d) << 10)
                                 : d <= 30u ? (unsigned short)(1u << (30u - d)) : (unsigned short)0;
    const __half2 m2 = __halves2half2(__ushort_as_half(mbits), __ushort_as_half(mbits));
    const uint4 v = *reinterpret_cast<const uint4*>(vals + 16 * b);
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int jp = 0; jp < 2; ++jp) {
        uint32_t packed = 0;
#pragma unroll
        for (int j = 2 * jp; j < 2 * jp + 2; ++j) {
          __half2_raw h = __nv_cvt_fp4x2_to_halfraw2(
              static_cast<__nv_fp4x2_storage_t>((words[i] >> (8 * j)) & 0xFFu), __NV_E2M1);
          const __half2 x = __hmul2(*reinterpret_cast<const __half2*>(&h), m2);
          const __nv_fp8x2_storage_t f8 =
              __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&x), __NV_SATFINITE, __NV_E4M3);
          packed |= uint32_t(f8) << (16 * (j & 1));
        }
        o[(i & 1) * 2 + jp] = packed;
      }
      if (i & 1) {
        // words i-1, i: 16 E4M3 bytes = output chunk 2b + i/2
        const int c = 2 * b + (i >> 1);
        *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
}

// kEwg epilogue warpgroups (FP8 keys): 1 for one query row, where the kernel
// is bound by HBM; 2 when a unit has several rows (decode with n_q > 1,
// prefill), where the reduction of 32 x rows columns per token is the work.
template <bool kMx, int kEwg>
__global__ void __launch_bounds__(64 + 128 * kEwg + (kMx ? kMxConvThreads : 0), (kMx || kEwg > 1) ? 1 : 2)
    indexer_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap, IdxTc a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.stages, NA = a.nacc, G = a.group;
  const int qbytes = a.n_q * kIdxHeads * kIdxDim;
  uint8_t* keys = smem;                                           // S x G x 16 KB
  uint8_t* qbuf = keys + size_t(S) * G * kKeyTileBytes;           // 2 x qbytes
  float* wsm = reinterpret_cast<float*>(qbuf + 2 * qbytes);       // wide epilogue: 8 warps x 8 rows x 32 heads
  float* scl = wsm + (kEwg > 1 ? 4 * kEwg * kMaxNQ * kIdxHeads : 0);  // S x G x 128
  uint8_t* raw = reinterpret_cast<uint8_t*>(scl + size_t(S) * G * kTileTok);  // MXFP4: R x 8,704 B
  const int R = kMx ? a.raw_slots : 0;
  uint64_t* bars = reinterpret_cast<uint64_t*>(raw + size_t(R) * kMxRawTile);
  uint64_t* full = bars;
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + NA;
  uint64_t* qfull = tempty + NA;
  uint64_t* qempty = qfull + 2;
  uint64_t* rfull = qempty + 2;   // MXFP4 raw slots: landed
  uint64_t* rempty = rfull + R;   // MXFP4 raw slots: converted
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rempty + R);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) { ptx::mbar_init(full + i, kMx ? 4 : 1); ptx::mbar_init(empty + i, 1 + 4 * kEwg); }
    for (int i = 0; i < R; ++i) { ptx::mbar_init(rfull + i, 1); ptx::mbar_init(rempty + i, 4); }
    for (int i = 0; i < NA; ++i) { ptx::mbar_init(tfull + i, 1); ptx::mbar_init(tempty + i, 4 * kEwg); }
    for (int i = 0; i < 2; ++i) { ptx::mbar_init(qfull + i, 1); ptx::mbar_init(qempty + i, 1); }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, a.tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the tile plan and the query come from the previous kernel
  const long long T = a.tile_prefix[a.units - 1];
  const long long t_begin = T * blockIdx.x / gridDim.x;
  const long long t_end = T * (blockIdx.x + 1) / gridDim.x;

  auto fail = [&]() {
    *abort_flag = 1;
    atomicOr(a.err, DSA_DEVERR_TIMEOUT);
  };

  // Tiles are consumed in order; every G consecutive tiles of the CTA's range
  // share one pipeline stage (one barrier round trip per G x 16.5 KB).
  if (t_begin < t_end) {
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      // The whole warp looks 32 tiles ahead: lane i loads the block-table
      // entries of tile (chunk + i) one chunk before their copies are issued,
      // so no copy waits on a dependent global load.
      if (lane == 0) {
        if (!kMx) ptx::prefetch_tmap(&kmap);
        ptx::prefetch_tmap(&qmap);
      }
      int rs = 0;         // MXFP4 raw slot
      uint32_t rph = 0;   // its phase bit
      // keys are read once: keep them from pushing the score rows (read next
      // by the top-k passes) out of L2
      const uint64_t pol = ptx::policy_evict_first();
      TileWalk base;
      walk_start(a, t_begin, base);
      int base_np = (unit_info(a, base.b).ctx + kPage - 1) / kPage;
      TilePages cur = tile_pages(a, base, base_np, t_end, lane);
      int cur_b = -1, nq = -1;
      int s = 0;          // ring stage
      uint32_t ph = 0;    // its phase bit
      bool ok = true;
      for (long long tc = t_begin; tc < t_end && ok; tc += 32) {
        TileWalk nb = base;
        int nb_np = base_np;
        advance_walk(a, nb, nb_np, 32);
        const TilePages nxt = tile_pages(a, nb, nb_np, t_end, lane);
        const int n = int(t_end - tc < 32 ? t_end - tc : 32);
        for (int i0 = 0; i0 < n; i0 += G) {
          const int ng = min(G, n - i0);
          if constexpr (kMx) {
            // raw page pairs, one slot per tile; lanes 0 / 1 copy page 0 / 1
            for (int g = 0; g < ng; ++g) {
              const int pg0 = __shfl_sync(0xffffffffu, cur.pg0, i0 + g);
              const int pg1 = __shfl_sync(0xffffffffu, cur.pg1, i0 + g);
              const int two = __shfl_sync(0xffffffffu, cur.two, i0 + g);
              if (lane == 0) {
                if (*abort_flag) ok = false;
                if (ok && !ptx::mbar_wait(rempty + rs, rph ^ 1u)) { fail(); ok = false; }
                if (ok) ptx::mbar_arrive_expect_tx(rfull + rs, (two ? 2u : 1u) * kMxPageBytes);
              }
              ok = __shfl_sync(0xffffffffu, int(ok), 0) != 0;
              if (!ok) break;
              if (lane < 1 + two) {
                const int pg = page_or_zero(a, lane ? pg1 : pg0);
                ptx::bulk_load_hint(raw + size_t(rs) * kMxRawTile + lane * kMxPageBytes,
                                    a.key_pool + size_t(pg) * a.key_page_stride, kMxPageBytes, rfull + rs, pol);
              }
              if (++rs == R) { rs = 0; rph ^= 1u; }
            }
            if (!ok) break;
          } else {
          uint32_t bytes = 0;
          for (int g = 0; g < ng; ++g)
            bytes += (__shfl_sync(0xffffffffu, cur.two, i0 + g) ? 2u : 1u) * (kPage * kIdxDim + kPage * 4);
          if (lane == 0) {
            if (*abort_flag) ok = false;
            if (ok && !ptx::mbar_wait(empty + s, ph ^ 1u)) { fail(); ok = false; }
          }
          ok = __shfl_sync(0xffffffffu, int(ok), 0) != 0;
          if (!ok) break;
          if (lane == 0) ptx::mbar_arrive_expect_tx(full + s, bytes);
          // lanes 2g and 2g+1 issue the copies of tile g (keys and scales of its
          // first and second page; measured 2% faster than one lane per tile);
          // all key copies of the stage go out before its query loads, since a
          // query slot is released by the MMA warp only once it has this stage
          // in hand
          {
            const int gg = lane >> 1, page = lane & 1;
            const int src = i0 + min(gg, ng - 1);
            const int pg0 = __shfl_sync(0xffffffffu, cur.pg0, src);
            const int pg1 = __shfl_sync(0xffffffffu, cur.pg1, src);
            const int two = __shfl_sync(0xffffffffu, cur.two, src);
            if (gg < ng && (page == 0 || two)) {
              const int p = page_or_zero(a, page ? pg1 : pg0);
              uint8_t* kdst = keys + (size_t(s) * G + gg) * kKeyTileBytes + page * kPage * kIdxDim;
              float* sdst = scl + (size_t(s) * G + gg) * kTileTok + page * kPage;
              ptx::tma_load_3d_hint(kdst, &kmap, full + s, 0, 0, p, pol);
              ptx::bulk_load_hint(sdst, a.key_pool + size_t(p) * a.key_page_stride + kPage * kIdxDim, kPage * 4,
                                  full + s, pol);
            }
          }
          }
          for (int g = 0; g < ng; ++g) {
            const int b = __shfl_sync(0xffffffffu, cur.b, i0 + g);
            if (lane == 0 && b != cur_b) {
              ++nq;
              const int slot = nq & 1;
              if (!ptx::mbar_wait(qempty + slot, (uint32_t(nq >> 1) & 1u) ^ 1u)) { fail(); ok = false; }
              if (ok) {
                ptx::mbar_arrive_expect_tx(qfull + slot, qbytes);
                ptx::tma_load_2d(qbuf + slot * qbytes, &qmap, qfull + slot, 0, unit_info(a, b).row0 * kIdxHeads);
                cur_b = b;
              }
            }
          }
          if (++s == S) { s = 0; ph ^= 1u; }
          ok = __shfl_sync(0xffffffffu, int(ok), 0) != 0;
          if (!ok) break;
        }
        base = nb;
        base_np = nb_np;
        cur = nxt;
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        const uint32_t id = ptx::idesc(0, 0, kTileTok, uint32_t(a.n_q * kIdxHeads));
        TileWalk w;
        walk_start(a, t_begin, w);
        int cur_b = -1, nq = -1;
        int s = 0, acc = 0;
        uint32_t ph = 0, aph = 0;
        bool ok = true;
        for (long long t0 = t_begin; t0 < t_end && ok; t0 += G) {
          const int ng = int(t_end - t0 < G ? t_end - t0 : G);
          if (*abort_flag || !ptx::mbar_wait(tempty + acc, aph ^ 1u) || !ptx::mbar_wait(full + s, ph)) {
            fail();
            break;
          }
          ptx::tc_fence_after();
          for (int g = 0; g < ng; ++g, walk_next(a, w)) {
            if (w.b != cur_b) {
              if (cur_b >= 0) ptx::mma_commit(qempty + (nq & 1));
              ++nq;
              if (!ptx::mbar_wait(qfull + (nq & 1), uint32_t(nq >> 1) & 1u)) { fail(); ok = false; break; }
              ptx::tc_fence_after();
              cur_b = w.b;
            }
            const uint32_t a_base = ptx::smem_u32(keys + (size_t(s) * G + g) * kKeyTileBytes);
            const uint32_t b_base = ptx::smem_u32(qbuf + (nq & 1) * qbytes);
            const uint32_t d = tmem + uint32_t((acc * G + g) * a.ncol);
            // tile-major order: the four K steps of a tile back to back (measured
            // faster than interleaving the tiles of a stage)
#pragma unroll
            for (int kk = 0; kk < kIdxDim / 32; ++kk)
              ptx::mma_f8f6f4(d, ptx::sdesc_sw128(a_base + kk * 32), ptx::sdesc_sw128(b_base + kk * 32), id,
                              kk > 0 ? 1u : 0u);
          }
          if (!ok) break;
          ptx::mma_commit(empty + s);
          ptx::mma_commit(tfull + acc);
          if (++s == S) { s = 0; ph ^= 1u; }
          if (++acc == NA) { acc = 0; aph ^= 1u; }
        }
      }
    } else if (kMx && warp >= 2 + 4 * kEwg) {
      // ------------------------------------------------------------ MXFP4 converters
      // thread ct rewrites token row ct of every tile (page ct / 64, slot ct % 64)
      const int ct = threadIdx.x - (64 + 128 * kEwg);
      const int half = ct >> 6, slot = ct & 63;
      int rs = 0, s = 0, g = 0;
      uint32_t rph = 0, ph = 0;
      for (long long t = t_begin; t < t_end; ++t) {
        if (*abort_flag) break;
        if (g == 0 && !ptx::mbar_wait(empty + s, ph ^ 1u)) { fail(); break; }
        if (!ptx::mbar_wait(rfull + rs, rph)) { fail(); break; }
        const uint8_t* page = raw + size_t(rs) * kMxRawTile + half * kMxPageBytes;
        mx_convert_row(page + slot * (kIdxDim / 2),
                       *reinterpret_cast<const uint32_t*>(page + kPage * (kIdxDim / 2) + 4 * slot),
                       keys + (size_t(s) * G + g) * kKeyTileBytes + ct * kIdxDim, ct,
                       scl + (size_t(s) * G + g) * kTileTok + ct);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(rempty + rs);
        if (++rs == R) { rs = 0; rph ^= 1u; }
        if (++g == G || t + 1 == t_end) {
          ptx::fence_proxy_async_smem();  // the MMA reads the keys through the async proxy
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(full + s);
          g = 0;
          if (++s == S) { s = 0; ph ^= 1u; }
        }
      }
    } else if (warp >= 2 && warp < 2 + 4 * kEwg) {
      // ------------------------------------------------------------ epilogue
      const int quad = warp & 3;      // TMEM lanes 32 quad .. 32 quad + 31
      const int eg = (warp - 2) >> 2;  // warpgroup: reduces blocks eg, eg + kEwg, ...
      const int rowt = quad * 32 + lane;
      TileWalk w;
      walk_start(a, t_begin, w);
      int cur_b = -1;
      UnitInfo ui{0, 0, 0, 0};
      float wl[kMaxNQ];  // lane h holds w'_h of each query row of the current request
      float* wme = wsm + (warp - 2) * (kMaxNQ * kIdxHeads);  // wide epilogue: this warp's weights
      float wr[kIdxHeads];  // one query row: all head weights
      int s = 0, acc = 0;
      uint32_t aph = 0;
      for (long long t0 = t_begin; t0 < t_end; t0 += G) {
        const int ng = int(t_end - t0 < G ? t_end - t0 : G);
        if (*abort_flag) break;
        if (!ptx::mbar_wait(tfull + acc, aph)) { fail(); break; }
        ptx::tc_fence_after();
        float sc[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) sc[g] = g < ng ? scl[(size_t(s) * G + g) * kTileTok + rowt] : 0.f;
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(empty + s);
        // the stage's accumulators are nb = ng * n_q blocks of 32 columns,
        // block (g, t) = tile g, query row t; this warpgroup reduces blocks
        // eg, eg + kEwg, ... and steps over the others; the load of its next
        // block is in flight while the current one is reduced
        const uint32_t col0 = tmem + (uint32_t(quad * 32) << 16) + uint32_t(acc * G * a.ncol);
        const int nb = ng * a.n_q;
        EpiState e{0, 0};
        int pos = 0;  // block the epilogue position e / w points at
        float va[32], vb[32];
        if (eg < nb) {
          ptx::tmem_ld32_nowait(col0 + uint32_t(eg * 32), va);
          ptx::tmem_ld_wait(va);
        }
#pragma unroll 1
        for (int c = eg; c < nb; c += 2 * kEwg) {
          const int c1 = c + kEwg, c2 = c + 2 * kEwg;
          if (c1 < nb) ptx::tmem_ld32_nowait(col0 + uint32_t(c1 * 32), vb);
          for (; pos < c; ++pos) epi_skip(a, w, e);
          if constexpr (kEwg > 1) epi_block_wide(a, va, sc, rowt, lane, w, e, cur_b, ui, wme);
          else epi_block(a, va, sc, rowt, lane, w, e, cur_b, ui, wl, wr);
          ++pos;
          if (c1 < nb) {
            ptx::tmem_ld_wait(vb);
            if (c2 < nb) ptx::tmem_ld32_nowait(col0 + uint32_t(c2 * 32), va);
            for (; pos < c1; ++pos) epi_skip(a, w, e);
            if constexpr (kEwg > 1) epi_block_wide(a, vb, sc, rowt, lane, w, e, cur_b, ui, wme);
            else epi_block(a, vb, sc, rowt, lane, w, e, cur_b, ui, wl, wr);
            ++pos;
            if (c2 < nb) ptx::tmem_ld_wait(va);
          }
        }
        for (; pos < nb; ++pos) epi_skip(a, w, e);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(tempty + acc);
        if (++s == S) s = 0;
        if (++acc == NA) { acc = 0; aph ^= 1u; }
      }
    }
  }
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, a.tmem_cols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

}  // namespace

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

bool encode_map(CUtensorMap* m, CUtensorMapDataType dtype, const void* base, int rank, const uint64_t* dims,
                const uint64_t* strides, const uint32_t* box, bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, dtype, cuuint32_t(rank), const_cast<void*>(base),
                  reinterpret_cast<const cuuint64_t*>(dims), reinterpret_cast<const cuuint64_t*>(strides),
                  reinterpret_cast<const cuuint32_t*>(box), es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_indexer(const dsa_params_t& p, const WsLayout& L, char* ws, const void* key_pool,
                           const int32_t* block_table, const int32_t* ctx_lens, float* scores,
                           int64_t score_stride, cudaStream_t st, int world, int rank, bool keep128) {
  const UnitMap map = unit_map(p.n_q, world, rank);
  const int gsz = map.gsz;
  const uint8_t* q8 = reinterpret_cast<const uint8_t*>(ws + L.q8);
  const float* wq = reinterpret_cast<const float*>(ws + L.wq);
  int* err = reinterpret_cast<int*>(ws + L.err);
  const bool mx = p.key_fmt == DSA_KEY_MXFP4_68;
  CUtensorMap kmap, qmap;
  std::memset(&kmap, 0, sizeof(kmap));  // unused by the MXFP4 kernel (raw pages go by bulk copy)
  if (!mx) {
    const uint64_t dims[3] = {uint64_t(kIdxDim), uint64_t(kPage), uint64_t(p.num_pages)};
    const uint64_t strides[2] = {uint64_t(kIdxDim), uint64_t(p.key_page_stride)};
    const uint32_t box[3] = {uint32_t(kIdxDim), uint32_t(kPage), 1};
    if (!encode_map(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, key_pool, 3, dims, strides, box, true)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {uint64_t(kIdxDim), uint64_t(L.rows) * kIdxHeads};
    const uint64_t strides[1] = {uint64_t(kIdxDim)};
    const uint32_t box[2] = {uint32_t(kIdxDim), uint32_t(gsz * kIdxHeads)};
    if (!encode_map(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, q8, 2, dims, strides, box, true)) return cudaErrorInvalidValue;
  }
  IdxTc a;
  a.block_table = block_table;
  a.ctx_lens = ctx_lens;
  a.tile_prefix = reinterpret_cast<const int32_t*>(ws + L.tiles);
  a.wq = wq;
  a.key_pool = static_cast<const uint8_t*>(key_pool);
  a.scores = scores;
  // the group maxima feed only dsa_decode's top-k (a stand-alone dsa_topk
  // computes its own), so other calls skip them
  a.gmax = keep128 ? reinterpret_cast<uint32_t*>(ws + L.gmax) : nullptr;
  a.gmax128 = keep128 ? reinterpret_cast<uint32_t*>(ws + L.gmax128) : nullptr;
  a.gstride = L.gstride;
  a.g128stride = L.g128stride;
  a.score_stride = score_stride;
  a.key_page_stride = p.key_page_stride;
  a.units = p.batch * map.groups;
  a.n_q = gsz;
  a.map = map;
  a.max_pages = p.max_pages_per_req;
  a.num_pages = p.num_pages;
  a.ncol = gsz * kIdxHeads;
  // FP8 keys, one query row: two CTAs per SM, each with half of the shared
  // memory and TMEM (two independent pipelines per SM measured 4% faster than
  // one with twice the tiles per stage). Tiles per stage: as many as fit 256
  // accumulator columns, at most 2 (4 with one CTA per SM).
  const int cps = (!mx && gsz == 1) ? 2 : 1;
  a.group = std::max(1, std::min(cps == 2 || mx ? 2 : 4, 256 / a.ncol));
  const int slot_cols = a.group * a.ncol;
  a.nacc = std::max(1, std::min(4, 512 / cps / slot_cols));
  int cols = 32;
  while (cols < a.nacc * slot_cols) cols <<= 1;
  a.tmem_cols = cols;
  const size_t stage_bytes = size_t(a.group) * (kKeyTileBytes + kScaleTileBytes);
  // several query rows: more epilogue warpgroups (three with FP8 keys, two
  // beside the MXFP4 converters), whose weights are staged in shared memory
  const bool wide = gsz > 1;
  const size_t fixed = 1024 + 2 * size_t(gsz) * kIdxHeads * kIdxDim + 512 +
                       (wide ? size_t(12) * kMaxNQ * kIdxHeads * 4 : 0);
  const size_t budget = (cps == 2 ? 113 * 1024 : 227 * 1024) - fixed;
  if (mx) {
    // three key stages; the rest of shared memory holds raw page pairs in flight
    a.stages = 3;
    a.raw_slots = int(std::min<size_t>(16, (budget - 3 * stage_bytes) / kMxRawTile));
  } else {
    a.stages = int(std::min<size_t>(8, budget / stage_bytes));
    a.raw_slots = 0;
  }
  a.err = err;
  const size_t smem = fixed + size_t(a.stages) * stage_bytes + size_t(a.raw_slots) * kMxRawTile;
  const void* fn = mx ? (wide ? reinterpret_cast<const void*>(indexer_tc_kernel<true, 2>)
                             : reinterpret_cast<const void*>(indexer_tc_kernel<true, 1>))
                 : wide ? reinterpret_cast<const void*>(indexer_tc_kernel<false, 3>)
                        : reinterpret_cast<const void*>(indexer_tc_kernel<false, 1>);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  // enough tiles for every SM is the common case; with fewer, one CTA per tile
  const long long max_tiles = (long long)a.units * ((L.cap + kTileTok - 1) / kTileTok);
  const int grid = int(std::min<long long>(cps * sm_count(), std::max<long long>(1, max_tiles)));
  if (mx && wide)
    return launch_pdl(indexer_tc_kernel<true, 2>, dim3(grid), dim3(64 + 256 + kMxConvThreads), smem, st, kmap, qmap, a);
  if (mx) return launch_pdl(indexer_tc_kernel<true, 1>, dim3(grid), dim3(64 + 128 + kMxConvThreads), smem, st, kmap, qmap, a);
  if (wide) return launch_pdl(indexer_tc_kernel<false, 3>, dim3(grid), dim3(64 + 384), smem, st, kmap, qmap, a);
  return launch_pdl(indexer_tc_kernel<false, 1>, dim3(grid), dim3(kTcThreads), smem, st, kmap, qmap, a);
}

}  // namespace dsa
