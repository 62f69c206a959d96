// Stage 3: exact absorbed-MLA attention over the selected latents, split over
// the K selected slots, then an LSE merge of the splits.
//
// ("vLLM 为 Kimi K3.1 Pro 提供 Day-0 支持", "K3.1 Pro 中的稀疏注意力": attention runs
// exactly over the kept tokens' 576-B FP8 latents, one latent shared by all 96
// heads; "长上下文：带稀疏 indexer 的 decode 上下文并行": partial outputs merge by
// log-sum-exp.)
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "dsa_internal.cuh"
#include "sm103_ptx.cuh"

namespace dsa {

namespace {

// ---------------------------------------------------------------------------
// Tensor-core split-KV attention (sm_103a) on 2-CTA clusters. A work unit is
// one (row, split): kSplitTok consecutive slots of the row's top-k list. Each
// cluster takes a contiguous run of units in (row, split) order, keeps the
// query while the row does not change, and streams the units' 64-token tiles
// through one pipeline: tile indices, barrier phases and the score exchange
// run on across unit boundaries, so a unit's epilogue overlaps the next unit's
// gathers and QK^T. (A batch of a few rows gets one unit per cluster.)
//
// A 96-head x 512-dim fp32 output needs all 512 TMEM columns, so the pair
// splits the work by latent dims: CTA c owns nope dims [256c, 256c+256) (its
// half of the output, TMEM columns [0, 256)) and CTA 0 also the 64 rope dims.
// Each CTA multiplies only its own dims, S_c = Q[:, own] . C[:, own]^T, and
// the two partial score tiles are exchanged through distributed shared memory;
// both CTAs add them (a + b, the same IEEE result on either side), so both run
// the identical softmax and each finishes its half of O = P . V.
// The 96 heads are the M = 128 rows (rows 96..127 are padding, never read).
//   warps 0..2  softmax / epilogue: one head row per thread, online softmax in
//               base 2 with lazy rescale of O (when the max grows by > 2^8)
//   warp  3     TMEM owner, Q by TMA, MMA issuer (QK^T of tile k+1 is issued
//               before PV of tile k, so it overlaps the softmax)
//   warps 4..7  converters: resolve each unit's selected slots to latent rows
//               (four buffers, by unit), gather the rows (paged, 16-B loads one
//               tile ahead) and expand this CTA's dims E4M3 -> bf16 exactly
//               into a 128-B swizzled K-major tile (2 buffers); the per-tensor
//               latent scale is not applied there but to the scores' scale and
//               the output's 1 / l
// The epilogue stages O / l per warp as 32 x 32 swizzled tiles, alternating the
// warp's own staging tile and its quarter of P, and writes the split partials
// with TMA stores (the tile buffers belong to the next unit); a cluster's last
// unit stages whole rows in the freed tile buffers instead and writes them with
// one 1-KB bulk store per head.
// ---------------------------------------------------------------------------
constexpr int kNT = 64;                     // tokens per tile
constexpr int kQBlk = kHeads * 128;         // 12,288 B per Q K-block (96 rows of 64 bf16)
constexpr int kLBlk = kNT * 128;            // 8,192 B per latent K-block (64 rows)
constexpr int kOwnKB = 5;                   // K-blocks of CTA 0 (4 nope + rope); CTA 1 owns 4
constexpr int kQBytes = kOwnKB * kQBlk;     // 61,440
constexpr int kLatBuf = kOwnKB * kLBlk;     // 40,960 per buffer
constexpr int kPBytes = 128 * 128;          // 16,384
constexpr int kXRow = 64 * 4 + 16;          // one row of a partial score tile (+16 B against bank conflicts)
constexpr int kXBuf = kHeads * kXRow;       // 26,112
constexpr uint32_t kXBytes = kHeads * 64 * 4;  // score bytes the peer sends per tile
constexpr int kTcMlaThreads = 256;
constexpr uint32_t kSCol = 256;             // score tiles at TMEM columns [256, 384)
constexpr int kSplitTiles = kSplitTok / kNT;
constexpr int kNumBars = 16;
constexpr int kUnitBufs = 4;                // row-address buffers, by unit
constexpr int kStage = 32 * 128;            // one softmax warp's 32 x 32 fp32 output tile
constexpr int kORow = 256 * 4 + 16;         // a head's output row staged in the free tile buffers
static_assert(kHeads * kORow <= 2 * kLatBuf + kPBytes + 2 * kXBuf, "output staging overlaps the tile buffers");
static_assert(3 * kStage <= kPBytes, "each softmax warp's quarter of P holds a staging tile");
constexpr size_t kTcMlaSmem = 1024 + kQBytes + 2 * kLatBuf + kPBytes + 2 * kXBuf + 3 * kStage +
                              kUnitBufs * (kSplitTok * 8 + kSplitTiles * 8) + kNumBars * 8 + 16;
static_assert(kTcMlaSmem <= 232448, "shared memory of one CTA");

struct MlaTc {
  const int32_t* block_table;
  const int32_t* ctx_lens;
  const int32_t* topk_idx;
  const uint8_t* lat_pool;
  int64_t lat_stride;
  int lat_row, lat_nvfp4;  // bytes per latent row; 1 for the NVFP4 row format
  int max_pages, num_pages, n_q, cap, K, splits, per_split, rows;
  float sm_scale_log2, lat_scale;
  float* opart;
  float* lpart;
  int* err;
  int early;  // set up and fetch Q before the wait on the previous kernel (dsa_decode: q is a caller input)
};

__device__ __forceinline__ uint32_t bf16x2_from_e4m3x2(uint16_t two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
  const __nv_bfloat162 b = __float22bfloat162_rn(f);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// 16 E4M3 bytes -> 16 bf16 (exactly), as two 16-B chunks. The per-tensor
// latent scale is not applied here: it multiplies the scores' scale and the
// output instead (one factor of the whole sum), so the tiles hold the exact
// quantised values.
__device__ __forceinline__ void expand_e4m3x16(const uint4 w, uint4& lo, uint4& hi) {
  lo.x = bf16x2_from_e4m3x2(uint16_t(w.x)); lo.y = bf16x2_from_e4m3x2(uint16_t(w.x >> 16));
  lo.z = bf16x2_from_e4m3x2(uint16_t(w.y)); lo.w = bf16x2_from_e4m3x2(uint16_t(w.y >> 16));
  hi.x = bf16x2_from_e4m3x2(uint16_t(w.z)); hi.y = bf16x2_from_e4m3x2(uint16_t(w.z >> 16));
  hi.z = bf16x2_from_e4m3x2(uint16_t(w.w)); hi.w = bf16x2_from_e4m3x2(uint16_t(w.w >> 16));
}

// Byte offset inside a 576-B latent row of this CTA's 16-B piece q, for
// NPC = 20 (CTA 0: nope [0, 256) then rope) or NPC = 16 (CTA 1: nope [256, 512)).
template <int NPC>
__device__ __forceinline__ int piece_offset(int q) {
  return NPC == 20 ? (q < 16 ? 16 * q : 512 + 16 * (q - 16)) : 256 + 16 * q;
}

// Gather this CTA's pieces of tile k's selected rows into registers (zeros for
// unused slots). Piece pc = ct + 128u: token pc / NPC, piece pc % NPC of its row.
template <int NPC>
__device__ __forceinline__ void conv_load(uint4 (&buf)[NPC / 2], const uint8_t* const* rowptr, int ct, int k) {
  const uint8_t* const* rp = rowptr + k * kNT;
#pragma unroll
  for (int u = 0; u < NPC / 2; ++u) {
    const int pc = ct + 128 * u;
    const int jj = pc / NPC, q = pc - jj * NPC;
    const uint8_t* p = rp[jj];
    buf[u] = p ? __ldg(reinterpret_cast<const uint4*>(p + piece_offset<NPC>(q))) : make_uint4(0, 0, 0, 0);
  }
}

// Expand stream tile k into LAT[k & 1] once the tile that last used that buffer is done.
template <int NPC>
__device__ __forceinline__ bool conv_store(const uint4 (&buf)[NPC / 2], const MlaTc& a, int ct, int lane, int k,
                                           uint8_t* LAT, uint64_t* lat_full, uint64_t* lat_free) {
  const int bk = k & 1;
  bool ok = true;
  if (k >= 2 && !ptx::mbar_wait(lat_free + bk, uint32_t((k >> 1) - 1) & 1u)) ok = false;
  if (ok) {
    uint8_t* lat = LAT + bk * kLatBuf;
#pragma unroll
    for (int u = 0; u < NPC / 2; ++u) {
      const int pc = ct + 128 * u;
      const int jj = pc / NPC, q = pc - jj * NPC;
      const int kl = q >> 2, c = (q & 3) * 2;
      uint4 lo, hi;
      expand_e4m3x16(buf[u], lo, hi);
      uint8_t* rowb = lat + kl * kLBlk + jj * 128;
      *reinterpret_cast<uint4*>(rowb + ((c ^ (jj & 7)) << 4)) = lo;
      *reinterpret_cast<uint4*>(rowb + (((c + 1) ^ (jj & 7)) << 4)) = hi;
    }
    ptx::fence_proxy_async_smem();
  }
  __syncwarp();
  if (lane == 0) ptx::mbar_arrive(lat_full + bk);
  return ok;
}

// Converter warps (128 threads): a unit's tiles 0..nt-1 (stream tiles g0 + k)
// into LAT[(g0 + k) & 1], the loads of tile k+1 in flight while tile k waits
// for its buffer and is expanded.
// (One call site of each step: the expansion is long, and the kernel's code
// already strains the instruction cache.)
template <int NPC>
__device__ void converter_role(const MlaTc& a, int ct, int lane, int nt, int g0, const uint8_t* const* rowptr,
                               uint8_t* LAT, uint64_t* lat_full, uint64_t* lat_free, bool& ok) {
  uint4 cur[NPC / 2], nxt[NPC / 2];
  conv_load<NPC>(cur, rowptr, ct, 0);
#pragma unroll 1
  for (int k = 0; k < nt; ++k) {
    if (k + 1 < nt) conv_load<NPC>(nxt, rowptr, ct, k + 1);
    if (!conv_store<NPC>(cur, a, ct, lane, g0 + k, LAT, lat_full, lat_free)) { ok = false; return; }
#pragma unroll
    for (int u = 0; u < NPC / 2; ++u) cur[u] = nxt[u];
  }
}

// ---------------------------------------------------------------------------
// NVFP4 latent rows (352 B: [256 B E2M1, element 2i in the low nibble][32 B
// E4M3 scales, one per 16 nope values][64 B E4M3 rope]). A unit is 16 bytes of
// a row: an E2M1 unit holds 32 nope values (two scales), a rope unit 16 E4M3
// values. CTA 0 takes E2M1 units 0..7 (nope [0, 256)) and rope units 8..11;
// CTA 1 takes E2M1 units 8..15 (nope [256, 512)).
// ---------------------------------------------------------------------------
template <int HALF>
struct NvUnits {
  static constexpr int kPerTok = HALF == 0 ? 12 : 8;
  static constexpr int kPerThread = kNT * kPerTok / 128;
};

struct NvUnit {
  uint4 v;
  uint32_t s;  // the unit's two E4M3 scales (E2M1 units)
};

template <int HALF>
__device__ __forceinline__ void conv_load_nv(NvUnit (&buf)[NvUnits<HALF>::kPerThread], const uint8_t* const* rowptr,
                                             int ct, int k) {
  constexpr int NU = NvUnits<HALF>::kPerTok;
  const uint8_t* const* rp = rowptr + k * kNT;
#pragma unroll
  for (int u = 0; u < NvUnits<HALF>::kPerThread; ++u) {
    const int pc = ct + 128 * u;
    const int jj = pc / NU, q = pc - jj * NU;
    const uint8_t* p = rp[jj];
    buf[u].v = make_uint4(0, 0, 0, 0);
    buf[u].s = 0;
    if (p) {
      if (q < 8) {
        const int e = HALF * 8 + q;  // E2M1 unit of the row
        buf[u].v = __ldg(reinterpret_cast<const uint4*>(p + 16 * e));
        buf[u].s = __ldg(reinterpret_cast<const uint16_t*>(p + 256 + 2 * e));
      } else {
        buf[u].v = __ldg(reinterpret_cast<const uint4*>(p + 288 + 16 * (q - 8)));
      }
    }
  }
}

// 8 E2M1 values (one 32-bit word) times `scale` -> 8 bf16 (one 16-B chunk).
__device__ __forceinline__ uint4 e2m1x8_scaled(uint32_t w, float scale) {
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2_raw h = __nv_cvt_fp4x2_to_halfraw2(static_cast<__nv_fp4x2_storage_t>((w >> (8 * i)) & 0xFFu), __NV_E2M1);
    const float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
    o[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(byte & 0xFFu), __NV_E4M3);
  return __half2float(*reinterpret_cast<const __half*>(&h));
}

template <int HALF>
__device__ __forceinline__ bool conv_store_nv(const NvUnit (&buf)[NvUnits<HALF>::kPerThread], const MlaTc& a, int ct,
                                              int lane, int k, uint8_t* LAT, uint64_t* lat_full, uint64_t* lat_free) {
  constexpr int NU = NvUnits<HALF>::kPerTok;
  const int bk = k & 1;
  bool ok = true;
  if (k >= 2 && !ptx::mbar_wait(lat_free + bk, uint32_t((k >> 1) - 1) & 1u)) ok = false;
  if (ok) {
    uint8_t* lat = LAT + bk * kLatBuf;
#pragma unroll
    for (int u = 0; u < NvUnits<HALF>::kPerThread; ++u) {
      const int pc = ct + 128 * u;
      const int jj = pc / NU, q = pc - jj * NU;
      uint8_t* rowb;
      if (q < 8) {
        // nope dims [32q, 32q + 32) of this CTA: K-block q / 2, chunks 4 (q & 1) .. + 3
        rowb = lat + (q >> 1) * kLBlk + jj * 128;
        const float s0 = e4m3_to_float(buf[u].s);  // E2M1 x E4M3: exact in bf16
        const float s1 = e4m3_to_float(buf[u].s >> 8);
        const int c0 = (q & 1) * 4;
        *reinterpret_cast<uint4*>(rowb + (((c0 + 0) ^ (jj & 7)) << 4)) = e2m1x8_scaled(buf[u].v.x, s0);
        *reinterpret_cast<uint4*>(rowb + (((c0 + 1) ^ (jj & 7)) << 4)) = e2m1x8_scaled(buf[u].v.y, s0);
        *reinterpret_cast<uint4*>(rowb + (((c0 + 2) ^ (jj & 7)) << 4)) = e2m1x8_scaled(buf[u].v.z, s1);
        *reinterpret_cast<uint4*>(rowb + (((c0 + 3) ^ (jj & 7)) << 4)) = e2m1x8_scaled(buf[u].v.w, s1);
      } else {
        // rope dims [16 (q - 8), + 16): K-block 4, chunks 2 (q - 8) and + 1
        rowb = lat + 4 * kLBlk + jj * 128;
        const int c = (q - 8) * 2;
        uint4 lo, hi;
        expand_e4m3x16(buf[u].v, lo, hi);
        *reinterpret_cast<uint4*>(rowb + ((c ^ (jj & 7)) << 4)) = lo;
        *reinterpret_cast<uint4*>(rowb + (((c + 1) ^ (jj & 7)) << 4)) = hi;
      }
    }
    ptx::fence_proxy_async_smem();
  }
  __syncwarp();
  if (lane == 0) ptx::mbar_arrive(lat_full + bk);
  return ok;
}

template <int HALF>
__device__ void converter_role_nv(const MlaTc& a, int ct, int lane, int nt, int g0, const uint8_t* const* rowptr,
                                  uint8_t* LAT, uint64_t* lat_full, uint64_t* lat_free, bool& ok) {
  NvUnit cur[NvUnits<HALF>::kPerThread], nxt[NvUnits<HALF>::kPerThread];
  conv_load_nv<HALF>(cur, rowptr, ct, 0);
#pragma unroll 1
  for (int k = 0; k < nt; ++k) {
    if (k + 1 < nt) conv_load_nv<HALF>(nxt, rowptr, ct, k + 1);
    if (!conv_store_nv<HALF>(cur, a, ct, lane, g0 + k, LAT, lat_full, lat_free)) { ok = false; return; }
#pragma unroll
    for (int u = 0; u < NvUnits<HALF>::kPerThread; ++u) cur[u] = nxt[u];
  }
}

// kNv: NVFP4 latent rows (else FP8); one converter kind per instance keeps the
// registers of the other out of the unit loop.
template <bool kNv>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kTcMlaThreads, 1)
    sparse_mla_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
                         MlaTc a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Qs = sm;
  uint8_t* LAT = Qs + kQBytes;                     // 2 buffers
  uint8_t* Ps = LAT + 2 * kLatBuf;
  uint8_t* X = Ps + kPBytes;                       // 2 buffers: the peer's partial scores
  uint8_t* ST = X + 2 * kXBuf;                     // 3 output staging tiles (1024-B aligned)
  const uint8_t** rowptr = reinterpret_cast<const uint8_t**>(ST + 3 * kStage);                 // [4][kSplitTok]
  unsigned long long* vmask = reinterpret_cast<unsigned long long*>(rowptr + kUnitBufs * kSplitTok);  // [4][tiles]
  uint64_t* bars = reinterpret_cast<uint64_t*>(vmask + kUnitBufs * kSplitTiles);
  uint64_t* q_full = bars + 0;
  uint64_t* lat_full = bars + 1;   // [2]
  uint64_t* lat_free = bars + 3;   // [2]  (PV of the buffer's last tile done)
  uint64_t* s_full = bars + 5;     // [2]
  uint64_t* s_free = bars + 7;     // [2]
  uint64_t* p_full = bars + 9;
  uint64_t* x_full = bars + 10;    // [2]  the peer's partial scores have landed in X
  uint64_t* q_free = bars + 12;    // every MMA on the current query done (before a new one lands)
  uint64_t* mma_done = bars + 13;  // every MMA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);

  const int half = int(ptx::cluster_ctarank());
  const int peer = half ^ 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = half == 0 ? 5 : 4;
  // this cluster's units [u0, u1) of rows * splits, and its total tiles (all
  // units of a call have ceil(min(K - j0, kSplitTok) / 64) tiles by split)
  const int U = a.rows * a.splits;
  const int nclu = int(gridDim.x) >> 1, clu = int(blockIdx.x) >> 1;
  const int u0 = int(int64_t(clu) * U / nclu), u1 = int(int64_t(clu + 1) * U / nclu);
  auto unit_tiles = [&](int u) {
    const int j0 = (u % a.splits) * a.per_split;
    const int j1 = min(a.K, j0 + a.per_split);
    return (j1 - j0 + kNT - 1) / kNT;
  };
  int gtot = 0;
  for (int u = u0; u < u1; ++u) gtot += unit_tiles(u);

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    ptx::mbar_init(q_free, 1);
    ptx::mbar_init(mma_done, 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(lat_full + i, 4);
      ptx::mbar_init(lat_free + i, 1);
      ptx::mbar_init(s_full + i, 1);
      ptx::mbar_init(s_free + i, 3);
      ptx::mbar_init(x_full + i, 1);
    }
    ptx::mbar_init(p_full, 3);
    // the peer's first two score tiles may arrive as soon as the pair has synced
    if (gtot > 0) ptx::mbar_arrive_expect_tx(x_full + 0, kXBytes);
    if (gtot > 1) ptx::mbar_arrive_expect_tx(x_full + 1, kXBytes);
    ptx::fence_mbar_init();
  }
  if (warp == 3) {
    ptx::tmem_alloc(tmem_slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // the peer's barriers exist before any remote arrive
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;
  // this CTA's K-blocks of the query of row r: CTA 0 nope 0..3 and the rope, CTA 1 nope 4..7
  auto issue_q = [&](int r) {
    ptx::mbar_arrive_expect_tx(q_full, nkb * kQBlk);
    for (int kl = 0; kl < nkb; ++kl) {
      const int kbg = half == 0 ? (kl < 4 ? kl : 8) : 4 + kl;
      ptx::tma_load_2d(Qs + kl * kQBlk, &qmap, q_full, kbg * 64, r * kHeads);
    }
  };
  int q_row = -1;
  bool q_pending = false;
  if (a.early && warp == 3 && u0 < u1) {
    q_row = u0 / a.splits;
    if (ptx::elect_one()) issue_q(q_row);
    __syncwarp();
    q_pending = true;
  }
  // everything above is on-chip set-up or a read of the caller's query; what
  // comes next reads the top-k list of the previous kernel
  pdl_wait();
  pdl_trigger();  // the split combine may take free SMs now (it waits for this grid)

  if (warp == 3) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp walks the loop (so every operand below is computed in
    // converged code); one elected lane issues each batch of MMAs, commits and
    // copies.
    {
      const uint32_t id_qk = ptx::idesc(1, 1, 128, kNT);
      const uint32_t id_pv = ptx::idesc(1, 1, 128, 256, 0, 1);
      const uint32_t q0 = ptx::smem_u32(Qs), l0 = ptx::smem_u32(LAT), p0 = ptx::smem_u32(Ps);
      int g = 0, qn = 0, qf = 0, last_k = 0;
      // PV of stream tile j, the kj-th of its unit: O (+)= P . V[j & 1]
      auto pv = [&](int j, int kj) {
        if (!ok || !ptx::mbar_wait(p_full, uint32_t(j) & 1u)) { ok = false; return; }
        ptx::tc_fence_after();
        const uint32_t lat = l0 + (j & 1) * kLatBuf;
        if (ptx::elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kNT / 16; ++kk)
            ptx::mma_f16(tmem, ptx::sdesc_sw128(p0 + kk * 32), ptx::sdesc_sw128_mn(lat + kk * 16 * 128, kLBlk, 1024),
                         id_pv, (kj > 0 || kk > 0) ? 1u : 0u);
          ptx::mma_commit(lat_free + (j & 1));
        }
        __syncwarp();
      };
      for (int u = u0; u < u1 && ok; ++u) {
        const int r = u / a.splits, nt = unit_tiles(u);
        for (int k = 0; k < nt && ok; ++k, ++g) {
          // at a unit boundary the previous unit's last PV goes first, so that
          // its epilogue never waits for a query reload
          if (k == 0 && g >= 1) pv(g - 1, last_k);
          if (k == 0 && r != q_row) {
            if (q_row >= 0) {  // every MMA reading the old query is done before it is overwritten
              if (ptx::elect_one()) ptx::mma_commit(q_free);
              __syncwarp();
              if (!ptx::mbar_wait(q_free, uint32_t(qf++) & 1u)) { ok = false; break; }
            }
            if (ptx::elect_one()) issue_q(r);
            __syncwarp();
            q_row = r;
            q_pending = true;
          }
          if (q_pending) {
            if (!ptx::mbar_wait(q_full, uint32_t(qn++) & 1u)) { ok = false; break; }
            q_pending = false;
          }
          const int bk = g & 1;
          const uint32_t kph = uint32_t(g >> 1) & 1u;
          if (!ptx::mbar_wait(lat_full + bk, kph)) { ok = false; break; }
          if (g >= 2 && !ptx::mbar_wait(s_free + bk, kph ^ 1u)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t lat = l0 + bk * kLatBuf;
          if (ptx::elect_one()) {
            for (int kl = 0; kl < nkb; ++kl)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                ptx::mma_f16(tmem + kSCol + bk * kNT, ptx::sdesc_sw128(q0 + kl * kQBlk + kk * 32),
                             ptx::sdesc_sw128(lat + kl * kLBlk + kk * 32), id_qk, (kl | kk) ? 1u : 0u);
            ptx::mma_commit(s_full + bk);
          }
          __syncwarp();
          if (k >= 1) pv(g - 1, k - 1);
          last_k = k;
        }
      }
      if (ok && g >= 1) pv(g - 1, last_k);
      // nothing of this warp's left in flight when TMEM is released
      if (ptx::elect_one()) ptx::mma_commit(mma_done);
      __syncwarp();
      ptx::mbar_wait(mma_done, 0);
      if (q_pending) ptx::mbar_wait(q_full, uint32_t(qn) & 1u);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ converters
    const int ct = threadIdx.x - 128;
    int g = 0;
    for (int u = u0, ui = 0; u < u1 && ok; ++u, ++ui) {
      const int r = u / a.splits, split = u % a.splits, nt = unit_tiles(u);
      const int b = r / a.n_q, t = r - b * a.n_q;
      const int j0 = split * a.per_split, j1 = min(a.K, j0 + a.per_split);
      const int ctx = a.ctx_lens[b];
      const int L = (ctx < a.n_q || ctx > a.cap) ? 0 : ctx - a.n_q + t + 1;
      const uint8_t** rp = rowptr + (ui % kUnitBufs) * kSplitTok;
      unsigned long long* vm = vmask + (ui % kUnitBufs) * kSplitTiles;
      // Resolve every selected slot of the unit once (slot -> page -> row address).
      // The buffer was last used by unit ui - 4, whose tiles are all past PV
      // (the converters' own buffer waits ordered them), so it is free.
      for (int jj = ct; jj < nt * kNT; jj += 128) {
        const int j = j0 + jj;
        const uint8_t* p = nullptr;
        if (j < j1) {
          const int sidx = a.topk_idx[size_t(r) * a.K + j];
          if (sidx >= 0 && sidx < L) {
            const int pg = a.block_table[size_t(b) * a.max_pages + sidx / kPage];
            if (pg >= 0 && pg < a.num_pages)
              p = a.lat_pool + size_t(pg) * a.lat_stride + size_t(sidx % kPage) * a.lat_row;
            else if (half == 0)
              atomicOr(a.err, DSA_DEVERR_BLOCK_TABLE);
          } else if (sidx != -1 && half == 0) {
            atomicOr(a.err, DSA_DEVERR_TOPK_INDEX);
          }
        }
        rp[jj] = p;
        const unsigned m = __ballot_sync(0xffffffffu, p != nullptr);
        if (lane == 0) reinterpret_cast<uint32_t*>(vm)[jj >> 5] = m;
      }
      ptx::named_bar_sync(1, 128);
      if constexpr (kNv) {
        if (half == 0)
          converter_role_nv<0>(a, ct, lane, nt, g, rp, LAT, lat_full, lat_free, ok);
        else
          converter_role_nv<1>(a, ct, lane, nt, g, rp, LAT, lat_full, lat_free, ok);
      } else if (half == 0) {
        converter_role<20>(a, ct, lane, nt, g, rp, LAT, lat_full, lat_free, ok);
      } else {
        converter_role<16>(a, ct, lane, nt, g, rp, LAT, lat_full, lat_free, ok);
      }
      g += nt;
    }
  } else if (warp < 3) {
    // ------------------------------------------------------------ softmax / epilogue
    const int h = warp * 32 + lane;
    const uint32_t lane_base = uint32_t(warp * 32) << 16;
    const uint32_t x_mine = ptx::smem_u32(X) + h * kXRow;
    const uint32_t x_peer = ptx::mapa_shared(x_mine, peer);
    uint8_t* stg = ST + warp * kStage;
    uint8_t* pstg = Ps + warp * kStage;  // this warp's quarter of P, a second staging tile in the epilogue
    int g = 0;
    for (int u = u0, ui = 0; u < u1 && ok; ++u, ++ui) {
      const int r = u / a.splits, split = u % a.splits, nt = unit_tiles(u);
      const unsigned long long* vmu = vmask + (ui % kUnitBufs) * kSplitTiles;
      float m_use = -INFINITY, l = 0.f;
      for (int k = 0; k < nt; ++k, ++g) {
        const int bk = g & 1;
        const uint32_t kph = uint32_t(g >> 1) & 1u;
        // lat_full orders the converters' validity mask before this read
        if (!ptx::mbar_wait(lat_full + bk, kph) || !ptx::mbar_wait(s_full + bk, kph)) { ok = false; break; }
        ptx::tc_fence_after();
        float sv[64];
        ptx::tmem_ld32(tmem + lane_base + kSCol + bk * kNT, *reinterpret_cast<float(*)[32]>(&sv[0]));
        ptx::tmem_ld32(tmem + lane_base + kSCol + bk * kNT + 32, *reinterpret_cast<float(*)[32]>(&sv[32]));
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(s_free + bk);
        // exchange partial scores with the peer CTA: asynchronous remote stores
        // whose bytes complete on the peer's x_full[bk]. The peer's X[bk] is free
        // again: this CTA got here after receiving the peer's tile g - 1, which
        // every peer thread sent after reading its row of X[bk] (tile g - 2).
        {
          const uint32_t dst = x_peer + bk * kXBuf;
          const uint32_t rbar = ptx::mapa_shared(ptx::smem_u32(x_full + bk), peer);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            ptx::st_async_f4(dst + i * 16, make_float4(sv[4 * i], sv[4 * i + 1], sv[4 * i + 2], sv[4 * i + 3]), rbar);
        }
        if (!ptx::mbar_wait_cluster(x_full + bk, kph)) { ok = false; break; }
        const float4* xr = reinterpret_cast<const float4*>(X + bk * kXBuf + h * kXRow);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float4 x = xr[i];
          sv[4 * i] += x.x; sv[4 * i + 1] += x.y; sv[4 * i + 2] += x.z; sv[4 * i + 3] += x.w;
        }
        // warp 0 re-arms x_full[bk] for stream tile g + 2 (bytes that arrive
        // first count down until the arrival; the phase cannot complete before it)
        if (warp == 0 && lane == 0 && g + 2 < gtot) ptx::mbar_arrive_expect_tx(x_full + bk, kXBytes);
        unsigned long long vm = vmu[0];
#pragma unroll
        for (int i = 1; i < kSplitTiles; ++i)
          if (k == i) vm = vmu[i];
        float tmax = -INFINITY;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          sv[i] = ((vm >> i) & 1ull) ? sv[i] * a.sm_scale_log2 : -INFINITY;
          tmax = fmaxf(tmax, sv[i]);
        }
        // P and O are free once the previous stream tile's PV has completed
        if (g >= 1 && !ptx::mbar_wait(lat_free + ((g - 1) & 1), uint32_t((g - 1) >> 1) & 1u)) { ok = false; break; }
        ptx::tc_fence_after();
        bool need = false;
        float alpha = 1.f;
        if (m_use == -INFINITY) {
          m_use = tmax;
        } else if (tmax > m_use + 8.f) {
          need = true;
          alpha = ptx::ex2_approx(m_use - tmax);
          m_use = tmax;
        }
        if (__any_sync(0xffffffffu, need)) {
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
            const float p0 = m_use == -INFINITY ? 0.f : ptx::ex2_approx(sv[i] - m_use);
            const float p1 = m_use == -INFINITY ? 0.f : ptx::ex2_approx(sv[i + 1] - m_use);
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
      if (!ok) break;
      // epilogue: O / l of this head row and this CTA's 256 dims once the unit's
      // last PV is done
      const int gl = g - 1;
      if (!ptx::mbar_wait(lat_free + (gl & 1), uint32_t(gl >> 1) & 1u)) { ok = false; break; }
      ptx::tc_fence_after();
      const float inv = l > 0.f ? a.lat_scale / l : 0.f;  // O = latent_scale * (sum p c) / l
      const int orow = (r * a.splits + split) * kHeads + warp * 32;
      // 32 columns at a time, the next chunk's TMEM load in flight while this
      // one is scaled and stored (a wait covers every load issued before it)
      const bool tail = u + 1 == u1;
      uint8_t* orow_s = LAT + size_t(h) * kORow;
      auto emit = [&](const float (&o)[32], int c) {
        if (tail) {
          // the cluster's last unit: every tile buffer, P and X are free (the
          // last PV has read them, every peer score has landed), so each
          // thread stages its whole 1-KB row there for one bulk store
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(orow_s + (c + i) * 4) =
                make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
        } else {
          // 32 heads x 32 dims -> a swizzled staging tile (row = head, 16-B
          // chunk j at j ^ (row & 7)) -> one TMA store. The warp alternates two
          // tiles, its own and its quarter of P (free from the unit's last PV
          // until this warp writes the next P), so each wait is for the store
          // two chunks back, which has long read its tile.
          uint8_t* st = ((c >> 5) & 1) ? pstg : stg;
          if (lane == 0) ptx::bulk_wait_read1();
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(st + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                make_float4(o[4 * j] * inv, o[4 * j + 1] * inv, o[4 * j + 2] * inv, o[4 * j + 3] * inv);
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_2d(&omap, st, half * 256 + c, orow);
            ptx::bulk_commit();
          }
        }
      };
      {
        float oa[32], ob[32];
        ptx::tmem_ld32_nowait(tmem + lane_base, oa);
        ptx::tmem_ld_wait(oa);
#pragma unroll 1
        for (int c = 0; c < 256; c += 64) {
          ptx::tmem_ld32_nowait(tmem + lane_base + c + 32, ob);
          emit(oa, c);
          ptx::tmem_ld_wait(ob);
          if (c + 64 < 256) ptx::tmem_ld32_nowait(tmem + lane_base + c + 64, oa);
          emit(ob, c + 32);
          if (c + 64 < 256) ptx::tmem_ld_wait(oa);
        }
      }
      if (tail) {
        ptx::fence_proxy_async_smem();
        ptx::bulk_store(a.opart + (size_t(orow) + lane) * kDNope + half * 256, orow_s, 256 * 4);
        ptx::bulk_commit();
      } else {
        // the stores have read P's quarter before this warp writes the next P
        if (lane == 0) ptx::bulk_wait_read();
        __syncwarp();
      }
      if (half == 0)
        a.lpart[(size_t(r) * a.splits + split) * kHeads + h] = l > 0.f ? (m_use + log2f(l)) * 0.6931471805599453f
                                                                        : -INFINITY;
      // the reads of O are ordered before the next unit's first PV (p_full)
      ptx::tc_fence_before();
    }
    ptx::bulk_wait_all();  // the partials are written before the grid ends
  }
  if (!ok) atomicOr(a.err, DSA_DEVERR_TIMEOUT);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // no remote access to a CTA that has exited
  if (warp == 3) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// LSE merge of the splits of one row: out = sum_i e^{lse_i - lse} O_i, lse = ln sum_i e^{lse_i}.
// One CTA per (row, 3 heads): 128 threads per head, 4 dims each (32 CTAs a
// row: a batch of 4 rows is one wave). In every warp
// lane i < splits holds split i's lse, so the weights come from two shuffle
// reductions; every split's partial row is read at once.
constexpr int kCombThreads = 384;
constexpr int kCombHeads = kCombThreads / 128;
constexpr size_t kCombSpreadSmem = 120 * 1024;  // more than half an SM's shared memory: one CTA per SM

__global__ void __launch_bounds__(kCombThreads) mla_combine_kernel(const float* __restrict__ opart,
                                                                   const float* __restrict__ lpart, int splits,
                                                                   __nv_bfloat16* __restrict__ out,
                                                                   float* __restrict__ lse) {
  pdl_wait();
  const int r = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.y * kCombHeads + (threadIdx.x >> 7);
  const int d4 = threadIdx.x & 127;  // dims 4*d4 .. 4*d4+3
  // every split's partial in flight at once, together with the splits' lse
  // (splits <= kMaxSplits; a slot past the last split reads split 0 again and
  // gets weight 0), then added in split order
  const float4* src = reinterpret_cast<const float4*>(opart + (size_t(r) * splits * kHeads + h) * kDNope) + d4;
  const size_t split_stride = size_t(kHeads) * kDNope / 4;  // float4 per split
  float4 v[kMaxSplits];
#pragma unroll
  for (int u = 0; u < kMaxSplits; ++u) v[u] = __ldg(src + (u < splits ? u : 0) * split_stride);
  const float li = lane < splits ? __ldg(lpart + (size_t(r) * splits + lane) * kHeads + h) : -INFINITY;
  float m = li;
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float e = m == -INFINITY ? 0.f : expf(li - m);
  float tot = e;
#pragma unroll
  for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  const float L = m == -INFINITY ? -INFINITY : m + logf(tot);
  const float wgt = m == -INFINITY ? 0.f : expf(li - L);
  float wv[kMaxSplits];
#pragma unroll
  for (int u = 0; u < kMaxSplits; ++u) {
    const float wi = __shfl_sync(0xffffffffu, wgt, u & 31);
    wv[u] = u < splits ? wi : 0.f;
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int u = 0; u < kMaxSplits; ++u) {
    acc.x = fmaf(wv[u], v[u].x, acc.x); acc.y = fmaf(wv[u], v[u].y, acc.y);
    acc.z = fmaf(wv[u], v[u].z, acc.z); acc.w = fmaf(wv[u], v[u].w, acc.w);
  }
  const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 pk;
  pk.x = *reinterpret_cast<const uint32_t*>(&lo);
  pk.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(out + (size_t(r) * kHeads + h) * kDNope + 4 * d4) = pk;
  if (lse && d4 == 0) lse[size_t(r) * kHeads + h] = L;
}

}  // namespace

cudaError_t launch_sparse_mla(const dsa_params_t& p, const WsLayout& L, char* ws, const void* q,
                              const void* lat_pool, const int32_t* block_table, const int32_t* ctx_lens,
                              const int32_t* topk_idx, void* out, float* lse, cudaStream_t st, bool early) {
  CUtensorMap qmap;
  {
    const uint64_t dims[2] = {uint64_t(kDQK), uint64_t(L.rows) * kHeads};
    const uint64_t strides[1] = {uint64_t(kDQK) * 2};
    const uint32_t box[2] = {64, uint32_t(kHeads)};
    if (!encode_map(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, 2, dims, strides, box, true))
      return cudaErrorInvalidValue;
  }
  CUtensorMap omap;
  {
    // the split partials [rows * splits * 96][512] fp32, written in 32 x 32 tiles
    const uint64_t dims[2] = {uint64_t(kDNope), uint64_t(L.rows) * L.splits * kHeads};
    const uint64_t strides[1] = {uint64_t(kDNope) * 4};
    const uint32_t box[2] = {32, 32};
    if (!encode_map(&omap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, ws + L.opart, 2, dims, strides, box, true))
      return cudaErrorInvalidValue;
  }
  MlaTc t;
  t.block_table = block_table;
  t.ctx_lens = ctx_lens;
  t.topk_idx = topk_idx;
  t.lat_pool = static_cast<const uint8_t*>(lat_pool);
  t.lat_stride = p.lat_page_stride;
  t.lat_nvfp4 = p.lat_fmt == DSA_LAT_NVFP4_352;
  t.lat_row = t.lat_nvfp4 ? kDNope / 2 + kDNope / 16 + kDRope : kLatRowFp8;
  t.max_pages = p.max_pages_per_req;
  t.num_pages = p.num_pages;
  t.n_q = p.n_q;
  t.cap = L.cap;
  t.K = p.topk;
  t.splits = L.splits;
  t.per_split = kSplitTok;
  t.rows = L.rows;
  // the tiles hold the latents without the per-tensor scale: it joins the
  // scores' scale here and the output's 1 / l in the epilogue
  t.sm_scale_log2 = p.softmax_scale * p.latent_scale * 1.4426950408889634f;
  t.lat_scale = p.latent_scale;
  t.opart = reinterpret_cast<float*>(ws + L.opart);
  t.lpart = reinterpret_cast<float*>(ws + L.lpart);
  t.err = reinterpret_cast<int*>(ws + L.err);
  t.early = early ? 1 : 0;
  auto kern = t.lat_nvfp4 ? sparse_mla_tc_kernel<true> : sparse_mla_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kTcMlaSmem));
  if (e != cudaSuccess) return e;
  // one cluster per unit, or a cluster per pair of SMs each taking a run of units
  const int units = L.rows * L.splits;
  const int clusters = std::max(1, std::min(units, sm_count() / 2));
  e = launch_pdl(kern, dim3(2 * clusters), dim3(kTcMlaThreads), kTcMlaSmem, st, qmap, omap, t);
  if (e != cudaSuccess) return e;
  // The combine's CTAs become resident while the attention still holds most
  // SMs; with fewer CTAs than SMs, a shared-memory request that leaves room for
  // one per SM keeps them from stacking on the few free SMs (their loads would
  // then share one SM's bandwidth) and spreads them as the attention's SMs free up.
  const int cctas = L.rows * (kHeads / kCombHeads);
  const size_t csmem = cctas <= sm_count() ? kCombSpreadSmem : 0;
  e = cudaFuncSetAttribute(mla_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kCombSpreadSmem));
  if (e != cudaSuccess) return e;
  return launch_pdl(mla_combine_kernel, dim3(L.rows, kHeads / kCombHeads), dim3(kCombThreads), csmem, st,
                    static_cast<const float*>(t.opart), static_cast<const float*>(t.lpart), int(L.splits),
                    static_cast<__nv_bfloat16*>(out), lse);
}

}  // namespace dsa
