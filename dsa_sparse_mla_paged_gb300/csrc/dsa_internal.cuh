// Internal declarations shared by the libdsa translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/dsa.h"

namespace dsa {

constexpr int kIdxHeads = 32;
constexpr int kIdxDim = 128;
constexpr int kHeads = 96;
constexpr int kDNope = 512;
constexpr int kDRope = 64;
constexpr int kDQK = kDNope + kDRope;
constexpr int kPage = 64;
constexpr int kKeyPageBytesFp8 = kPage * (kIdxDim + 4);  // 8448
constexpr int kLatRowFp8 = kDQK;                         // 576
constexpr int kMaxNQ = 8;
constexpr int kMaxTopK = 2048;

// top-k: each row keeps at most kCandCap candidates for its exact selection,
// filtered by CTAs of at least kTopkChunk tokens each (one record per CTA).
constexpr int kCandCap = 8192;
constexpr int kTopkChunk = 1024;
constexpr int kRowState = 16;     // int32 words of per-row selection state

// sparse attention: the K selected slots of a row are cut into splits of this
// many tokens, one CTA pair each. The split size depends on nothing but K, so a
// request's result does not depend on the batch it is in.
constexpr int kSplitTok = 128;
constexpr int kMaxSplits = (kMaxTopK + kSplitTok - 1) / kSplitTok;

// emulated decode context parallelism: at most this many token shards
constexpr int kDcpMaxWorld = 16;

// the fused front end handles at most this many query rows (64 passes of 8)
constexpr int kFeMaxRows = 512;
constexpr int kFeMaxPasses = kFeMaxRows / 4;

// Byte offsets of the workspace regions (all 256-B aligned).
struct WsLayout {
  size_t err;       // int32 error word
  size_t q8;        // uint8 [rows][32][128] quantised indexer query
  size_t wq;        // float [rows][32] folded head weights
  size_t tiles;     // int32 [rows] inclusive prefix of 128-token tiles per scorer unit
  size_t state;     // int32 [rows][kRowState]
  size_t chunkinfo; // int32 [rows][max_chunks][2] (offset, count) of each top-k CTA's candidates
  size_t cand;      // uint64 [rows][kCandCap] top-k candidates (key << 32 | token)
  size_t gmax;      // uint32 [rows][gstride] order key of the largest score of each 32 tokens
  size_t gmax128;   // uint32 [rows][g128stride] the same per 128 tokens (dsa_decode; zero between calls)
  size_t opart;     // float [rows][splits][96][512]
  size_t lpart;     // float [rows][splits][96]
  size_t topk;      // int32 [rows][topk] (dsa_decode without topk_idx_out)
  size_t dcp_key;   // uint32 [rows][kDcpMaxWorld][topk] shard lists: bf16 keys by position
  size_t dcp_tok;   // int32 [rows][kDcpMaxWorld][topk] shard lists: tokens by position
  size_t dcp_cnt;   // int32 [rows][kDcpMaxWorld] shard list lengths
  size_t fe_part;   // fp32 [4][rows][128] the front end's key partial sums
  size_t fe_q;      // fp32 [rows][32][128] the front end's head outputs
  size_t fe_cnt;    // int32 [33][kFeMaxPasses] the front end's arrival counters
  size_t dcp_keys16;  // uint16 [rows][W][S] shard-major score keys, W * S <= cap + 8 * kDcpMaxWorld
  size_t scores;    // float [rows][cap]
  size_t total;
  int rows, cap, max_chunks, splits, gstride, g128stride;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// KV splits of the attention for top-k size `topk` (same function for sizing and launch).
inline int attention_splits(int topk) { return (topk + kSplitTok - 1) / kSplitTok; }

inline WsLayout ws_layout(const dsa_params_t& p) {
  WsLayout L{};
  L.rows = p.batch * p.n_q;
  L.cap = p.max_pages_per_req * p.page_size;
  L.max_chunks = (L.cap + kTopkChunk - 1) / kTopkChunk;
  L.splits = attention_splits(p.topk);
  L.gstride = ((L.cap >> 5) + 3) & ~3;
  L.g128stride = ((L.cap >> 7) + 3) & ~3;
  size_t o = 0;
  L.err = o; o = align256(o + 256);
  L.q8 = o; o = align256(o + size_t(L.rows) * kIdxHeads * kIdxDim);
  L.wq = o; o = align256(o + size_t(L.rows) * kIdxHeads * 4);
  L.tiles = o; o = align256(o + size_t(L.rows) * 4);
  L.state = o; o = align256(o + size_t(L.rows) * kRowState * 4);
  L.chunkinfo = o; o = align256(o + size_t(L.rows) * L.max_chunks * 2 * 4);
  L.cand = o; o = align256(o + size_t(L.rows) * kCandCap * 8);
  L.gmax = o; o = align256(o + size_t(L.rows) * L.gstride * 4);
  L.gmax128 = o; o = align256(o + size_t(L.rows) * L.g128stride * 4);
  L.opart = o; o = align256(o + size_t(L.rows) * L.splits * kHeads * kDNope * 4);
  L.lpart = o; o = align256(o + size_t(L.rows) * L.splits * kHeads * 4);
  L.topk = o; o = align256(o + size_t(L.rows) * p.topk * 4);
  L.dcp_key = o; o = align256(o + size_t(L.rows) * kDcpMaxWorld * p.topk * 4);
  L.dcp_tok = o; o = align256(o + size_t(L.rows) * kDcpMaxWorld * p.topk * 4);
  L.dcp_cnt = o; o = align256(o + size_t(L.rows) * kDcpMaxWorld * 4);
  L.fe_part = o; o = align256(o + size_t(4) * L.rows * kIdxDim * 4);
  L.fe_q = o; o = align256(o + size_t(L.rows) * kIdxHeads * kIdxDim * 4);
  L.fe_cnt = o; o = align256(o + size_t(kIdxHeads + 1) * kFeMaxPasses * 4);
  L.dcp_keys16 = o; o = align256(o + size_t(L.rows) * (size_t(L.cap) + 8 * kDcpMaxWorld) * 2);
  L.scores = o; o = align256(o + size_t(L.rows) * L.cap * 4);
  L.total = o;
  return L;
}

// Order-preserving 32-bit key of an fp32 score (larger score -> larger key;
// -0 and +0 share one key). Top-k compares scores only through this key.
__device__ __forceinline__ uint32_t score_order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Visible length of row (b, t): ctx_b - n_q + t + 1, or -1 when ctx_b is invalid.
__device__ __forceinline__ int row_visible_len(const int32_t* ctx_lens, int b, int t, int n_q,
                                               int cap, int* err) {
  int c = ctx_lens[b];
  if (c < n_q || c > cap) {
    if (t == 0 && threadIdx.x == 0) atomicOr(err, DSA_DEVERR_CTX);
    return -1;
  }
  return c - n_q + t + 1;
}

// ---------------------------------------------------------------- programmatic dependent launch
// Every kernel of the library is launched with programmatic stream
// serialisation, so the next kernel in the stream is scheduled as soon as the
// current one lets it (pdl_trigger, or the exit of all its CTAs) instead of
// after its completion and memory flush. Each kernel does only on-chip set-up
// (shared memory, barriers, TMEM) before pdl_wait, which returns once every
// earlier grid in the stream has completed and its memory is visible; no
// global access comes before it. Only the small query-quantisation kernel
// triggers early (the scorer's prologue then overlaps it); a waiting grid that
// shared SMs with a long-running one slowed that one down (measured), so the
// others let their dependents in when they exit.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Number of SMs of the current device.
int sm_count();
// Tiled TMA tensor map (cuTensorMapEncodeTiled through the runtime's driver entry point).
bool encode_map(CUtensorMap* m, CUtensorMapDataType dtype, const void* base, int rank, const uint64_t* dims,
                const uint64_t* strides, const uint32_t* box, bool swizzle128);

// ---------------------------------------------------------------- launchers
// (each returns cudaGetLastError() of its launches)

// The scorer's work units: the query rows of a request in groups of at most
// kMaxNQ (decode: one group per request; prefill: many). With token sharding
// ("预填充：按 token 而非按头分片注意力": each request cut into 2W slices, rank r
// taking slices r and 2W - 1 - r), a call covers only its rank's groups.
struct UnitMap {
  int rows_per_req;      // n_q
  int gsz;               // query rows per group: min(n_q, kMaxNQ)
  int groups;            // groups per request in this call
  int slice_groups;      // groups of the first slice (all of them without sharding)
  int slice_a, slice_b;  // first group of each slice
};

__host__ __device__ inline UnitMap unit_map(int n_q, int world, int rank) {
  UnitMap m;
  m.rows_per_req = n_q;
  m.gsz = n_q < kMaxNQ ? n_q : kMaxNQ;
  if (world <= 1) {
    m.groups = m.slice_groups = (n_q + m.gsz - 1) / m.gsz;
    m.slice_a = m.slice_b = 0;
  } else {  // n_q is a multiple of 2W x kMaxNQ
    m.slice_groups = n_q / (2 * world) / m.gsz;
    m.groups = 2 * m.slice_groups;
    m.slice_a = rank * m.slice_groups;
    m.slice_b = (2 * world - 1 - rank) * m.slice_groups;
  }
  return m;
}

__host__ __device__ __forceinline__ int unit_first_row(const UnitMap& m, int gl) {
  const int g = gl < m.slice_groups ? m.slice_a + gl : m.slice_b + (gl - m.slice_groups);
  return g * m.gsz;
}

// Work plan of the scorer, by one CTA of NT threads: tiles of 128 tokens (two
// pages) per unit, inclusive prefix over the units. A unit's context is its
// last row's: ctx_b - n_q + first + valid. An invalid context length gets no
// tiles and sets DSA_DEVERR_CTX.
template <int NT>
__device__ __forceinline__ void build_tile_plan(const int32_t* __restrict__ ctx_lens, int units, UnitMap m, int cap,
                                                int* __restrict__ tile_prefix, int* err) {
  constexpr int NW = NT / 32;
  __shared__ int wsum[NW];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int carry = 0;
  for (int u0 = 0; u0 < units; u0 += NT) {
    const int u = u0 + int(threadIdx.x);
    int n = 0;
    if (u < units) {
      const int b = u / m.groups;
      const int c = ctx_lens[b];
      if (c < m.rows_per_req || c > cap) {
        atomicOr(err, DSA_DEVERR_CTX);
      } else {
        const int first = unit_first_row(m, u - b * m.groups);
        const int valid = min(m.gsz, m.rows_per_req - first);
        n = (c - m.rows_per_req + first + valid + 127) >> 7;
      }
    }
    int x = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    int pre = carry;
    for (int i = 0; i < warp; ++i) pre += wsum[i];
    if (u < units) tile_prefix[u] = pre + x;
    for (int i = 0; i < NW; ++i) carry += wsum[i];
    __syncthreads();
  }
}

cudaError_t launch_idx_q_quant(const dsa_params_t& p, const WsLayout& L, char* ws, const void* q_idx,
                               const float* w, const int32_t* ctx_lens, cudaStream_t st, int world = 1,
                               int rank = 0);
// keep128: also keep the score keys' group maxima in the workspace (each 32
// tokens' largest, and each 128 tokens' folded by atomic max) for the top-k of
// the same call (dsa_decode, whose top-k clears the 128-token ones after use).
cudaError_t launch_indexer(const dsa_params_t& p, const WsLayout& L, char* ws, const void* key_pool,
                           const int32_t* block_table, const int32_t* ctx_lens, float* scores,
                           int64_t score_stride, cudaStream_t st, int world = 1, int rank = 0,
                           bool keep128 = false);
// have_gmax: the scorer of the same call has just written the group maxima of
// these scores into the workspace (dsa_decode); otherwise a first kernel
// computes them from the scores. lat_pool (dsa_decode, else null): the
// candidates' latent rows are prefetched into L2 for the attention.
cudaError_t launch_topk(const dsa_params_t& p, const WsLayout& L, char* ws, const float* scores,
                        int64_t score_stride, const int32_t* ctx_lens, const int32_t* block_table,
                        int32_t* topk_idx, int32_t* phys_rows, cudaStream_t st, bool have_gmax,
                        const void* lat_pool = nullptr);
cudaError_t launch_dcp_merge(const dsa_params_t& p, const WsLayout& L, char* ws, const float* scores,
                             int64_t score_stride, const int32_t* ctx_lens, int world, int32_t* topk_idx,
                             int32_t* stats, cudaStream_t st);
cudaError_t launch_dcp_lse_combine(int rows, int parts, const void* part_out, const float* part_lse, void* out,
                                   float* lse, cudaStream_t st);
struct FrontendIn {
  const void* c_q;
  const void* gamma;
  const void* w_q;
  const float* w;
  const void* x;
  const void* w_k;
  void* key_pool;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  void* q8_out;
  float* w_out;
  int d_c, d_model;
  float eps;
};
cudaError_t launch_idx_frontend(const dsa_params_t& p, const WsLayout& L, char* ws, const FrontendIn& in,
                                cudaStream_t st);
// early: the call follows this library's own kernels in one chain (dsa_decode),
// so the query and the set-up may be fetched before the wait on the top-k.
cudaError_t launch_sparse_mla(const dsa_params_t& p, const WsLayout& L, char* ws, const void* q,
                              const void* lat_pool, const int32_t* block_table,
                              const int32_t* ctx_lens, const int32_t* topk_idx, void* out,
                              float* lse, cudaStream_t st, bool early = false);

}  // namespace dsa
