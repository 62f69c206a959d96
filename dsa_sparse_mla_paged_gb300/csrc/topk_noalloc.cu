// dsa_topk_noalloc: the exact top-k stage without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they select
// tokens: a plugin inside an inference server whose memory pool owns every
// device byte, code running in a real-time decode loop that must not call
// into the allocator (cudaMalloc can synchronise the device), or a C caller
// that is handed only input and output pointers. For them this entry point
// keeps the top-k scratch (per-row selection state, per-chunk candidate
// offsets, the candidate buffer, the rows' 32- and 128-token score maxima) in one
// file-scope device array that every GPU loading the library holds until the
// process exits.
#include <mutex>

#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kNoAllocMaxRows = 64;                 // batch * n_q
constexpr int kNoAllocMaxCtx = 1 << 20;             // max_pages_per_req * page_size
constexpr size_t kNoAllocBytes =
    256 +                                                                        // error word
    size_t(kNoAllocMaxRows) * kRowState * 4 +                                    // row state
    size_t(kNoAllocMaxRows) * (kNoAllocMaxCtx / kTopkChunk) * 2 * 4 +            // chunk (offset, count)
    size_t(kNoAllocMaxRows) * kCandCap * 8 +                                     // candidates
    size_t(kNoAllocMaxRows) * (kNoAllocMaxCtx / 32) * 4 +                        // 32-token maxima
    size_t(kNoAllocMaxRows) * (kNoAllocMaxCtx / 128) * 4 +                       // 128-token maxima
    6 * 256;                                                                     // region alignment

// The scratch itself (about 15.2 MB). Only host code below takes its address.
static __device__ __align__(256) unsigned char g_topk_scratch[kNoAllocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

// The top-k regions of a workspace, packed into the static array. Every call
// clears the per-row state in its first kernel, so nothing needs clearing here.
WsLayout noalloc_layout(const dsa_params_t& p) {
  WsLayout L{};
  L.rows = p.batch * p.n_q;
  L.cap = p.max_pages_per_req * p.page_size;
  L.max_chunks = (L.cap + kTopkChunk - 1) / kTopkChunk;
  L.splits = 1;
  L.gstride = ((L.cap >> 5) + 3) & ~3;
  L.g128stride = ((L.cap >> 7) + 3) & ~3;
  size_t o = 0;
  L.err = o; o = align256(o + 256);
  L.state = o; o = align256(o + size_t(L.rows) * kRowState * 4);
  L.chunkinfo = o; o = align256(o + size_t(L.rows) * L.max_chunks * 2 * 4);
  L.cand = o; o = align256(o + size_t(L.rows) * kCandCap * 8);
  L.gmax = o; o = align256(o + size_t(L.rows) * L.gstride * 4);
  L.gmax128 = o; o = align256(o + size_t(L.rows) * L.g128stride * 4);
  L.total = o;
  return L;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status_t dsa_topk_noalloc(const dsa_params_t* params, const float* scores, int64_t score_stride,
                                         const int32_t* ctx_lens, const int32_t* block_table, int32_t* topk_idx,
                                         int32_t* phys_rows, cudaStream_t stream) {
  if (!params) return DSA_ERR_INVALID;
  size_t ws_bytes = 0;
  dsa_status_t s = dsa_workspace_size(params, &ws_bytes);  // full parameter validation
  if (s != DSA_OK) return s;
  if (int64_t(params->batch) * params->n_q > kNoAllocMaxRows ||
      int64_t(params->max_pages_per_req) * params->page_size > kNoAllocMaxCtx)
    return DSA_ERR_UNSUPPORTED;
  if (!scores || (reinterpret_cast<uintptr_t>(scores) & 15) || score_stride < 1 || (score_stride & 3))
    return DSA_ERR_INVALID;
  if (!ctx_lens || !topk_idx) return DSA_ERR_INVALID;
  if (phys_rows && (!(params->flags & DSA_EMIT_PHYS_ROWS) || !block_table)) return DSA_ERR_INVALID;
  const WsLayout L = noalloc_layout(*params);
  if (L.total > kNoAllocBytes) return DSA_ERR_UNSUPPORTED;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return DSA_ERR_CUDA;
  const cudaError_t e = launch_topk(*params, L, static_cast<char*>(base), scores, score_stride, ctx_lens,
                                    block_table, topk_idx, phys_rows, stream, false);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
