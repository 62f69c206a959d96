// libdsa C ABI: host-side validation, workspace carving and stage launches.
#include <cstdint>
#include <cstring>
#include <initializer_list>

#include "dsa_internal.cuh"

using namespace dsa;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dsa_status_t check_params(const dsa_params_t* p) {
  if (!p) return DSA_ERR_INVALID;
  if (p->batch < 1 || p->n_q < 1 || p->max_pages_per_req < 1 || p->num_pages < 1) return DSA_ERR_INVALID;
  if (p->topk < 1) return DSA_ERR_INVALID;
  if (p->topk > kMaxTopK) return DSA_ERR_UNSUPPORTED;
  if (p->page_size != kPage || p->idx_heads != kIdxHeads || p->idx_dim != kIdxDim ||
      p->heads != kHeads || p->d_nope != kDNope || p->d_rope != kDRope)
    return DSA_ERR_UNSUPPORTED;
  if (p->key_fmt != DSA_KEY_FP8_132 && p->key_fmt != DSA_KEY_MXFP4_68) return DSA_ERR_INVALID;
  if (p->lat_fmt != DSA_LAT_FP8_576 && p->lat_fmt != DSA_LAT_NVFP4_352) return DSA_ERR_INVALID;
  const int64_t key_row = p->key_fmt == DSA_KEY_FP8_132 ? p->idx_dim + 4 : p->idx_dim / 2 + p->idx_dim / 32;
  const int64_t lat_row = p->lat_fmt == DSA_LAT_FP8_576 ? p->d_nope + p->d_rope
                                                        : p->d_nope / 2 + p->d_nope / 16 + p->d_rope;
  const int64_t key_page = int64_t(p->page_size) * key_row;
  const int64_t lat_page = int64_t(p->page_size) * lat_row;
  if (p->key_page_stride < key_page || (p->key_page_stride & 15)) return DSA_ERR_INVALID;
  if (p->lat_page_stride < lat_page || (p->lat_page_stride & 15)) return DSA_ERR_INVALID;
  if (!(p->softmax_scale > 0.f) || !(p->latent_scale > 0.f)) return DSA_ERR_INVALID;
  if (p->flags & ~int32_t(DSA_EMIT_PHYS_ROWS | DSA_Q_PREPARED)) return DSA_ERR_INVALID;
  // keep every index of the kernels inside int32 / the grid limits
  if (int64_t(p->max_pages_per_req) * p->page_size > (int64_t(1) << 28)) return DSA_ERR_UNSUPPORTED;
  if (int64_t(p->batch) * p->n_q > 65535) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

dsa_status_t check_ws(const dsa_params_t* p, void* ws, size_t ws_bytes, WsLayout* L) {
  if (!ws || !aligned16(ws)) return DSA_ERR_INVALID;
  *L = ws_layout(*p);
  if (ws_bytes < L->total) return DSA_ERR_WORKSPACE;
  return DSA_OK;
}

dsa_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA; }

dsa_status_t check_indexer_args(const dsa_params_t* p, const void* q_idx, const float* w,
                                const void* key_pool, const int32_t* bt, const int32_t* ctx) {
  if (!key_pool || !bt || !ctx || !aligned16(key_pool)) return DSA_ERR_INVALID;
  if (p->flags & DSA_Q_PREPARED)  // the query is already in the workspace (decode rows only)
    return p->n_q > kMaxNQ ? DSA_ERR_UNSUPPORTED : DSA_OK;
  if (!q_idx || !w) return DSA_ERR_INVALID;
  if (!aligned16(q_idx) || !aligned16(key_pool) || (reinterpret_cast<uintptr_t>(w) & 3)) return DSA_ERR_INVALID;
  return DSA_OK;
}

dsa_status_t check_mla_args(const void* q, const void* lat_pool, const int32_t* bt, const int32_t* ctx,
                            void* out) {
  if (!q || !lat_pool || !bt || !ctx || !out) return DSA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(lat_pool) || !aligned16(out)) return DSA_ERR_INVALID;
  return DSA_OK;
}

}  // namespace

extern "C" {

dsa_status_t dsa_workspace_size(const dsa_params_t* params, size_t* bytes) {
  dsa_status_t s = check_params(params);
  if (s != DSA_OK) return s;
  if (!bytes) return DSA_ERR_INVALID;
  *bytes = ws_layout(*params).total;
  return DSA_OK;
}

dsa_status_t dsa_indexer_scores(const dsa_params_t* params, const void* q_idx, const float* w,
                                const void* key_pool, const int32_t* block_table,
                                const int32_t* ctx_lens, float* scores, int64_t score_stride,
                                void* ws, size_t ws_bytes, cudaStream_t stream) {
  dsa_status_t s = check_params(params);
  if (s != DSA_OK) return s;
  if ((s = check_indexer_args(params, q_idx, w, key_pool, block_table, ctx_lens)) != DSA_OK) return s;
  if (!scores || !aligned16(scores) || score_stride < 1 || (score_stride & 3)) return DSA_ERR_INVALID;
  WsLayout L;
  if ((s = check_ws(params, ws, ws_bytes, &L)) != DSA_OK) return s;
  char* w8 = static_cast<char*>(ws);
  cudaError_t e = (params->flags & DSA_Q_PREPARED) ? cudaSuccess
                                                   : launch_idx_q_quant(*params, L, w8, q_idx, w, ctx_lens, stream);
  if (e == cudaSuccess)
    e = launch_indexer(*params, L, w8, key_pool, block_table, ctx_lens, scores, score_stride, stream);
  return cuda_status(e);
}

dsa_status_t dsa_indexer_prefill_scores(const dsa_params_t* params, int32_t world, int32_t rank, const void* q_idx,
                                        const float* w, const void* key_pool, const int32_t* block_table,
                                        const int32_t* ctx_lens, float* scores, int64_t score_stride, void* ws,
                                        size_t ws_bytes, cudaStream_t stream) {
  dsa_status_t s = check_params(params);
  if (s != DSA_OK) return s;
  if (world < 1 || rank < 0 || rank >= world) return DSA_ERR_INVALID;
  if (world > 1 && params->n_q % (2 * world * kMaxNQ)) return DSA_ERR_INVALID;
  if (params->flags & DSA_Q_PREPARED) return DSA_ERR_INVALID;
  if ((s = check_indexer_args(params, q_idx, w, key_pool, block_table, ctx_lens)) != DSA_OK) return s;
  if (!scores || !aligned16(scores) || score_stride < 1 || (score_stride & 3)) return DSA_ERR_INVALID;
  WsLayout L;
  if ((s = check_ws(params, ws, ws_bytes, &L)) != DSA_OK) return s;
  char* w8 = static_cast<char*>(ws);
  cudaError_t e = launch_idx_q_quant(*params, L, w8, q_idx, w, ctx_lens, stream, world, rank);
  if (e == cudaSuccess)
    e = launch_indexer(*params, L, w8, key_pool, block_table, ctx_lens, scores, score_stride, stream, world, rank);
  return cuda_status(e);
}

dsa_status_t dsa_topk(const dsa_params_t* params, const float* scores, int64_t score_stride,
                      const int32_t* ctx_lens, const int32_t* block_table, int32_t* topk_idx,
                      int32_t* phys_rows, void* ws, size_t ws_bytes, cudaStream_t stream) {
  dsa_status_t s = check_params(params);
  if (s != DSA_OK) return s;
  if (!scores || !aligned16(scores) || score_stride < 1 || (score_stride & 3)) return DSA_ERR_INVALID;
  if (!ctx_lens || !topk_idx) return DSA_ERR_INVALID;
  if (phys_rows && (!(params->flags & DSA_EMIT_PHYS_ROWS) || !block_table)) return DSA_ERR_INVALID;
  WsLayout L;
  if ((s = check_ws(params, ws, ws_bytes, &L)) != DSA_OK) return s;
  return cuda_status(launch_topk(*params, L, static_cast<char*>(ws), scores, score_stride, ctx_lens,
                                 block_table, topk_idx, phys_rows, stream, false));
}

dsa_status_t dsa_indexer_frontend(const dsa_params_t* params, const dsa_frontend_dims_t* dims, const void* c_q,
                                  const void* gamma_q, const void* w_q, const float* w, const void* x,
                                  const void* w_k, void* key_pool, const int32_t* block_table,
                                  const int32_t* ctx_lens, void* q8_out, float* w_out, void* ws, size_t ws_bytes,
                                  cudaStream_t stream) {
  dsa_status_t s = check_params(params);
  if (s != DSA_OK) return s;
  if (!dims) return DSA_ERR_INVALID;
  for (int d : {dims->d_c, dims->d_model})
    if (d < 256 || d > 8192 || (d % 256)) return DSA_ERR_UNSUPPORTED;
  if (!(dims->eps >= 0.f) || !(dims->eps < 1e30f)) return DSA_ERR_INVALID;
  if (int64_t(params->batch) * params->n_q > kFeMaxRows || params->n_q > kMaxNQ) return DSA_ERR_UNSUPPORTED;
  for (const void* ptr : {c_q, gamma_q, w_q, x, w_k, static_cast<const void*>(key_pool)})
    if (!ptr || !aligned16(ptr)) return DSA_ERR_INVALID;
  if (!w || (reinterpret_cast<uintptr_t>(w) & 3) || !block_table || !ctx_lens) return DSA_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(q8_out) & 3) || (reinterpret_cast<uintptr_t>(w_out) & 3)) return DSA_ERR_INVALID;
  WsLayout L;
  if ((s = check_ws(params, ws, ws_bytes, &L)) != DSA_OK) return s;
  FrontendIn in{c_q, gamma_q, w_q, w, x, w_k, key_pool, block_table, ctx_lens, q8_out, w_out,
                dims->d_c, dims->d_model, dims->eps};
  return cuda_status(launch_idx_frontend(*params, L, static_cast<char*>(ws), in, stream));
}

dsa_status_t dsa_dcp_topk_merge(const dsa_params_t* params, const float* scores, int64_t score_stride,
                                const int32_t* ctx_lens, int32_t world, int32_t* topk_idx, int32_t* stats,
                                void* ws, size_t ws_bytes, cudaStream_t stream) {
  dsa_status_t s = check_params(params);
  if (s != DSA_OK) return s;
  if (!scores || !aligned16(scores) || score_stride < 1 || (score_stride & 3)) return DSA_ERR_INVALID;
  if (!ctx_lens || !topk_idx) return DSA_ERR_INVALID;
  if (world < 1 || world > dsa::kDcpMaxWorld) return DSA_ERR_INVALID;
  WsLayout L;
  if ((s = check_ws(params, ws, ws_bytes, &L)) != DSA_OK) return s;
  return cuda_status(launch_dcp_merge(*params, L, static_cast<char*>(ws), scores, score_stride, ctx_lens, world,
                                      topk_idx, stats, stream));
}

dsa_status_t dsa_lse_combine(const dsa_params_t* params, int32_t parts, const void* part_out,
                             const float* part_lse, void* out, float* lse, cudaStream_t stream) {
  dsa_status_t s = check_params(params);
  if (s != DSA_OK) return s;
  if (parts < 1 || parts > dsa::kDcpMaxWorld) return DSA_ERR_INVALID;
  if (!part_out || !part_lse || !out || !aligned16(part_out) || !aligned16(out)) return DSA_ERR_INVALID;
  return cuda_status(
      launch_dcp_lse_combine(params->batch * params->n_q, parts, part_out, part_lse, out, lse, stream));
}

dsa_status_t dsa_sparse_mla_decode(const dsa_params_t* params, const void* q, const void* lat_pool,
                                   const int32_t* block_table, const int32_t* ctx_lens,
                                   const int32_t* topk_idx, void* out, float* lse, void* ws,
                                   size_t ws_bytes, cudaStream_t stream) {
  dsa_status_t s = check_params(params);
  if (s != DSA_OK) return s;
  if ((s = check_mla_args(q, lat_pool, block_table, ctx_lens, out)) != DSA_OK) return s;
  if (!topk_idx) return DSA_ERR_INVALID;
  WsLayout L;
  if ((s = check_ws(params, ws, ws_bytes, &L)) != DSA_OK) return s;
  return cuda_status(launch_sparse_mla(*params, L, static_cast<char*>(ws), q, lat_pool, block_table,
                                       ctx_lens, topk_idx, out, lse, stream));
}

dsa_status_t dsa_decode(const dsa_params_t* params, const void* q_idx, const float* w,
                        const void* key_pool, const void* q, const void* lat_pool,
                        const int32_t* block_table, const int32_t* ctx_lens, void* out, float* lse,
                        int32_t* topk_idx_out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  dsa_status_t s = check_params(params);
  if (s != DSA_OK) return s;
  if ((s = check_indexer_args(params, q_idx, w, key_pool, block_table, ctx_lens)) != DSA_OK) return s;
  if ((s = check_mla_args(q, lat_pool, block_table, ctx_lens, out)) != DSA_OK) return s;
  WsLayout L;
  if ((s = check_ws(params, ws, ws_bytes, &L)) != DSA_OK) return s;
  char* w8 = static_cast<char*>(ws);
  if (!topk_idx_out) topk_idx_out = reinterpret_cast<int32_t*>(w8 + L.topk);
  float* scores = reinterpret_cast<float*>(w8 + L.scores);
  cudaError_t e = (params->flags & DSA_Q_PREPARED) ? cudaSuccess
                                                   : launch_idx_q_quant(*params, L, w8, q_idx, w, ctx_lens, stream);
  if (e == cudaSuccess)
    e = launch_indexer(*params, L, w8, key_pool, block_table, ctx_lens, scores, L.cap, stream, 1, 0, true);
  if (e == cudaSuccess)
    e = launch_topk(*params, L, w8, scores, L.cap, ctx_lens, block_table, topk_idx_out, nullptr, stream, true,
                    lat_pool);
  if (e == cudaSuccess)
    e = launch_sparse_mla(*params, L, w8, q, lat_pool, block_table, ctx_lens, topk_idx_out, out, lse,
                          stream, true);
  return cuda_status(e);
}

dsa_status_t dsa_get_device_error(void* ws, cudaStream_t stream, int32_t* code) {
  if (!ws || !code) return DSA_ERR_INVALID;
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof(int32_t), stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  *code = v;
  return (v & DSA_DEVERR_TIMEOUT) ? DSA_ERR_TIMEOUT : DSA_OK;
}

const char* dsa_status_string(dsa_status_t status) {
  switch (status) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID: return "DSA_ERR_INVALID: invalid argument";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED: size or format not implemented";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE: workspace too small";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA: CUDA launch or runtime error";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT: device wait gave up";
  }
  return "unknown dsa_status_t";
}

}  // extern "C"
