/*
 * dsa.h -- C ABI of libdsa: the decode step of a DeepSeek-style sparse
 * attention (DSA) layer over a paged FP8 cache, for one GB300 GPU (sm_103a).
 *
 * The step has three stages, as the vLLM article "vLLM 为 Kimi K3.1 Pro 提供
 * Day-0 支持" states them in its section "K3.1 Pro 中的稀疏注意力" (sparse
 * attention in K3.1 Pro):
 *   1. a lightning indexer scores every earlier token of a request with 32
 *      light heads over a per-token FP8 index key (128 E4M3 values + one fp32
 *      scale = 132 B):  score(t, s) = sum_h w_h * ReLU(q_h . k_s);
 *   2. the 2,048 best-scoring tokens are kept (exact top-k);
 *   3. MLA attention runs exactly over those tokens only, reading each one's
 *      576-B FP8 latent (512 "nope" + 64 "rope" values) shared by all 96
 *      query heads.
 * The caches are paged; the kernels reach them through a block table, which
 * maps each request's logical pages to physical pages (section "面向三种状态的
 * KV 缓存" describes the translation to page addresses done before each step).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Notation: B = params.batch requests, n_q = query tokens per request,
 *   ctx_b = context length of request b INCLUDING its n_q new tokens (whose
 *   keys and latents are already in the cache), L_{b,t} = ctx_b - n_q + t + 1
 *   = tokens query t may see (causal within the step), K = params.topk.
 *   A "row" is one (b, t) pair; rows are ordered b-major: row = b * n_q + t.
 * - Ownership: the caller owns every buffer, including the workspace. The
 *   library never allocates, frees or synchronises (dsa_get_device_error is
 *   the one call that synchronises the stream it is given).
 * - All pointers except `params`, `bytes` and `code` are DEVICE pointers.
 *   All calls are asynchronous on `stream` (0 = the legacy default stream).
 * - Host validation: null pointers, unsupported sizes or formats, misaligned
 *   buffers (q, q_idx, pools, scores, workspace: 16 B; page strides: a
 *   multiple of 16 B) and a short workspace are rejected with
 *   DSA_ERR_INVALID / DSA_ERR_UNSUPPORTED / DSA_ERR_WORKSPACE before anything
 *   is launched.
 * - Device-detected bad data (a block-table entry outside [0, num_pages), a
 *   ctx_b outside [n_q, max_pages_per_req * page_size], a top-k index outside
 *   [-1, L_{b,t})) never traps: the kernels skip the access, leave the affected
 *   row's results unspecified (finite), and OR a bit into the workspace's error
 *   word, which dsa_get_device_error reads back.
 * - The workspace must be zero-filled once after allocation; afterwards the
 *   library keeps it consistent itself. Calls that share one workspace must
 *   be ordered (same stream, or synchronised by the caller).
 * - Launch failures return DSA_ERR_CUDA.
 * - Results are deterministic: the same inputs give the same bits, whatever
 *   the batch composition.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same definition as the CUDA runtime's. */
typedef struct CUstream_st* cudaStream_t;

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID = 1,      /* a null pointer, a bad size or a misaligned buffer */
  DSA_ERR_UNSUPPORTED = 2,  /* a size or format this build does not implement */
  DSA_ERR_WORKSPACE = 3,    /* ws_bytes below dsa_workspace_size() */
  DSA_ERR_CUDA = 4,         /* a CUDA launch or runtime call failed */
  DSA_ERR_TIMEOUT = 5       /* a bounded device wait gave up (dsa_get_device_error) */
} dsa_status_t;

/* Index-key formats (section "面向三种状态的 KV 缓存": index key 132 B in FP8,
 * 68 B in MXFP4). Page layout of one page of page_size tokens:
 *   DSA_KEY_FP8_132 : [page_size x 128 B E4M3][page_size x 4 B fp32 scale]
 *   DSA_KEY_MXFP4_68: [page_size x 64 B E2M1 pairs][page_size x 4 B E8M0]  */
typedef enum { DSA_KEY_FP8_132 = 0, DSA_KEY_MXFP4_68 = 1 } dsa_key_fmt_t;

/* Latent formats (same section: 576 B in FP8, 352 B in NVFP4). A page is
 * page_size consecutive rows:
 *   DSA_LAT_FP8_576  : [512 E4M3 nope][64 E4M3 rope]
 *   DSA_LAT_NVFP4_352: [256 B E2M1 pairs][32 B E4M3 scale per 16][64 B E4M3 rope] */
typedef enum { DSA_LAT_FP8_576 = 0, DSA_LAT_NVFP4_352 = 1 } dsa_lat_fmt_t;

/* flags */
#define DSA_EMIT_PHYS_ROWS 0x1  /* dsa_topk also writes physical cache rows */
#define DSA_Q_PREPARED 0x2      /* dsa_indexer_scores / dsa_decode take the quantised query,
                                   the folded weights and the scorer's plan that
                                   dsa_indexer_frontend left in the same workspace (same
                                   params and ctx_lens); q_idx and w may be NULL;
                                   n_q <= 8 (else DSA_ERR_UNSUPPORTED) */

/* Device error word bits (dsa_get_device_error). */
#define DSA_DEVERR_BLOCK_TABLE 0x1  /* a block-table entry outside [0, num_pages) */
#define DSA_DEVERR_CTX 0x2          /* ctx_b outside [n_q, max_pages_per_req * page_size] */
#define DSA_DEVERR_TOPK_INDEX 0x4   /* a top-k index outside [-1, L_{b,t}) */
#define DSA_DEVERR_TIMEOUT 0x8      /* a bounded in-kernel wait gave up (results unspecified) */

typedef struct {
  int32_t batch;              /* B >= 1 */
  int32_t n_q;                /* query tokens per request (decode 1..8, a prefill chunk more;
                                 batch * n_q <= 65535); the scorer takes them 8 at a time */
  int32_t topk;               /* K, 1..2048 (the article's K is 2048) */
  int32_t page_size;          /* tokens per page; this build: 64 */
  int32_t max_pages_per_req;  /* row stride of block_table (entries); ctx_b <= this * page_size */
  int32_t idx_heads;          /* 32 */
  int32_t idx_dim;            /* 128 */
  int32_t heads;              /* 96 */
  int32_t d_nope;             /* 512 */
  int32_t d_rope;             /* 64 */
  int32_t key_fmt;            /* dsa_key_fmt_t */
  int32_t lat_fmt;            /* dsa_lat_fmt_t */
  int64_t key_page_stride;    /* bytes between key pages (>= page bytes, multiple of 16) */
  int64_t lat_page_stride;    /* bytes between latent pages (>= page bytes, multiple of 16) */
  int32_t num_pages;          /* pages in each pool (bounds check of block-table entries) */
  float softmax_scale;        /* e.g. 1/sqrt(192) */
  float latent_scale;         /* per-tensor latent scale (1.0 for unscaled) */
  int32_t flags;              /* DSA_EMIT_PHYS_ROWS */
} dsa_params_t;

/* Bytes of workspace the calls below need for `params`. The workspace holds
 * the device error word, the quantised indexer query, the top-k candidates,
 * the split-KV partial outputs and (for dsa_decode) the fp32 scores of every
 * row over max_pages_per_req * page_size tokens. */
dsa_status_t dsa_workspace_size(const dsa_params_t* params, size_t* bytes);

/* Stage 1, the lightning indexer ("K3.1 Pro 中的稀疏注意力"), with the FP8 query
 * quantisation of the fused front end ("低延迟解码：融合的 DSA 解码路径": the
 * indexer query is quantised to FP8 with its scale folded into the head
 * weights):
 *   amax_h = max_d |q[h,d]|, q8_h = E4M3_rne_sat(q_h * (448/amax_h)),
 *   w'_h = w_h * (amax_h/448)        (IEEE fp32, round to nearest);
 *   score[row][s] = sum_h w'_h * max(0, q8_h . k_s)
 * for s < L_{b,t}; entries s >= L_{b,t} are left untouched. The key k_s is
 * E4M3(k) * scale_s (DSA_KEY_FP8_132) or E2M1(k) * 2^(e_blk - 127) with one
 * E8M0 exponent e_blk per 32 values (DSA_KEY_MXFP4_68, section "量化：原生 MXFP4
 * 索引器"); exact while a token's four exponents lie within 14 of each other;
 * beyond that each value of a block more than 14 below the token's largest is
 * off by at most 2^(e_max - 143) (it is scored as the nearest multiple of 2^-9
 * of 2^(e_max - 133)).
 *   q_idx  bf16 [B, n_q, idx_heads, idx_dim]      (16-B aligned)
 *   w      fp32 [B, n_q, idx_heads]
 *   key_pool   num_pages pages of key_page_stride bytes (16-B aligned)
 *   block_table int32 [B, max_pages_per_req]; entries past ceil(ctx_b/page_size) unused
 *   ctx_lens   int32 [B]
 *   scores fp32 [B * n_q, score_stride], score_stride >= max ctx, multiple of 4 */
dsa_status_t dsa_indexer_scores(const dsa_params_t* params, const void* q_idx, const float* w,
                                const void* key_pool, const int32_t* block_table,
                                const int32_t* ctx_lens, float* scores, int64_t score_stride,
                                void* ws, size_t ws_bytes, cudaStream_t stream);

/* Stage 1 for a prefill chunk with token sharding ("预填充：按 token 而非按头分片注意力":
 * the GPUs divide a prefill's query tokens, not its heads, and pair slices so
 * that causal work evens out: with 8 GPUs and 16 slices, GPU r has r and 15 - r).
 * Here: the n_q rows of each request are cut into 2 * world
 * equal slices and the call scores only rank's two slices, r and
 * 2 * world - 1 - r, exactly as dsa_indexer_scores would (scores of the other
 * rows are not written). world = 1 scores every row (= dsa_indexer_scores).
 *   world, rank  1 <= world, 0 <= rank < world; world > 1 needs n_q to be a
 *                multiple of 16 * world (slices of whole 8-row groups)
 * Other arguments, layouts and errors as dsa_indexer_scores (no DSA_Q_PREPARED). */
dsa_status_t dsa_indexer_prefill_scores(const dsa_params_t* params, int32_t world, int32_t rank, const void* q_idx,
                                        const float* w, const void* key_pool, const int32_t* block_table,
                                        const int32_t* ctx_lens, float* scores, int64_t score_stride, void* ws,
                                        size_t ws_bytes, cudaStream_t stream);

/* Stage 2, exact top-k ("K3.1 Pro 中的稀疏注意力": keep the top 2,048 tokens).
 * For each row: the min(K, L) tokens with the highest fp32 score, ties going to
 * the lower token index (-0 == +0), written in ascending token order to
 * topk_idx[row][0 .. min(K, L)), the rest of the row set to -1.
 *   scores   fp32 [B * n_q, score_stride] (only s < L_{b,t} is read)
 *   topk_idx int32 [B * n_q, K]
 *   phys_rows int32 [B * n_q, K] or NULL: page * page_size + slot of each
 *            selected token ("融合的 indexer ... 输出注意力读取的物理 KV 行"),
 *            -1 padded; needs DSA_EMIT_PHYS_ROWS and block_table. */
dsa_status_t dsa_topk(const dsa_params_t* params, const float* scores, int64_t score_stride,
                      const int32_t* ctx_lens, const int32_t* block_table, int32_t* topk_idx,
                      int32_t* phys_rows, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Stage 3, exact absorbed-MLA attention over the selected tokens
 * ("K3.1 Pro 中的稀疏注意力": attention runs exactly, but only over those tokens).
 * For each row and head h, with c_s = E4M3(latent_s) * latent_scale
 * (DSA_LAT_FP8_576), or for DSA_LAT_NVFP4_352 the 512 nope values
 * E2M1 * E4M3(block scale of 16) and the 64 rope values E4M3, all times
 * latent_scale (recipes page, "NVFP4 KV cache"):
 *   logit_s = softmax_scale * q_h . c_s  (576 dims), s in S = {topk_idx >= 0}
 *   out[h]  = sum_s softmax(logit)_s * c_s[0:512]          (bf16, RNE)
 *   lse[h]  = ln sum_s exp(logit_s)                        (fp32)
 * An empty S gives out = 0 and lse = -inf.
 *   q        bf16 [B, n_q, heads, d_nope + d_rope] (16-B aligned)
 *   lat_pool num_pages pages of lat_page_stride bytes (16-B aligned)
 *   topk_idx int32 [B * n_q, K] logical token indices, -1 = unused slot
 *   out      bf16 [B, n_q, heads, d_nope]
 *   lse      fp32 [B, n_q, heads] or NULL */
dsa_status_t dsa_sparse_mla_decode(const dsa_params_t* params, const void* q, const void* lat_pool,
                                   const int32_t* block_table, const int32_t* ctx_lens,
                                   const int32_t* topk_idx, void* out, float* lse, void* ws,
                                   size_t ws_bytes, cudaStream_t stream);

/* The fused step: stage 1 -> stage 2 -> stage 3 on one stream, no host sync.
 * topk_idx_out (int32 [B * n_q, K]) may be NULL; the scores stay in the
 * workspace. Arguments as above. */
dsa_status_t dsa_decode(const dsa_params_t* params, const void* q_idx, const float* w,
                        const void* key_pool, const void* q, const void* lat_pool,
                        const int32_t* block_table, const int32_t* ctx_lens, void* out,
                        float* lse, int32_t* topk_idx_out, void* ws, size_t ws_bytes,
                        cudaStream_t stream);

/* Widths of the fused front end's inputs (not fixed by the article). */
typedef struct {
  int32_t d_c;      /* query latent width, the query norm's input: 256 .. 8192, a multiple of 256 */
  int32_t d_model;  /* hidden width, the key projection's input: 256 .. 8192, a multiple of 256 */
  float eps;        /* RMS norm epsilon, >= 0 */
} dsa_frontend_dims_t;

/* The fused indexer front end ("低延迟解码：融合的 DSA 解码路径": one kernel for the
 * work ahead of the scorer -- normalise the query latent, project it onto the
 * indexer heads, make it FP8 with the scale moved into the head weights, and
 * produce the new token's index key). For row (b, t):
 *   n  = bf16(c_q / sqrt(mean(c_q^2) + eps) * gamma_q)     (fp32 arithmetic)
 *   q  = bf16(n @ w_q^T), q[h] = q[128 h .. 128 h + 127]   (fp32 accumulation)
 *   q8[h] = E4M3_rne_satfinite(q[h] * (448 / amax_h)), w'[h] = w[h] * (amax_h / 448)
 *        (the recipe of dsa_indexer_scores' own quantisation)
 *   k  = bf16(x @ w_k^T), quantised to the key format (FP8: one fp32 scale
 *        amax / 448 per token, codes E4M3(k * 448 / amax); MXFP4: per 32 values
 *        E8M0 exponent e = floor(log2 amax) - 2 and E2M1(v / 2^e), nearest-even,
 *        saturating) and written to the cache slot of token ctx_b - n_q + t.
 * The quantised query, w' and the scorer's plan go to the workspace, where a
 * following dsa_indexer_scores / dsa_decode with DSA_Q_PREPARED reads them.
 *   c_q     bf16 [B * n_q, d_c]          gamma_q bf16 [d_c]
 *   w_q     bf16 [32 * 128, d_c]         (a linear layer's [out, in] weight)
 *   w       fp32 [B * n_q, 32]           head weights
 *   x       bf16 [B * n_q, d_model]      w_k bf16 [128, d_model]
 *   key_pool written at one slot per row (16-B aligned, like every bf16 input)
 *   q8_out  E4M3 [B * n_q, 32, 128] or NULL; w_out fp32 [B * n_q, 32] or NULL (copies)
 * Limits: n_q <= 8 and B * n_q <= 512 (else DSA_ERR_UNSUPPORTED).
 * Errors: a row with an invalid ctx_b or block-table entry writes no key and
 * sets DSA_DEVERR_CTX / DSA_DEVERR_BLOCK_TABLE in the workspace. */
dsa_status_t dsa_indexer_frontend(const dsa_params_t* params, const dsa_frontend_dims_t* dims, const void* c_q,
                                  const void* gamma_q, const void* w_q, const float* w, const void* x,
                                  const void* w_k, void* key_pool, const int32_t* block_table,
                                  const int32_t* ctx_lens, void* q8_out, float* w_out, void* ws, size_t ws_bytes,
                                  cudaStream_t stream);

/* Stage 2 as W decode-context-parallel GPUs would run it, emulated on one GPU
 * ("vLLM 为 Kimi K3.1 Pro 提供 Day-0 支持", section "长上下文：带稀疏 indexer 的
 * decode 上下文并行", "流量减少 10× 的精确 top-k 合并"). Shard r of a row holds
 * the tokens s < L with s mod W == r. Each shard orders its tokens by the
 * round-to-nearest-even bf16 of the score (higher first, -0 == +0), then by
 * token; j is a token's position in that order. A candidate travels as the
 * 32-bit word key16 << 16 | (4095 - j) << 4 | (15 - r), key16 being the
 * order-preserving 16-bit key of the bf16 score, so word order is the global
 * order (key desc, position asc, shard asc).
 *   exchange 1  every shard sends its first m = ceil(1.5 K / W) candidates
 *               (at most K; all it holds, if fewer); the K largest words are
 *               selected.
 *   exchange 2  only if some shard holds more than m tokens among its first K
 *               and all m it sent were selected: each such shard sends its
 *               first min(K, L_r) and the K largest words are selected again.
 * The result is the top min(K, L) of all tokens under the global order, written
 * like dsa_topk (ascending token order, -1 padded); rows with L <= K keep every
 * token. Against dsa_topk run on the bf16-rounded scores it is identical for
 * W = 1; for W > 1 it keeps the same tokens above the K-th bf16 value and as
 * many at that value, but picks among the tokens tied at it by (position in
 * shard, shard) rather than by token index, so that pick depends on W. Against
 * dsa_topk on the fp32 scores it also differs where bf16 rounding reorders.
 *   world   W, 1 .. 16 (shard and position must fit the word's 16 low bits)
 *   scores, score_stride, ctx_lens, topk_idx  as dsa_topk
 *   stats   int32 [B * n_q, 2] or NULL: per row the bit mask of shards that
 *           re-sent in exchange 2, and the words all shards sent in both
 *           exchanges (a row with L <= K reports 0 and L)
 * Errors as dsa_topk; the workspace holds the shard lists. */
dsa_status_t dsa_dcp_topk_merge(const dsa_params_t* params, const float* scores, int64_t score_stride,
                                const int32_t* ctx_lens, int32_t world, int32_t* topk_idx, int32_t* stats,
                                void* ws, size_t ws_bytes, cudaStream_t stream);

/* The cross-shard step of decode context parallelism (same section as
 * dsa_dcp_topk_merge): each of `parts` shards attended over its own winners
 * (dsa_sparse_mla_decode with the other shards' slots set to -1), and the
 * partial results are merged by their log-sum-exp:
 *   lse[h] = ln sum_i exp(lse_i[h]),  out[h] = sum_i exp(lse_i[h] - lse[h]) * out_i[h]
 * in fp32, out rounded to bf16 (RNE). A part with lse_i = -inf (no tokens)
 * adds nothing; if every part is empty, out = 0 and lse = -inf.
 *   parts    1 .. 16
 *   part_out bf16 [parts][B * n_q][heads][d_nope] (16-B aligned)
 *   part_lse fp32 [parts][B * n_q][heads]
 *   out      bf16 [B * n_q][heads][d_nope] (16-B aligned); lse fp32 [B * n_q][heads] or NULL
 * No workspace; no device error word. */
dsa_status_t dsa_lse_combine(const dsa_params_t* params, int32_t parts, const void* part_out,
                             const float* part_lse, void* out, float* lse, cudaStream_t stream);

/* Stage 2 without a workspace, for callers that cannot allocate device memory
 * when they select tokens (a plugin whose host owns every device byte, a
 * real-time loop that must not enter the allocator, a caller handed only input
 * and output pointers). The article has no counterpart: this is a deployment
 * variant of dsa_topk, with the same arguments minus the workspace and the same
 * results bit for bit.
 * - Scratch: one static device array of about 15.2 MB inside libdsa, held by
 *   every GPU that loads the library until the process exits. The call
 *   allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 * - Limits: batch * n_q <= 64 and max_pages_per_req * page_size <= 1,048,576;
 *   larger problems return DSA_ERR_UNSUPPORTED and launch nothing.
 * - The first call on a device loads libdsa's device code on it (with CUDA's
 *   default lazy module loading, this is when the array is reserved) and looks
 *   up the array's address; that first call may allocate and synchronise.
 *   Make it outside any real-time loop and before any stream capture: later
 *   calls on that device allocate nothing.
 * - The address is cached per device for the life of the process: after a
 *   cudaDeviceReset the cached address is stale and the call must not be used
 *   on that device again.
 * - Every call shares the array: calls whose kernels overlap on the GPU (two
 *   streams, two threads) race and give wrong results; order them. Each call
 *   clears the parts that must start at zero itself.
 * - Bad data found on the device is skipped as in dsa_topk, but there is no
 *   workspace error word to report it through. */
dsa_status_t dsa_topk_noalloc(const dsa_params_t* params, const float* scores, int64_t score_stride,
                              const int32_t* ctx_lens, const int32_t* block_table, int32_t* topk_idx,
                              int32_t* phys_rows, cudaStream_t stream);

/* Synchronises `stream`, then reads and clears the device error word of the
 * workspace `ws` into *code (0 = no error; DSA_DEVERR_* bits otherwise).
 * Returns DSA_ERR_TIMEOUT (with *code written) when the word holds
 * DSA_DEVERR_TIMEOUT: a bounded in-kernel wait gave up, the kernel unwound
 * (no copy or MMA left in flight, tensor memory freed) and the results of the
 * calls since the last check are unspecified; the context and the workspace
 * stay usable. DSA_OK otherwise; DSA_ERR_CUDA if the copy fails. */
dsa_status_t dsa_get_device_error(void* ws, cudaStream_t stream, int32_t* code);

/* Diagnostics: runs the bounded-wait abort path on purpose. One warp waits on
 * an mbarrier that nothing arrives on, gives up after `poll_limit` polls
 * (1 <= poll_limit <= 2^20) and ORs DSA_DEVERR_TIMEOUT into the error word of
 * `ws` (>= 4 bytes, 16-B aligned), as a pipeline kernel that timed out does.
 * Not part of the decode path. */
dsa_status_t dsa_selftest_wait_timeout(void* ws, size_t ws_bytes, uint32_t poll_limit, cudaStream_t stream);

/* Static description of a status code. */
const char* dsa_status_string(dsa_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
