"""The DSA decode step written out plainly in float64 -- TEST INFRASTRUCTURE ONLY.

Notation: request b, query token t (0 <= t < n_q), context length ctx_b
(including the step's n_q new tokens, whose keys and latents the step has
already written to the cache), visible length L_{b,t} = ctx_b - n_q + t + 1,
top-k K = 2048, page size P = 64.

Sources (page title, section):
  [SA]   "vLLM 为 Kimi K3.1 Pro 提供 Day-0 支持", "K3.1 Pro 中的稀疏注意力"
  [KV3]  same page, "面向三种状态的 KV 缓存"
  [KVF]  same page, "KV 缓存占用"
  [FUSE] same page, "低延迟解码：融合的 DSA 解码路径"
  [DCP]  same page, "长上下文：带稀疏 indexer 的 decode 上下文并行"
  [MX4]  same page, "量化：原生 MXFP4 索引器"
  [NEWS] "vLLM Adds Day-0 Support for Moonshot AI's Kimi K3.1 Pro",
         "Sparse attention targets long-context costs"
  [REC]  "moonshotai/Kimi-K3.1-Pro", "NVFP4 KV cache"
"""
from __future__ import annotations

import math

import numpy as np

from .formats import (
    bf16_decode,
    e2m1_unpack,
    e4m3_decode,
    e4m3_encode_rne_satfinite,
    e8m0_decode,
    f32_from_bytes,
)

IDX_HEADS, IDX_DIM = 32, 128
HEADS, D_NOPE, D_ROPE = 96, 512, 64
D_QK = D_NOPE + D_ROPE


def visible_len(ctx_b: int, n_q: int, t: int) -> int:
    """Tokens query t of a step may see.

    Reading: the pages say the indexer scores "every earlier token" [SA] and
    that the fused path writes the new token's latent and index key into the
    cache before attention [FUSE]; so the new tokens are part of the context and
    query t of n_q sees positions 0 .. ctx_b - n_q + t (causal within the step).
    """
    return int(ctx_b) - n_q + t + 1


# ----------------------------------------------------------------------------
# page translation [KV3]: logical token s -> (physical page, slot)
# ----------------------------------------------------------------------------

def token_pages(block_table_row: np.ndarray, L: int, page_size: int):
    s = np.arange(L, dtype=np.int64)
    return block_table_row[s // page_size].astype(np.int64), s % page_size


def read_fp8_keys(key_pool, pages, slots, page_size):
    """E4M3 codes [n,128] and fp32 scales [n] of the given tokens.

    Page layout (this library's, the article fixes only 132 B/token):
    [page_size x 128 B values][page_size x 4 B fp32 scale].
    """
    vals = np.empty((len(pages), IDX_DIM), dtype=np.uint8)
    scales = np.empty(len(pages), dtype=np.float32)
    for i in range(0, len(pages), 1 << 18):
        p, s = pages[i:i + (1 << 18)], slots[i:i + (1 << 18)]
        cols = s[:, None] * IDX_DIM + np.arange(IDX_DIM)
        vals[i:i + len(p)] = key_pool[p[:, None], cols]
        off = page_size * IDX_DIM + 4 * s
        raw = key_pool[p[:, None], off[:, None] + np.arange(4)]
        scales[i:i + len(p)] = f32_from_bytes(raw).reshape(-1)
    return vals, scales


def dequant_fp8_keys(key_pool, pages, slots, page_size) -> np.ndarray:
    """k_hat[s, d] = E4M3(k_s[d]) * scale_s, float64 [n, 128] ([SA]: FP8 key with its scale)."""
    vals, scales = read_fp8_keys(key_pool, pages, slots, page_size)
    return e4m3_decode(vals) * scales.astype(np.float64)[:, None]


def dequant_mxfp4_keys(key_pool, pages, slots, page_size) -> np.ndarray:
    """MXFP4 index key [MX4]: 128 E2M1 values, one E8M0 exponent per 32, float64 [n, 128].

    Page layout: [page_size x 64 B E2M1 pairs][page_size x 4 B E8M0].
    """
    n = len(pages)
    cols = slots[:, None] * 64 + np.arange(64)
    packed = key_pool[pages[:, None], cols]
    sc = key_pool[pages[:, None], page_size * 64 + 4 * slots[:, None] + np.arange(4)]
    v = e2m1_unpack(packed).reshape(n, 4, 32) * e8m0_decode(sc)[:, :, None]
    return v.reshape(n, IDX_DIM)


def dequant_fp8_latents(lat_pool, pages, slots, latent_scale) -> np.ndarray:
    """c_hat[s] = E4M3(c_s) * latent_scale, float64 [n, 576] (512 nope then 64 rope) [NEWS]."""
    cols = slots[:, None] * D_QK + np.arange(D_QK)
    return e4m3_decode(lat_pool[pages[:, None], cols]) * float(latent_scale)


def dequant_nvfp4_latents(lat_pool, pages, slots, latent_scale) -> np.ndarray:
    """NVFP4 latent [REC], 352 B: 512 E2M1 with one E4M3 scale per 16, then 64 E4M3 rope.

    Reading: no per-tensor global scale beyond ``latent_scale``.
    Row layout: [256 B E2M1 pairs][32 B E4M3 block scales][64 B E4M3 rope].
    """
    n = len(pages)
    cols = slots[:, None] * 352 + np.arange(352)
    row = lat_pool[pages[:, None], cols]
    nope = e2m1_unpack(row[:, :256]).reshape(n, 32, 16) * e4m3_decode(row[:, 256:288])[:, :, None]
    rope = e4m3_decode(row[:, 288:352])
    return np.concatenate([nope.reshape(n, D_NOPE), rope], axis=1) * float(latent_scale)


def dequant_keys(inp, b: int, L: int) -> np.ndarray:
    pages, slots = token_pages(inp.block_table[b], L, inp.page_size)
    if inp.key_fmt == "fp8":
        return dequant_fp8_keys(inp.key_pool, pages, slots, inp.page_size)
    return dequant_mxfp4_keys(inp.key_pool, pages, slots, inp.page_size)


def dequant_latents(inp, b: int, tokens: np.ndarray) -> np.ndarray:
    tokens = np.asarray(tokens, dtype=np.int64)
    pages = inp.block_table[b][tokens // inp.page_size].astype(np.int64)
    slots = tokens % inp.page_size
    if inp.lat_fmt == "fp8":
        return dequant_fp8_latents(inp.lat_pool, pages, slots, inp.latent_scale)
    return dequant_nvfp4_latents(inp.lat_pool, pages, slots, inp.latent_scale)


# ----------------------------------------------------------------------------
# indexer query quantisation [FUSE]
# ----------------------------------------------------------------------------

def quantize_index_query(q_idx: np.ndarray, w: np.ndarray):
    """FP8 indexer query with its scale folded into the head weights [FUSE].

    q_idx: float32 [32, 128] (bf16 values); w: float32 [32].
    Reading (the page says only "FP8 quantisation, folded into the head
    weights"): one scale per head, all in IEEE fp32 with round-to-nearest:
        amax_h = max_d |q[h, d]|
        inv_h  = 448 / amax_h           (1 when amax_h == 0)
        q8[h]  = E4M3_rne_satfinite(q[h] * inv_h)
        w'_h   = w_h * (amax_h / 448)
    Returns (E4M3 codes uint8 [32, 128], w' float32 [32]).
    """
    q = np.asarray(q_idx, dtype=np.float32)
    amax = np.abs(q).max(axis=1).astype(np.float32)
    f448 = np.float32(448.0)
    with np.errstate(divide="ignore"):
        inv = np.where(amax > 0, f448 / np.where(amax > 0, amax, np.float32(1)), np.float32(1)).astype(np.float32)
    codes = e4m3_encode_rne_satfinite((q * inv[:, None]).astype(np.float32))
    w_prime = (np.asarray(w, dtype=np.float32) * (amax / f448).astype(np.float32)).astype(np.float32)
    return codes, w_prime


def indexer_scores_from(qv: np.ndarray, w: np.ndarray, k_hat: np.ndarray) -> np.ndarray:
    """score[s] = sum_h w_h * max(0, q_h . k_hat_s), float64 [n] ([SA]; [MX4]: weighted cross-head sum).

    qv float64 [32, 128], w float64 [32], k_hat float64 [n, 128].
    """
    dots = k_hat @ qv.T
    return np.maximum(dots, 0.0) @ np.asarray(w, dtype=np.float64)


def indexer_scores(inp, b: int, t: int, exact_query: bool = False) -> np.ndarray:
    """fp32 scores of query (b, t) over its L_{b,t} visible tokens.

    Default: the FP8 query recipe of ``quantize_index_query``. With
    ``exact_query`` the bf16 query and raw weights are used unquantised.
    The fp64 sum is rounded once to fp32, the precision the selection works in.
    """
    L = visible_len(inp.ctx[b], inp.n_q, t)
    qf = bf16_decode(inp.q_idx[b, t]).astype(np.float32)
    if exact_query:
        qv, wv = qf.astype(np.float64), inp.w[b, t].astype(np.float64)
    else:
        codes, wp = quantize_index_query(qf, inp.w[b, t])
        qv, wv = e4m3_decode(codes), wp.astype(np.float64)
    out = np.empty(L, dtype=np.float32)
    step = 1 << 18
    bt = inp.block_table[b]
    for s0 in range(0, L, step):
        s1 = min(L, s0 + step)
        tok = np.arange(s0, s1, dtype=np.int64)
        pages, slots = bt[tok // inp.page_size].astype(np.int64), tok % inp.page_size
        if inp.key_fmt == "fp8":
            k_hat = dequant_fp8_keys(inp.key_pool, pages, slots, inp.page_size)
        else:
            k_hat = dequant_mxfp4_keys(inp.key_pool, pages, slots, inp.page_size)
        out[s0:s1] = indexer_scores_from(qv, wv, k_hat).astype(np.float32)
    return out


# ----------------------------------------------------------------------------
# exact top-k [SA], [NEWS]
# ----------------------------------------------------------------------------

def topk_select(scores: np.ndarray, k: int = 2048) -> np.ndarray:
    """Exact top-k of fp32 scores; int32 [k], ascending token index, -1 padded.

    Order: higher score first, and among equal scores the lower token index
    (the pages ask for "consistent tie handling" in the merge; this library
    fixes the lower index). -0 and +0 compare equal. With L <= k every token is
    kept. NaN scores are invalid input.
    """
    s = np.asarray(scores, dtype=np.float32)
    assert not np.isnan(s).any(), "NaN scores are invalid input"
    L = s.shape[0]
    idx = np.arange(L)
    order = np.lexsort((idx, -s.astype(np.float64)))
    keep = np.sort(order[:min(k, L)])
    out = np.full(k, -1, dtype=np.int32)
    out[:len(keep)] = keep
    return out


def kth_score(scores: np.ndarray, k: int = 2048) -> float:
    """The k-th largest score (the threshold tau), or -inf when L < k."""
    s = np.sort(np.asarray(scores, dtype=np.float64))[::-1]
    return float(s[k - 1]) if len(s) >= k else -math.inf


def physical_rows(block_table_row: np.ndarray, idx: np.ndarray, page_size: int) -> np.ndarray:
    """Physical cache row (page * page_size + slot) of each selected token, -1 kept."""
    idx = np.asarray(idx, dtype=np.int64)
    out = np.full(idx.shape, -1, dtype=np.int64)
    v = idx >= 0
    out[v] = block_table_row[idx[v] // page_size].astype(np.int64) * page_size + idx[v] % page_size
    return out.astype(np.int32)


# ----------------------------------------------------------------------------
# exact attention over the selected latents [SA]
# ----------------------------------------------------------------------------

def mla_attention(q: np.ndarray, c_hat: np.ndarray, softmax_scale: float):
    """Absorbed MLA for one query token over rows ``c_hat``.

    q float64 [96, 576]; c_hat float64 [n, 576], one latent shared by all heads.
    logit[h, s] = scale * q_h . c_hat_s; p = softmax over s;
    out[h] = sum_s p[h, s] * c_hat_s[:512]; lse[h] = ln sum_s exp(logit[h, s]).
    Reading: the value is the 512-wide nope part of the latent (the value
    projection runs after attention in the fused path [FUSE]); natural log.
    With n == 0: out = 0, lse = -inf.
    """
    if c_hat.shape[0] == 0:
        return np.zeros((q.shape[0], D_NOPE)), np.full(q.shape[0], -np.inf)
    logits = float(softmax_scale) * (q @ c_hat.T)
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    l = p.sum(axis=1, keepdims=True)
    out = (p @ c_hat[:, :D_NOPE]) / l
    lse = (m + np.log(l))[:, 0]
    return out, lse


def sparse_mla(inp, b: int, t: int, idx: np.ndarray):
    """Attention of query (b, t) over the tokens listed in ``idx`` (-1 entries skipped)."""
    idx = np.asarray(idx)
    sel = idx[idx >= 0].astype(np.int64)
    assert (sel < visible_len(inp.ctx[b], inp.n_q, t)).all(), "index past the visible context"
    c_hat = dequant_latents(inp, b, sel)
    q = bf16_decode(inp.q[b, t])
    return mla_attention(q, c_hat, inp.softmax_scale)


def dense_mla(inp, b: int, t: int):
    """Attention over every visible token (the dense-MLA baseline)."""
    L = visible_len(inp.ctx[b], inp.n_q, t)
    return sparse_mla(inp, b, t, np.arange(L))


def lse_combine(outs: np.ndarray, lses: np.ndarray):
    """Merge partial attention results over disjoint token sets [DCP].

    outs float64 [S, H, D], lses [S, H] -> (out [H, D], lse [H]):
    lse = ln sum_i exp(lse_i); out = sum_i exp(lse_i - lse) * out_i.
    Parts with lse_i = -inf (no tokens) contribute nothing.
    """
    lses = np.asarray(lses, dtype=np.float64)
    m = lses.max(axis=0)
    finite = np.isfinite(m)
    msafe = np.where(finite, m, 0.0)
    wsum = np.exp(lses - msafe).sum(axis=0)
    lse = np.where(finite, msafe + np.log(np.where(finite, wsum, 1.0)), -np.inf)
    wts = np.where(finite, np.exp(lses - np.where(finite, lse, 0.0)), 0.0)
    out = (wts[:, :, None] * np.asarray(outs, dtype=np.float64)).sum(axis=0)
    return out, lse


# ----------------------------------------------------------------------------
# the fused step
# ----------------------------------------------------------------------------

def decode(inp, exact_query: bool = False, requests=None):
    """Indexer -> exact top-k -> sparse MLA for every (b, t) (or the listed requests).

    Returns dict with per-(b, t) 'scores' (fp32 [L]), 'idx' (int32 [K]),
    'out' (float64 [96, 512]), 'lse' (float64 [96]).
    """
    res = {}
    bs = range(inp.batch) if requests is None else requests
    for b in bs:
        for t in range(inp.n_q):
            sc = indexer_scores(inp, b, t, exact_query=exact_query)
            idx = topk_select(sc, inp.topk)
            out, lse = sparse_mla(inp, b, t, idx)
            res[(b, t)] = dict(scores=sc, idx=idx, out=out, lse=lse)
    return res


# ----------------------------------------------------------------------------
# byte model [NEWS], [SA], [KVF]
# ----------------------------------------------------------------------------

KEY_BYTES = {"fp8": 132, "mxfp4": 68}
LAT_BYTES = {"fp8": 576, "nvfp4": 352}
Q_OUT_BYTES = IDX_HEADS * IDX_DIM * 2 + IDX_HEADS * 4 + HEADS * D_QK * 2 + HEADS * D_NOPE * 2


def request_bytes(ctx_b: int, n_q: int, union_selected: int, key_fmt="fp8", lat_fmt="fp8") -> int:
    """Bytes one request's decode step must move: every index key once, each
    selected latent once, and the query/weights/output of its n_q query tokens."""
    return KEY_BYTES[key_fmt] * int(ctx_b) + LAT_BYTES[lat_fmt] * int(union_selected) + n_q * Q_OUT_BYTES


def dense_request_bytes(ctx_b: int, lat_fmt="fp8") -> int:
    """Latent bytes of dense MLA for one request and layer."""
    return LAT_BYTES[lat_fmt] * int(ctx_b)
