"""Decode context parallelism: the exact top-k merge across W shards -- TEST INFRASTRUCTURE ONLY.

Source: "vLLM 为 Kimi K3.1 Pro 提供 Day-0 支持", section "长上下文：带稀疏 indexer 的
decode 上下文并行", subsection "流量减少 10× 的精确 top-k 合并".

The method, restated: a request's cache is divided by token over W GPUs
(GPU r owns the tokens s with s mod W == r), so each GPU can rank only its own
tokens and the global top-2048 has to be assembled across them. The exchange
is kept small: a GPU contributes a fixed number of its best tokens (1.5 * 2048
/ W), each as one 32-bit word holding its BF16 score, and every GPU runs the
same radix selection over all contributions. Exactness is restored by a check
after that selection: a GPU whose every contribution won may own further
winners, and it then contributes its complete local top-k for that row.

Readings (the page gives the steps, not the bits):
  * BF16 score: round-to-nearest-even of the fp32 score. Its order key is the
    16-bit order-preserving key of the bf16 bits (-0 == +0), as the fp32 top-k
    uses a 32-bit one.
  * A shard orders its tokens by (bf16 key desc, token asc); j is a token's
    position in that order.
  * The 32-bit pack: key16 << 16 | (4095 - j) << 4 | (15 - r), so a larger pack
    is a better candidate; the low half names the candidate by its position in
    the sender's list (the sender keeps the position -> token map) instead of a
    token id, which would not fit. W <= 16 and positions < 4096.
  * The global order is the pack order: bf16 key desc, then position asc, then
    shard asc. The first exchange sends m = ceil(1.5 K / W) candidates per shard (all a
    shard holds when it holds fewer), but never more than K: a shard's tokens
    past its first K cannot be in the top K, and m > K only when W = 1.
  * Re-send test: shard r sent m candidates, holds more than m tokens among its
    first K, and all m are among that exchange's top K; then it sends its first K
    instead (all it holds when fewer) and the selection runs again. (A shard
    that already sent its first K cannot hold more winners, so m >= K never
    re-sends.)
  * Exactness: the merged K tokens are the top K of *all* tokens under the same
    order (``ideal_topk``). They may differ from the fp32 top-k where bf16
    rounding ties or reorders scores (the page's BF16 exchange).
"""
from __future__ import annotations

import math

import numpy as np


def bf16_rne_bits(scores: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns of fp32 scores, rounded to nearest even."""
    u = np.ascontiguousarray(scores, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_order_key(bits: np.ndarray) -> np.ndarray:
    """16-bit order-preserving key of bf16 bit patterns (larger value -> larger key, -0 == +0)."""
    b = np.asarray(bits, dtype=np.uint32)
    b = np.where(b == 0x8000, 0, b)
    return np.where(b & 0x8000, (~b) & 0xFFFF, b | 0x8000).astype(np.uint32)


def shard_list(scores: np.ndarray, W: int, r: int):
    """Tokens of shard r in the shard's order (bf16 key desc, token asc) and their keys."""
    s = np.asarray(scores, dtype=np.float32)
    assert not np.isnan(s).any(), "NaN scores are invalid input"
    tok = np.arange(r, s.shape[0], W, dtype=np.int64)
    key = bf16_order_key(bf16_rne_bits(s[tok]))
    order = np.lexsort((tok, -key.astype(np.int64)))
    return tok[order], key[order]


def pack(key16: np.ndarray, j: np.ndarray, r: int) -> np.ndarray:
    """The 32-bit candidate word."""
    assert r < 16 and (np.asarray(j) < 4096).all()
    return (np.asarray(key16, np.uint64) << 16 | (4095 - np.asarray(j, np.uint64)) << 4 | (15 - r)).astype(np.uint32)


def _select(words: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest (distinct) words."""
    return np.argsort(-words.astype(np.int64), kind="stable")[:k]


def merge(scores: np.ndarray, W: int, k: int = 2048) -> dict:
    """The exact merge in one or two exchanges. Returns
    idx      int32 [k]: the selected tokens, ascending, -1 padded
    resent   shards that re-sent their first k
    words    32-bit words exchanged in all (each shard's sent words once per exchange it sends in)
    """
    assert 1 <= W <= 16 and k <= 4096
    m = math.ceil(1.5 * k / W)
    lists = [shard_list(scores, W, r) for r in range(W)]

    def exchange(counts):
        words, toks, owner = [], [], []
        for r, (tok, key) in enumerate(lists):
            n = min(counts[r], len(tok))
            words.append(pack(key[:n], np.arange(n), r))
            toks.append(tok[:n])
            owner.append(np.full(n, r))
        words, toks, owner = np.concatenate(words), np.concatenate(toks), np.concatenate(owner)
        sel = _select(words, k)
        return toks[sel], owner[sel]

    counts = [min(m, k)] * W
    sent = sum(min(m, k, len(t)) for t, _ in lists)
    tok_sel, own_sel = exchange(counts)
    resent = [r for r in range(W)
              if min(k, len(lists[r][0])) > m and int((own_sel == r).sum()) == m]
    if resent:
        for r in resent:
            counts[r] = k
            sent += min(k, len(lists[r][0]))
        tok_sel, _ = exchange(counts)
    out = np.full(k, -1, dtype=np.int32)
    keep = np.sort(tok_sel)
    out[:len(keep)] = keep
    return {"idx": out, "resent": resent, "words": sent, "m": m}


def ideal_topk(scores: np.ndarray, W: int, k: int = 2048) -> np.ndarray:
    """The top k of all tokens under the merge's order (every shard sending
    everything; a shard's tokens past its first k can never be among them)."""
    words, toks = [], []
    for r in range(W):
        tok, key = shard_list(scores, W, r)
        tok, key = tok[:k], key[:k]
        words.append(pack(key, np.arange(len(tok)), r))
        toks.append(tok)
    words, toks = np.concatenate(words), np.concatenate(toks)
    keep = np.sort(toks[_select(words, k)])
    out = np.full(k, -1, dtype=np.int32)
    out[:len(keep)] = keep
    return out
