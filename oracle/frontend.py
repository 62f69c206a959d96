"""The fused indexer front end of a decode step, written out plainly in float64 --
TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "vLLM 为 Kimi K3.1 Pro 提供 Day-0 支持", section "低延迟解码：融合的 DSA
解码路径" [FUSE], which fuses into a single kernel the work ahead of the scorer:
normalising the query latent, projecting it onto the indexer heads, turning the
result into FP8 with its scale moved into the head weights, and producing the
new token's index key. The MXFP4 key format is the page's "量化：原生 MXFP4 索引器"
[MX4] in the OCP Microscaling layout (formats.py).

Readings (the page names the steps, not their arithmetic):
  * Query norm = RMS norm over the query latent c (width d_c):
        n = c / sqrt(mean(c^2) + eps) * gamma,
    rounded once to bf16, the model's activation type.
  * Indexer query projection: q = n @ W_q^T (W_q [32 * 128, d_c], a linear
    layer's [out, in] weight), rounded once to bf16; q[h] = q[128 h : 128 h + 128].
  * Quantisation: ``dsa.quantize_index_query`` on the bf16 q (one E4M3 scale per
    head, folded into w).
  * New token's index key: k = bf16(x @ W_k^T) (x the hidden state, width
    d_model; W_k [128, d_model]). The page names a norm only for the query, so
    the key has none. Row (b, t) is token ctx_b - n_q + t, whose slot of the
    paged cache receives the key.
  * FP8 key (132 B): per token amax = max |k|, inv = 448 / amax (1 when amax = 0),
    codes = E4M3_rne_satfinite(k * inv), scale = amax / 448, all fp32 with
    round-to-nearest: the recipe of the query. The key read back is
    E4M3(code) * scale.
  * MXFP4 key (68 B): per 32 values amax, e = floor(log2 amax) - 2 (2 is E2M1's
    largest exponent), clamped to [-127, 127] (e = 0 when amax = 0); codes =
    E2M1_rne_satfinite(v / 2^e) (ties to the even code, magnitudes past 6 become
    6, the sign kept, -0 included); E8M0 byte = e + 127.
  * bf16 rounding of a float64 value is one rounding to nearest even (8
    significant bits); values stay in bf16's normal range here.
"""
from __future__ import annotations

import numpy as np

from .dsa import IDX_DIM, IDX_HEADS, quantize_index_query
from .formats import E2M1, e4m3_encode_rne_satfinite


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> nearest bf16 value (ties to even), returned as float64."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                    # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0), e - 8)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) of values that are exactly bf16."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    assert (f.astype(np.float64) == np.asarray(x, dtype=np.float64)).all()
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def rms_norm_bf16(c: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """Query norm [FUSE]: bf16(c / sqrt(mean(c^2) + eps) * gamma) over the last axis."""
    c = np.asarray(c, dtype=np.float64)
    ms = (c * c).mean(axis=-1, keepdims=True)
    return round_bf16(c / np.sqrt(ms + float(eps)) * np.asarray(gamma, dtype=np.float64))


def project_bf16(v: np.ndarray, weight: np.ndarray) -> np.ndarray:
    """A bias-free linear layer in float64, rounded once to bf16: bf16(v @ weight^T)."""
    return round_bf16(np.asarray(v, dtype=np.float64) @ np.asarray(weight, dtype=np.float64).T)


def frontend_query(c_q, gamma, w_q, w, eps):
    """Rows of c_q [rows, d_c] -> (q8 uint8 [rows, 32, 128], w' fp32 [rows, 32], q float64 [rows, 32, 128])."""
    n = rms_norm_bf16(c_q, gamma, eps)
    q = project_bf16(n, w_q).reshape(-1, IDX_HEADS, IDX_DIM)
    q8 = np.empty(q.shape, dtype=np.uint8)
    wp = np.empty((q.shape[0], IDX_HEADS), dtype=np.float32)
    for r in range(q.shape[0]):
        q8[r], wp[r] = quantize_index_query(q[r].astype(np.float32), np.asarray(w[r], dtype=np.float32))
    return q8, wp, q


def new_index_key(x, w_k) -> np.ndarray:
    """The new tokens' index keys, bf16 values as float64 [rows, 128]."""
    return project_bf16(x, w_k)


def quantize_key_fp8(k: np.ndarray):
    """One token's FP8 key: (E4M3 codes uint8 [128], fp32 scale)."""
    k32 = np.asarray(k, dtype=np.float32)
    amax = np.float32(np.abs(k32).max())
    inv = np.float32(448.0) / amax if amax > 0 else np.float32(1.0)
    codes = e4m3_encode_rne_satfinite((k32 * inv).astype(np.float32))
    return codes, np.float32(amax / np.float32(448.0))


def e2m1_encode_rne_satfinite(v: np.ndarray) -> np.ndarray:
    """Values -> E2M1 codes (sign in bit 3), nearest with ties to the even code, saturating at 6."""
    v = np.asarray(v, dtype=np.float64)
    mags = E2M1[:8]                       # 0, 0.5, 1, 1.5, 2, 3, 4, 6
    a = np.minimum(np.abs(v), 6.0)
    d = np.abs(a[..., None] - mags)       # distance to every magnitude
    best = d.min(axis=-1, keepdims=True)
    cand = d == best                      # one code, or two at a tie
    even = cand & (np.arange(8) % 2 == 0)
    code = np.where(even.any(axis=-1), even.argmax(axis=-1), cand.argmax(axis=-1))
    return (code | np.where(np.signbit(v), 8, 0)).astype(np.uint8)


def quantize_key_mxfp4(k: np.ndarray):
    """One token's MXFP4 key: (64 bytes of E2M1 pairs, element 2i in the low nibble; 4 E8M0 bytes)."""
    v = np.asarray(k, dtype=np.float64).reshape(4, 32)
    codes = np.empty((4, 32), dtype=np.uint8)
    e8 = np.empty(4, dtype=np.uint8)
    for blk in range(4):
        amax = np.abs(v[blk]).max()
        if amax == 0:
            e = 0
        else:
            _, ex = np.frexp(amax)            # amax = m * 2^ex, 0.5 <= m < 1
            e = int(np.clip(ex - 1 - 2, -127, 127))
        codes[blk] = e2m1_encode_rne_satfinite(v[blk] / 2.0 ** e)
        e8[blk] = e + 127
    c = codes.reshape(-1)
    return (c[0::2] | (c[1::2] << 4)).astype(np.uint8), e8


def new_token_position(ctx_b: int, n_q: int, t: int) -> int:
    return int(ctx_b) - int(n_q) + int(t)


def write_key(key_pool: np.ndarray, page: int, slot: int, k: np.ndarray, fmt: str, page_size: int = 64) -> None:
    """Quantise one key and store it in slot `slot` of page `page` (in place).

    Page layouts (this library's; the page fixes only the bytes per token):
      fp8   [page_size x 128 B E4M3][page_size x 4 B fp32 scale]
      mxfp4 [page_size x 64 B E2M1 pairs][page_size x 4 B E8M0]
    """
    if fmt == "fp8":
        codes, scale = quantize_key_fp8(k)
        key_pool[page, slot * IDX_DIM:(slot + 1) * IDX_DIM] = codes
        off = page_size * IDX_DIM + 4 * slot
        key_pool[page, off:off + 4] = np.frombuffer(np.float32(scale).tobytes(), dtype=np.uint8)
    else:
        packed, e8 = quantize_key_mxfp4(k)
        key_pool[page, slot * 64:(slot + 1) * 64] = packed
        off = page_size * 64 + 4 * slot
        key_pool[page, off:off + 4] = e8


def frontend(c_q, gamma, w_q, w, eps, x, w_k, key_pool, block_table, ctx, n_q, fmt, page_size=64):
    """The whole front end of one step. Returns (q8, w', keys) and writes every
    new key into a copy of key_pool, returned last."""
    q8, wp, _ = frontend_query(c_q, gamma, w_q, w, eps)
    keys = new_index_key(x, w_k)
    pool = np.array(key_pool, copy=True)
    for b in range(len(ctx)):
        for t in range(n_q):
            pos = new_token_position(ctx[b], n_q, t)
            page = int(block_table[b][pos // page_size])
            write_key(pool, page, pos % page_size, keys[b * n_q + t], fmt, page_size)
    return q8, wp, keys, pool
