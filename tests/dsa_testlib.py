"""Helpers shared by the tests: move generated inputs to the GPU and call libdsa."""
from __future__ import annotations

import numpy as np

import dsa_sparse_mla_paged_gb300 as dsa  # noqa: F401  (loaded before gen.device)
from gen.device import KEY_FMT, LAT_FMT, Dev, params_for  # noqa: F401

# acceptance bars
SCORE_RTOL = 1e-3          # indexer scores, relative
SCORE_FLOOR = 1e-6         # denominator floor, relative to the row's largest |score|
TIE_RTOL = 1e-5            # end-to-end selection: tokens this close to tau may differ
OUT_MAX_ABS = 2e-2         # attention output (bf16)
OUT_MEAN_ABS = 2e-3
LSE_ABS = 1e-3             # log-sum-exp (fp32 arithmetic on logits of size ~10)
# An fp32 evaluation of score(t, s) adds ~160 products (128 per head dot
# product, 32 heads); its error is relative to the sum of their magnitudes, not
# to the score, which can cancel to near zero (signed head weights, or a dot
# product whose terms cancel). Scores are therefore also measured against
# COND_FRAC times that magnitude sum (16 fp32 ulps of it at SCORE_RTOL).
COND_FRAC = 2.0 ** -10


def rows_scores_oracle(inp, rows=None):
    from oracle import dsa as O

    out = {}
    for b in range(inp.batch):
        for t in range(inp.n_q):
            r = b * inp.n_q + t
            if rows is None or r in rows:
                out[r] = O.indexer_scores(inp, b, t)
    return out


def score_error_scale(inp, b: int, t: int) -> np.ndarray:
    """Per token: sum_h |w'_h| * [q_h . k_s > 0] * sum_d |q_hd * k_sd|, the magnitude
    of the terms an fp32 evaluation of score(t, s) adds up (FP8 query recipe)."""
    from oracle import dsa as O
    from oracle.formats import bf16_decode, e4m3_decode

    L = O.visible_len(inp.ctx[b], inp.n_q, t)
    codes, wp = O.quantize_index_query(bf16_decode(inp.q_idx[b, t]).astype(np.float32), inp.w[b, t])
    qv, wa = e4m3_decode(codes), np.abs(wp.astype(np.float64))
    out = np.empty(L)
    for s0 in range(0, L, 1 << 17):
        s1 = min(L, s0 + (1 << 17))
        k = _keys_range(inp, b, s0, s1)
        d = k @ qv.T
        out[s0:s1] = np.where(d > 0, np.abs(k) @ np.abs(qv).T, 0.0) @ wa
    return out


def _keys_range(inp, b, s0, s1):
    from oracle import dsa as O

    tok = np.arange(s0, s1, dtype=np.int64)
    pages = inp.block_table[b][tok // inp.page_size].astype(np.int64)
    slots = tok % inp.page_size
    if inp.key_fmt == "fp8":
        return O.dequant_fp8_keys(inp.key_pool, pages, slots, inp.page_size)
    return O.dequant_mxfp4_keys(inp.key_pool, pages, slots, inp.page_size)


def rows_error_scale(inp, rows=None):
    return {b * inp.n_q + t: score_error_scale(inp, b, t) for b in range(inp.batch) for t in range(inp.n_q)
            if rows is None or b * inp.n_q + t in rows}


def check_scores(got: np.ndarray, ref: np.ndarray, errscale: np.ndarray | None = None):
    """Relative error with denominator max(|ref|, 1e-6 * max |ref|, COND_FRAC * errscale)."""
    ref64 = ref.astype(np.float64)
    den = np.maximum(np.abs(ref64), SCORE_FLOOR * max(np.abs(ref64).max(), 1e-30))
    if errscale is not None:
        den = np.maximum(den, COND_FRAC * errscale)
    rel = np.abs(got.astype(np.float64) - ref64) / den
    assert np.isfinite(got).all(), "non-finite GPU score"
    assert rel.max() <= SCORE_RTOL, f"max rel score error {rel.max():.3e} at {int(rel.argmax())}"
    return float(rel.max())


def selection_errscale(inp, es):
    """The error scale to widen the selection window with, or None.

    With non-negative head weights every term of score(t, s) over the heads is
    >= 0, so the score near tau carries no cancellation across heads and the
    strict window TIE_RTOL * |tau| applies unchanged. Only signed head weights
    (which can cancel a score towards zero while fp32 rounding still scales with
    the terms) take the wider window."""
    return es if np.any(np.asarray(inp.w) < 0) else None


# differing tokens that needed the wider (signed-weight) window, for reporting
WIDE_WINDOW_USES = []


def check_selection(got_idx: np.ndarray, ref_idx: np.ndarray, ref_scores: np.ndarray, k: int,
                    errscale: np.ndarray | None = None):
    """Equal sets except tokens whose oracle score is within TIE_RTOL*|tau| of tau;
    both ascending, -1 padded. Given errscale (signed head weights only, see
    selection_errscale), the window is widened to the score bar of check_scores
    for that token and the rank-k token."""
    from oracle import dsa as O

    for arr in (got_idx, ref_idx):
        v = arr[arr >= 0]
        assert (np.diff(v) > 0).all(), "not strictly ascending"
        assert (arr[len(v):] == -1).all(), "padding not -1"
    g, r = set(got_idx[got_idx >= 0].tolist()), set(ref_idx[ref_idx >= 0].tolist())
    assert len(g) == len(r)
    if g == r:
        return 0
    tau = O.kth_score(ref_scores, k)
    diff = np.array(sorted(g ^ r))
    dev = np.abs(ref_scores[diff].astype(np.float64) - tau)
    strict = np.full(len(diff), TIE_RTOL * abs(tau))
    win = strict
    if errscale is not None:
        order = np.lexsort((np.arange(len(ref_scores)), -ref_scores.astype(np.float64)))
        e_tau = errscale[order[k - 1]]
        win = np.maximum(strict, SCORE_RTOL * COND_FRAC * (errscale[diff] + e_tau))
        WIDE_WINDOW_USES.append(int((dev > strict).sum()))
    assert (dev <= win).all(), f"selection differs beyond near-ties: {diff[dev > win][:10]}"
    return len(diff)


def check_attention(out: np.ndarray, lse: np.ndarray, ref_out: np.ndarray, ref_lse: np.ndarray):
    err = np.abs(out.astype(np.float64) - ref_out)
    assert err.max() <= OUT_MAX_ABS, f"max abs {err.max():.3e}"
    assert err.mean() <= OUT_MEAN_ABS, f"mean abs {err.mean():.3e}"
    fin = np.isfinite(ref_lse)
    assert (np.isfinite(lse) == fin).all()
    if fin.any():
        assert np.abs(lse[fin] - ref_lse[fin]).max() <= LSE_ABS
    return float(err.max()), float(err.mean())


def bf16_to_np(t):
    import torch

    return t.float().cpu().numpy()
