"""Token-sharded prefill of the indexer -- TEST INFRASTRUCTURE ONLY.

Source: "vLLM 为 Kimi K3.1 Pro 提供 Day-0 支持", section "预填充：按 token 而非按头分片注意力":
in a large prefill the GPUs divide the query tokens rather than the heads, each
scoring its tokens against the whole context; the division pairs slices so that
the causal work evens out (8 GPUs, 16 slices, GPU r with slices r and 15 - r).

Reading: with W ranks, the n_q query rows of a request are cut into 2W equal
slices of consecutive rows; rank r owns slices r and 2W - 1 - r. The scores of
a row are those of ``dsa.indexer_scores`` whichever rank computes them.
"""
from __future__ import annotations

import numpy as np

from .dsa import visible_len


def rank_rows(n_q: int, world: int, rank: int) -> np.ndarray:
    """Query rows (0 .. n_q - 1) of one request that rank `rank` of `world` scores."""
    assert world >= 1 and 0 <= rank < world and n_q % (2 * world) == 0
    ss = n_q // (2 * world)
    a = np.arange(rank * ss, (rank + 1) * ss)
    b = np.arange((2 * world - 1 - rank) * ss, (2 * world - rank) * ss)
    return np.concatenate([a, b])


def causal_work(ctx_b: int, n_q: int, rows) -> int:
    """Keys scored by the given rows: sum of their visible lengths."""
    return int(sum(visible_len(ctx_b, n_q, int(t)) for t in rows))
