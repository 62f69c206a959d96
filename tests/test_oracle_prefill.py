"""Pins of the token-sharded prefill split: a partition of the rows, and equal
causal work per rank (the point of pairing slice r with slice 2W - 1 - r)."""
import numpy as np

from oracle import prefill as P
from oracle.dsa import visible_len


def test_ranks_partition_the_rows():
    for world in (1, 2, 4, 8):
        n_q = 16 * world
        rows = np.concatenate([P.rank_rows(n_q, world, r) for r in range(world)])
        assert np.array_equal(np.sort(rows), np.arange(n_q))
    assert np.array_equal(P.rank_rows(64, 1, 0), np.arange(64))
    # the page's case: 8 GPUs, 16 slices, GPU 0 takes slices 0 and 15, GPU 7 slices 7 and 8
    assert np.array_equal(P.rank_rows(16, 8, 0), [0, 15])
    assert np.array_equal(P.rank_rows(16, 8, 7), [7, 8])


def test_paired_slices_balance_causal_work_and_contiguous_ones_do_not():
    ctx, n_q, world = 2048 + 300, 2048, 8
    work = [P.causal_work(ctx, n_q, P.rank_rows(n_q, world, r)) for r in range(world)]
    assert len(set(work)) == 1                     # exactly equal
    total = sum(visible_len(ctx, n_q, t) for t in range(n_q))
    assert work[0] * world == total
    # cutting into W contiguous blocks instead leaves the last rank with the most work
    blocks = [P.causal_work(ctx, n_q, range(r * n_q // world, (r + 1) * n_q // world)) for r in range(world)]
    assert blocks[-1] > blocks[0] * 2
    # closed form: visible lengths ctx - n_q + t + 1 over rank r's rows
    ss = n_q // (2 * world)
    r = 3
    rows = list(range(r * ss, (r + 1) * ss)) + list(range((2 * world - 1 - r) * ss, (2 * world - r) * ss))
    assert work[r] == sum(ctx - n_q + t + 1 for t in rows) == ss * (2 * (ctx - n_q + 1) + n_q - 1)


def test_bench_counts_the_same_rows_as_the_split():
    import bench

    for world in (1, 2, 8):
        n_q = 64 * world
        for rank in range(world):
            assert bench._rank_rows(n_q, world, rank) == P.rank_rows(n_q, world, rank).tolist()
