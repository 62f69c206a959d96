"""GPU parity of the prefill-shaped indexer: many query rows per request, the
scorer taking them 8 at a time (each group with its own causal context), and
token sharding (rank r of W scores slices r and 2W - 1 - r). Bars as the decode
indexer's: scores within the score tolerance of the oracle; a sharded call
equals the unsharded one bit for bit on its rows and writes no other row."""
import numpy as np
import pytest

import dsa_sparse_mla_paged_gb300 as dsa
import gen
from oracle import dsa as O
from oracle import prefill as P

from dsa_testlib import (Dev, bf16_to_np, check_attention, check_scores, check_selection, rows_error_scale,
                         selection_errscale,
                         rows_scores_oracle)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need(lib, cuda_ok):
    yield


@pytest.mark.parametrize("b,nq,ctx,signed", [(2, 40, [3000, 200], False), (1, 37, [5000], True),
                                             (3, 9, [9, 700, 4100], False)])
def test_prefill_scores_match_oracle(b, nq, ctx, signed):
    inp = gen.make_inputs(b, nq, ctx, seed=80 + nq, bt_mode="permuted", signed_w=signed)
    d = Dev(inp)
    sc = d.scores().cpu().numpy()
    assert dsa.get_device_error(d.ws) == 0
    ref = rows_scores_oracle(inp)
    es = rows_error_scale(inp)
    for r, rs in ref.items():
        check_scores(sc[r, :len(rs)], rs, es[r])
        assert np.isnan(sc[r, len(rs):d.cap]).all()


@pytest.mark.parametrize("key_fmt", ["fp8", "mxfp4"])
def test_sharded_prefill_equals_unsharded_on_its_rows(key_fmt):
    import torch

    nq, world = 64, 4
    inp = gen.make_inputs(2, nq, [3000, 900], seed=84, bt_mode="permuted", key_fmt=key_fmt)
    d = Dev(inp)
    full = d.scores()
    stride = full.shape[1]
    seen = np.zeros(2 * nq, dtype=int)
    for rank in range(world):
        sc = torch.full_like(full, float("nan"))
        dsa.indexer_prefill_scores(d.p, world, rank, d.q_idx, d.w, d.key_pool, d.block_table, d.ctx, sc, stride,
                                   d.ws)
        torch.cuda.synchronize()
        mine = P.rank_rows(nq, world, rank)
        rows = np.concatenate([b * nq + mine for b in range(2)])
        other = np.setdiff1d(np.arange(2 * nq), rows)
        got = sc.cpu().numpy()
        assert np.array_equal(got[rows].view(np.uint32), full.cpu().numpy()[rows].view(np.uint32))
        assert np.isnan(got[other]).all()
        seen[rows] += 1
    assert (seen == 1).all()
    assert dsa.get_device_error(d.ws) == 0


def test_prefill_decode_end_to_end():
    """A 24-row prefill chunk through dsa_decode: indexer groups, top-k and
    attention for every row."""
    inp = gen.make_inputs(2, 24, [2100, 5000], seed=85, bt_mode="permuted")
    d = Dev(inp)
    out, lse, idx = d.decode()
    idx = idx.cpu().numpy()
    sc = d.scores().cpu().numpy()
    es = rows_error_scale(inp)
    res = O.decode(inp)
    for (b, t), r in res.items():
        row = b * inp.n_q + t
        check_scores(sc[row, :len(r["scores"])], r["scores"], es[row])
        check_selection(idx[row], r["idx"], r["scores"], inp.topk, selection_errscale(inp, es[row]))
    outs, lses = [], []
    for row in range(d.rows):
        o, l = O.sparse_mla(inp, row // inp.n_q, row % inp.n_q, idx[row])
        outs.append(o)
        lses.append(l)
    check_attention(bf16_to_np(out), lse.cpu().numpy(), np.stack(outs), np.stack(lses))


@pytest.mark.slow
def test_prefill_2k_on_150k_prefix_sampled_rows():
    """2,048 new tokens on a 150K-token cached prefix (the page's append case),
    one request; sampled rows against the oracle, every row's written length."""
    inp = gen.make_workload("b1_prefill2k_ctx150k")
    d = Dev(inp)
    sc = d.scores()
    assert dsa.get_device_error(d.ws) == 0
    es = rows_error_scale(inp, rows=[0, 7, 8, 1023, 2047])
    ref = rows_scores_oracle(inp, rows=[0, 7, 8, 1023, 2047])
    got = sc.cpu().numpy()
    for r, rs in ref.items():
        check_scores(got[r, :len(rs)], rs, es[r])
    for t in range(inp.n_q):
        L = O.visible_len(inp.ctx[0], inp.n_q, t)
        assert not np.isnan(got[t, L - 1]) and np.isnan(got[t, L:]).all()
