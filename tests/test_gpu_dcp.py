"""GPU parity of the decode-context-parallel exact top-k merge (W token shards
emulated on one GPU) against the oracle's merge (one or two exchanges): selected tokens
bit-exact, and the re-sent shard mask and the words exchanged equal.

Source: "vLLM 为 Kimi K3.1 Pro 提供 Day-0 支持", section "长上下文：带稀疏 indexer
的 decode 上下文并行", "流量减少 10× 的精确 top-k 合并".
"""
import numpy as np
import pytest

import dsa_sparse_mla_paged_gb300 as dsa
from oracle import dcp as D
from oracle import dsa as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need(lib, cuda_ok):
    yield


def _merge(ctx, mat, W, topk=2048, n_q=1, stats=True):
    """dsa_dcp_topk_merge on `mat` (fp32 [len(ctx) * n_q, >= max ctx])."""
    import torch

    rows = len(ctx) * n_q
    cap = max(ctx)
    pages = (cap + 63) // 64
    p = dsa.make_params(batch=len(ctx), n_q=n_q, max_pages_per_req=pages, num_pages=1, key_page_stride=64 * 132,
                        lat_page_stride=64 * 576, topk=topk, page_size=64)
    ws = torch.zeros(dsa.workspace_size(p), dtype=torch.uint8, device="cuda")
    stride = (cap + 3) // 4 * 4
    sc = torch.full((rows, stride), float("nan"), dtype=torch.float32, device="cuda")
    sc[:, :mat.shape[1]] = torch.from_numpy(np.ascontiguousarray(mat[:, :stride]))
    ctx_t = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    idx = torch.full((rows, topk), -7, dtype=torch.int32, device="cuda")
    st = torch.full((rows, 2), -7, dtype=torch.int32, device="cuda") if stats else None
    dsa.dcp_topk_merge(p, sc, stride, ctx_t, W, idx, st, ws)
    torch.cuda.synchronize()
    assert dsa.get_device_error(ws) == 0
    return idx.cpu().numpy(), (st.cpu().numpy() if stats else None)


def _check_rows(ctx, mat, W, topk=2048, n_q=1):
    idx, st = _merge(ctx, mat, W, topk, n_q)
    for b, c in enumerate(ctx):
        for t in range(n_q):
            r = b * n_q + t
            L = O.visible_len(c, n_q, t)
            res = D.merge(mat[r, :L], W, topk)
            assert np.array_equal(idx[r], res["idx"]), (W, r)
            mask = sum(1 << s for s in res["resent"])
            assert (st[r, 0], st[r, 1]) == (mask, res["words"]), (W, r, st[r], mask, res["words"])
    return idx, st


def _patterns(L, seed):
    rng = np.random.default_rng(seed)
    yield "normal", rng.standard_normal(L).astype(np.float32)
    yield "constant", np.full(L, 0.75, np.float32)
    yield "few_levels", (rng.integers(0, 9, L) * 0.5 - 2.0).astype(np.float32)
    z = rng.standard_normal(L).astype(np.float32)
    z[rng.random(L) < 0.3] = 0.0
    z[rng.random(L) < 0.3] = -0.0
    yield "signed_zeros", z
    big = rng.standard_normal(L).astype(np.float32)
    big[rng.integers(0, L, 10)] = np.float32(3e38)
    big[rng.integers(0, L, 10)] = -np.float32(3e38)
    yield "extremes", big
    # fp32 scores that differ only below bf16 precision: ties after rounding
    yield "bf16_ties", (1.0 + rng.integers(0, 64, L).astype(np.float32) * 2.0 ** -12).astype(np.float32)


CTX = [70000, 5, 4097, 2048, 2049, 1, 3 * 2048 + 11]


@pytest.mark.parametrize("W", [1, 2, 3, 8, 16])
def test_merge_equals_oracle(W):
    L = max(CTX)
    for name, _ in _patterns(1, 0):
        mat = np.zeros((len(CTX), L), np.float32)
        for b, c in enumerate(CTX):
            mat[b, :c] = dict(_patterns(c, 31 * b + W))[name]
        _check_rows(CTX, mat, W)


@pytest.mark.parametrize("W,boost,topk", [(8, [2], 2048), (8, [1, 5], 2048), (16, list(range(10)), 2048),
                                          (16, [3], 100), (4, [0, 3], 1000)])
def test_merge_resends_when_shards_hold_the_top_k(W, boost, topk):
    L = 200000
    mat = np.random.default_rng(40 + W).standard_normal((2, L)).astype(np.float32)
    for r in boost:
        mat[0, r::W] += 10.0
    idx, st = _check_rows([L, L], mat, W, topk)
    want = sum(1 << r for r in boost)
    assert st[0, 0] & want == want  # (an unboosted shard may re-send as well, as the oracle says)
    assert st[1, 0] == 0
    assert set((idx[0][idx[0] >= 0] % W).tolist()) <= set(boost)


def test_merge_query_rows_and_small_k():
    rng = np.random.default_rng(50)
    ctx = [9000, 130, 40000]
    n_q = 3
    mat = rng.standard_normal((len(ctx) * n_q, max(ctx))).astype(np.float32)
    for k in (1, 16, 100, 2047):
        for W in (2, 7):
            _check_rows(ctx, mat, W, k, n_q)


def test_one_shard_equals_topk_on_bf16_scores():
    import torch

    rng = np.random.default_rng(51)
    ctx = [100000, 3000]
    mat = rng.standard_normal((2, max(ctx))).astype(np.float32)
    mat = (D.bf16_rne_bits(mat).astype(np.uint32) << 16).view(np.float32).reshape(mat.shape)
    idx, st = _merge(ctx, mat, 1)
    for b, c in enumerate(ctx):
        assert np.array_equal(idx[b], O.topk_select(mat[b, :c], 2048))
    assert st[0, 1] == 2048 and st[1, 1] == 2048


def test_merge_without_stats():
    mat = np.random.default_rng(52).standard_normal((1, 30000)).astype(np.float32)
    idx, _ = _merge([30000], mat, 8, stats=False)
    assert np.array_equal(idx[0], D.merge(mat[0], 8, 2048)["idx"])


@pytest.mark.slow
def test_merge_at_full_context():
    """Four rows of 1,048,576 tokens, eight shards: every row equals the oracle."""
    ctx = [1 << 20] * 4
    rng = np.random.default_rng(53)
    mat = rng.standard_normal((4, 1 << 20)).astype(np.float32)
    mat[3, 6::8] += 4.0  # shard 6 holds most of row 3's top tokens
    idx, st = _check_rows(ctx, mat, 8)
    assert st[3, 0] == 1 << 6
    assert all(st[r, 1] == 8 * 384 for r in range(3))


# ----------------------------------------------------------------------------- cross-shard combine

def test_lse_combine_equals_oracle():
    import torch

    rng = np.random.default_rng(60)
    B, parts = 3, 5
    p = dsa.make_params(batch=B, n_q=1, max_pages_per_req=4, num_pages=1, key_page_stride=64 * 132,
                        lat_page_stride=64 * 576)
    po = rng.standard_normal((parts, B, 96, 512)).astype(np.float32)
    pl = (rng.standard_normal((parts, B, 96)) * 3 + 8).astype(np.float32)
    pl[1, 0, :] = -np.inf                      # a shard with no winners for row 0
    pl[:, 2, 7] = -np.inf                      # every shard empty for row 2, head 7
    pl[3, 1, 5] = pl[0, 1, 5] + 60.0           # one shard dominates
    po_bf = torch.from_numpy(po).to(torch.bfloat16)
    po_np = po_bf.float().numpy().astype(np.float64)
    dev_o = po_bf.cuda()
    dev_l = torch.from_numpy(pl).cuda()
    out = torch.full((B, 96, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, 96), 7.0, dtype=torch.float32, device="cuda")
    dsa.lse_combine(p, parts, dev_o, dev_l, out, lse)
    torch.cuda.synchronize()
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    for b in range(B):
        ro, rl = O.lse_combine(po_np[:, b], pl[:, b].astype(np.float64))
        # fp32 weights and sums, one bf16 rounding of the result
        assert (np.abs(o[b] - ro) <= 2.0 ** -8 * np.abs(ro) + 1e-5).all(), b
        fin = np.isfinite(rl)
        assert (np.isfinite(l[b]) == fin).all()
        assert np.abs(l[b][fin] - rl[fin]).max() <= 1e-5 * np.abs(rl[fin]).max()
    assert (o[2, 7] == 0).all() and np.isneginf(l[2, 7])


@pytest.mark.parametrize("W", [2, 4, 8])
def test_dcp_attention_equals_attention_over_the_merged_set(W):
    """Indexer -> DCP merge -> every shard attends over its own winners -> LSE
    combine: within the attention bars of the oracle's attention over the merged
    set."""
    import torch

    import gen
    from dsa_testlib import Dev, bf16_to_np, check_attention

    inp = gen.make_inputs(3, 1, [20000, 3000, 1500], seed=61 + W, bt_mode="permuted", holes=True)
    d = Dev(inp)
    sc = d.scores()
    idx = torch.full((3, 2048), -7, dtype=torch.int32, device="cuda")
    dsa.dcp_topk_merge(d.p, sc, sc.shape[1], d.ctx, W, idx, None, d.ws)
    outs, lses = [], []
    for r in range(W):
        own = torch.where((idx >= 0) & (idx % W == r), idx, torch.full_like(idx, -1))
        o, l = d.mla(own)
        outs.append(o)
        lses.append(l)
    out = torch.empty((3, 96, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((3, 96), dtype=torch.float32, device="cuda")
    dsa.lse_combine(d.p, W, torch.stack(outs), torch.stack(lses), out, lse)
    torch.cuda.synchronize()
    assert dsa.get_device_error(d.ws) == 0
    idx_np = idx.cpu().numpy()
    scores_np = sc.cpu().numpy()
    for b in range(3):
        L = inp.ctx[b]
        assert np.array_equal(idx_np[b], D.merge(scores_np[b, :L], W, 2048)["idx"])
        ro, rl = O.sparse_mla(inp, b, 0, idx_np[b])
        check_attention(bf16_to_np(out[b]), lse[b].cpu().numpy(), ro, rl)


@pytest.mark.parametrize("W", [2, 8])
def test_merge_against_the_bf16_top_k_with_ties_at_tau(W):
    """Against dsa_topk's rule on the bf16-rounded scores: the same tokens above
    the K-th bf16 value and as many at it (the choice among those follows the
    merge's (position, shard) order)."""
    rng = np.random.default_rng(70 + W)
    ctx = [30000, 12000]
    mat = (rng.integers(0, 24, (2, 30000)) * 0.0625).astype(np.float32)
    idx, _ = _check_rows(ctx, mat, W)
    for b, L in enumerate(ctx):
        bv = (D.bf16_rne_bits(mat[b, :L]).astype(np.uint32) << 16).view(np.float32)
        ref = O.topk_select(bv, 2048)
        tau = np.sort(bv)[::-1][2047]
        g = idx[b][idx[b] >= 0]
        assert set(g[bv[g] > tau]) == set(ref[bv[ref] > tau])
        assert (bv[g] == tau).sum() == (bv[ref] == tau).sum() and (bv[g] >= tau).all()
