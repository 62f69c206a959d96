"""GPU parity: every stage of libdsa against the CPU oracle on the same seeded inputs.

Bars: top-k bit-exact on identical fp32 scores; indexer scores within 1e-3
relative; end-to-end selection equal except tokens within 1e-5 relative of the
oracle's 2048th score; attention over the oracle's index set within max-abs
2e-2 and mean-abs 2e-3 (bf16 output).
"""
import functools

import numpy as np
import pytest

import gen
from oracle import dsa as O

from dsa_testlib import (Dev, bf16_to_np, check_attention, check_scores, check_selection,
                         rows_error_scale, rows_scores_oracle, score_error_scale, selection_errscale)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need(lib, cuda_ok):
    yield


SMALL = [
    # (batch, n_q, ctx, bt_mode, holes, key_pad, lat_pad, signed_w)
    (3, 1, [4096 + 37, 2049, 300], "permuted", True, 0, 0, False),
    (2, 3, [9000, 130], "permuted", False, 16, 32, True),
    (7, 1, [1, 63, 64, 65, 2047, 2048, 2049], "identity", False, 0, 0, False),
]


@functools.lru_cache(maxsize=None)
def _small(i):
    b, nq, ctx, mode, holes, kp, lp, sw = SMALL[i]
    return gen.make_inputs(b, nq, ctx, seed=100 + i, bt_mode=mode, holes=holes, key_page_pad=kp,
                           lat_page_pad=lp, signed_w=sw)


# ----------------------------------------------------------------------------- stage 1

@pytest.mark.parametrize("case", range(len(SMALL)))
def test_indexer_scores_small(case):
    inp = _small(case)
    d = Dev(inp)
    sc = d.scores().cpu().numpy()
    ref = rows_scores_oracle(inp)
    es = rows_error_scale(inp)
    for r, rs in ref.items():
        check_scores(sc[r, :len(rs)], rs, es[r])
        # entries past L are untouched
        assert np.isnan(sc[r, len(rs):d.cap]).all()


# ----------------------------------------------------------------------------- stage 2

def _score_patterns(L, seed):
    rng = np.random.default_rng(seed)
    yield "normal", rng.standard_normal(L).astype(np.float32)
    yield "constant", np.full(L, 0.75, np.float32)
    yield "few_levels", (rng.integers(0, 9, L) * 0.5 - 2.0).astype(np.float32)
    z = rng.standard_normal(L).astype(np.float32)
    z[rng.random(L) < 0.3] = 0.0
    z[rng.random(L) < 0.3] = -0.0
    yield "signed_zeros", z
    yield "neg_only", -np.abs(rng.standard_normal(L)).astype(np.float32) - 1.0
    big = rng.standard_normal(L).astype(np.float32)
    big[rng.integers(0, L, 10)] = np.float32(3e38)
    big[rng.integers(0, L, 10)] = -np.float32(3e38)
    yield "extremes", big


@pytest.mark.parametrize("ctx", [[1], [2047], [2048], [2049], [4096 * 3 + 5], [70000, 5, 4097, 2048 * 4]])
def test_topk_bit_exact_on_identical_scores(ctx):
    B = len(ctx)
    inp = gen.make_inputs(B, 1, ctx, seed=7)
    d = Dev(inp)
    L = max(ctx)
    for name, _ in _score_patterns(1, 0):
        mat = np.zeros((B, L), np.float32)
        for b in range(B):
            pats = dict(_score_patterns(ctx[b], 1000 * b + len(name)))
            mat[b, :ctx[b]] = pats[name]
        idx, _ = d.topk(mat)
        idx = idx.cpu().numpy()
        for b in range(B):
            ref = O.topk_select(mat[b, :ctx[b]], 2048)
            assert np.array_equal(idx[b], ref), (name, b)


def _planted_top_ties(L, seed):
    """N(0,1) scores with 300 copies of one high value straddling the K-th rank
    and 40 tokens one fp32 ulp either side of it."""
    rng = np.random.default_rng(seed)
    z = rng.standard_normal(L).astype(np.float32)
    v = np.sort(z)[::-1][2048 - 150]
    pos = rng.choice(L, 380, replace=False)
    z[pos[:300]] = v
    z[pos[300:340]] = np.nextafter(v, np.float32(np.inf))
    z[pos[340:]] = np.nextafter(v, np.float32(-np.inf))
    return z


@pytest.mark.parametrize("k", [2048, 100])
def test_topk_bit_exact_long_rows(k):
    """Rows long enough for the group-maxima bound (and one just below it), on
    score patterns that keep the candidate set small, straddle tau with ties, or
    overflow the candidate buffer (few levels: the whole-row select)."""
    ctx = [1 << 20, 262144 + 17, 100003, 73000]
    B = len(ctx)
    inp = gen.make_inputs(B, 1, ctx, seed=17, topk=k)
    d = Dev(inp)
    L = max(ctx)
    for name in ("normal", "top_ties", "few_levels", "extremes", "neg_only"):
        mat = np.zeros((B, L), np.float32)
        for b in range(B):
            if name == "top_ties":
                mat[b, :ctx[b]] = _planted_top_ties(ctx[b], 50 + b)
            else:
                mat[b, :ctx[b]] = dict(_score_patterns(ctx[b], 100 * b + len(name)))[name]
        idx, _ = d.topk(mat)
        idx = idx.cpu().numpy()
        for b in range(B):
            assert np.array_equal(idx[b], O.topk_select(mat[b, :ctx[b]], k)), (name, b)


@pytest.mark.parametrize("k", [1, 2, 16, 33])
def test_topk_small_k_many_rows(k):
    """Small K over rows of several chunks: the K-th key usually lies above
    the keys the first warp samples, in the top bin of the first histogram
    round (whose range can start past 2^32 in 32-bit arithmetic)."""
    rng = np.random.default_rng(40 + k)
    ctx = [int(x) for x in rng.integers(3000, 9000, 12)]
    inp = gen.make_inputs(len(ctx), 1, ctx, seed=41, topk=k)
    d = Dev(inp)
    mat = rng.standard_normal((len(ctx), max(ctx))).astype(np.float32)
    for rep in range(3):
        idx, _ = d.topk(mat)
        idx = idx.cpu().numpy()
        for b in range(len(ctx)):
            assert np.array_equal(idx[b], O.topk_select(mat[b, :ctx[b]], k)), (rep, b)


def test_topk_many_rows_mid_chunks():
    """64 rows of 16K tokens: 8K-token chunks, whose staging (32 KB) plus the
    kernel's static shared memory pass the default 48 KB limit."""
    ctx = [16384] * 64
    inp = gen.make_inputs(64, 1, ctx, seed=44)
    d = Dev(inp)
    mat = np.random.default_rng(44).standard_normal((64, 16384)).astype(np.float32)
    idx, _ = d.topk(mat)
    idx = idx.cpu().numpy()
    for b in (0, 17, 63):
        assert np.array_equal(idx[b], O.topk_select(mat[b], 2048)), b


@pytest.mark.parametrize("k", [2048, 256])
def test_topk_many_long_rows(k):
    """More rows than SMs, rows of 40K-70K tokens: three 32K-token chunks a row
    (the last one partial, some CTAs past the row's end), several waves of CTAs
    (a sampled bound at k = 2048, the group maxima at k = 256)."""
    rng = np.random.default_rng(46)
    ctx = [int(c) for c in rng.integers(40000, 70001, 160)]
    inp = gen.make_inputs(160, 1, ctx, seed=46, topk=k)
    d = Dev(inp)
    mat = rng.standard_normal((160, d.cap)).astype(np.float32)
    idx, _ = d.topk(mat)
    idx = idx.cpu().numpy()
    for b in (0, 1, 77, 151, 152, 159):
        assert np.array_equal(idx[b], O.topk_select(mat[b, :ctx[b]], k)), b


def test_topk_multi_token_rows_and_phys_rows():
    import dsa_sparse_mla_paged_gb300 as dsa

    inp = gen.make_inputs(2, 3, [5000, 9999], seed=8, bt_mode="permuted", holes=True)
    d = Dev(inp, flags=dsa.DSA_EMIT_PHYS_ROWS)
    rng = np.random.default_rng(1)
    mat = (rng.integers(0, 50, (6, 9999)) * 0.125).astype(np.float32)
    idx, pr = d.topk(mat, phys=True)
    idx, pr = idx.cpu().numpy(), pr.cpu().numpy()
    for b in range(2):
        for t in range(3):
            r = b * 3 + t
            L = O.visible_len(inp.ctx[b], 3, t)
            ref = O.topk_select(mat[r, :L], 2048)
            assert np.array_equal(idx[r], ref)
            assert np.array_equal(pr[r], O.physical_rows(inp.block_table[b], ref, 64))


def test_topk_small_k():
    inp = gen.make_inputs(2, 1, [100, 5000], seed=9, topk=16)
    d = Dev(inp)
    mat = np.random.default_rng(2).standard_normal((2, 5000)).astype(np.float32)
    idx, _ = d.topk(mat)
    for b in range(2):
        assert np.array_equal(idx.cpu().numpy()[b], O.topk_select(mat[b, :inp.ctx[b]], 16))


# ----------------------------------------------------------------------------- stage 3

def _oracle_mla_all(inp, idx):
    outs, lses = [], []
    for b in range(inp.batch):
        for t in range(inp.n_q):
            o, l = O.sparse_mla(inp, b, t, idx[b * inp.n_q + t])
            outs.append(o)
            lses.append(l)
    return np.stack(outs), np.stack(lses)


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_sparse_mla_over_oracle_indices(case):
    import torch

    inp = _small(case)
    d = Dev(inp)
    ref = {r: O.topk_select(s, 2048) for r, s in rows_scores_oracle(inp).items()}
    idx = np.stack([ref[r] for r in range(d.rows)])
    out, lse = d.mla(torch.from_numpy(idx).cuda())
    ro, rl = _oracle_mla_all(inp, idx)
    check_attention(bf16_to_np(out), lse.cpu().numpy(), ro, rl)


@pytest.mark.parametrize("lat_fmt", ["fp8", "nvfp4"])
def test_sparse_mla_latent_scale(lat_fmt):
    """A per-tensor latent scale other than 1 (and not a power of two) multiplies every
    dequantised latent value (the expansion then rounds each product to bf16)."""
    import dataclasses

    import torch

    key_fmt = "mxfp4" if lat_fmt == "nvfp4" else "fp8"
    inp = gen.make_inputs(2, 1, [5000, 3100], seed=21, bt_mode="permuted", key_fmt=key_fmt, lat_fmt=lat_fmt)
    inp = dataclasses.replace(inp, latent_scale=0.75)
    d = Dev(inp)
    ref = {r: O.topk_select(s, 2048) for r, s in rows_scores_oracle(inp).items()}
    idx = np.stack([ref[r] for r in range(d.rows)])
    out, lse = d.mla(torch.from_numpy(idx).cuda())
    ro, rl = _oracle_mla_all(inp, idx)
    check_attention(bf16_to_np(out), lse.cpu().numpy(), ro, rl)


def test_sparse_mla_holes_in_index_list():
    """-1 entries anywhere in the list are skipped; an all -1 row gives zeros and -inf."""
    import torch

    inp = gen.make_inputs(3, 1, [3000, 3000, 3000], seed=10, bt_mode="permuted")
    d = Dev(inp)
    rng = np.random.default_rng(3)
    idx = np.full((3, 2048), -1, np.int32)
    idx[0] = np.sort(rng.choice(3000, 2048, replace=False))
    idx[0, rng.integers(0, 2048, 300)] = -1
    idx[1, :5] = [2999, 0, 17, 17, 1500]  # unsorted and duplicated entries are legal
    out, lse = d.mla(torch.from_numpy(idx).cuda())
    ro, rl = _oracle_mla_all(inp, idx)
    check_attention(bf16_to_np(out), lse.cpu().numpy(), ro, rl)
    assert (bf16_to_np(out)[2] == 0).all() and np.isneginf(lse.cpu().numpy()[2]).all()


# ----------------------------------------------------------------------------- fused step

@pytest.mark.parametrize("case", range(len(SMALL)))
def test_decode_end_to_end_small(case):
    inp = _small(case)
    d = Dev(inp)
    out, lse, idx = d.decode()
    idx = idx.cpu().numpy()
    res = O.decode(inp)
    for (b, t), r in res.items():
        row = b * inp.n_q + t
        check_selection(idx[row], r["idx"], r["scores"], inp.topk,
                        selection_errscale(inp, score_error_scale(inp, b, t)))
    # attention over the GPU's own (validated) selection
    ro, rl = _oracle_mla_all(inp, idx)
    check_attention(bf16_to_np(out), lse.cpu().numpy(), ro, rl)


@pytest.mark.parametrize("nq,topk,ctx", [(8, 2048, [5000, 2100]), (2, 100, [3000, 90, 700]), (1, 1000, [1500, 40000])])
def test_decode_query_rows_and_k(nq, topk, ctx):
    """The largest query-row count (one 128-token tile per pipeline stage, shared
    head weights) and top-k sizes other than 2048 (fewer attention splits)."""
    inp = gen.make_inputs(len(ctx), nq, ctx, seed=300 + nq + topk, bt_mode="permuted", topk=topk)
    d = Dev(inp)
    out, lse, idx = d.decode()
    idx = idx.cpu().numpy()
    sc = d.scores().cpu().numpy()
    es = rows_error_scale(inp)
    for (b, t), r in O.decode(inp).items():
        row = b * inp.n_q + t
        check_scores(sc[row, :len(r["scores"])], r["scores"], es[row])
        check_selection(idx[row], r["idx"], r["scores"], inp.topk, selection_errscale(inp, es[row]))
    ro, rl = _oracle_mla_all(inp, idx)
    check_attention(bf16_to_np(out), lse.cpu().numpy(), ro, rl)


@pytest.mark.parametrize("nq,ctx", [(1, [150000, 90000]), (3, [100000])])
def test_decode_long_rows(nq, ctx):
    """Rows long enough that the top-k bound comes from the group maxima the
    scorer's epilogue writes (one and several query rows per request)."""
    inp = gen.make_inputs(len(ctx), nq, ctx, seed=330 + nq, bt_mode="permuted")
    d = Dev(inp)
    out, lse, idx = d.decode()
    idx = idx.cpu().numpy()
    res = O.decode(inp)
    for (b, t), r in res.items():
        row = b * inp.n_q + t
        check_selection(idx[row], r["idx"], r["scores"], inp.topk,
                        selection_errscale(inp, score_error_scale(inp, b, t)))
    ro, rl = _oracle_mla_all(inp, idx)
    check_attention(bf16_to_np(out), lse.cpu().numpy(), ro, rl)
    import dsa_sparse_mla_paged_gb300 as dsa

    assert dsa.get_device_error(d.ws) == 0


@pytest.mark.parametrize("kf,lf", [("fp8", "fp8"), ("mxfp4", "nvfp4")])
def test_decode_on_packed_block_rows(kf, lf):
    """A packed block-row cache (the article's cache: every layer's key page and
    latent page of one block in one power-of-two row): layer 1 of 3 is decoded in
    place through pool pointers into the row and the row size as page stride."""
    import torch
    import dsa_sparse_mla_paged_gb300 as dsa

    inp = gen.make_inputs(2, 2, [3000, 1500], seed=320, bt_mode="permuted", key_fmt=kf, lat_fmt=lf)
    kp, lp = inp.page_size * O.KEY_BYTES[kf], inp.page_size * O.LAT_BYTES[lf]
    layer = kp + lp
    row = 1 << (3 * layer - 1).bit_length()
    rng = np.random.default_rng(5)
    packed = rng.integers(0, 256, (inp.num_pages, row), dtype=np.uint8)  # other layers: any bytes
    packed[:, layer:layer + kp] = inp.key_pool[:, :kp]
    packed[:, layer + kp:2 * layer] = inp.lat_pool[:, :lp]
    d = Dev(inp)
    buf = torch.from_numpy(packed).cuda()
    d.key_pool = buf.view(-1)[layer:]
    d.lat_pool = buf.view(-1)[layer + kp:]
    d.p = dsa.make_params(batch=inp.batch, n_q=inp.n_q, max_pages_per_req=inp.max_pages, num_pages=inp.num_pages,
                          key_page_stride=row, lat_page_stride=row, key_fmt=d.p.key_fmt, lat_fmt=d.p.lat_fmt,
                          softmax_scale=inp.softmax_scale, latent_scale=inp.latent_scale)
    d.ws = torch.zeros(dsa.workspace_size(d.p), dtype=torch.uint8, device="cuda")
    out, lse, idx = d.decode()
    idx = idx.cpu().numpy()
    for (b, t), r in O.decode(inp).items():
        row_i = b * inp.n_q + t
        check_selection(idx[row_i], r["idx"], r["scores"], inp.topk,
                        selection_errscale(inp, score_error_scale(inp, b, t)))
    ro, rl = _oracle_mla_all(inp, idx)
    check_attention(bf16_to_np(out), lse.cpu().numpy(), ro, rl)
    assert dsa.get_device_error(d.ws) == 0


def test_determinism_and_batch_invariance():
    inp = gen.make_inputs(4, 1, [5000, 7000, 3000, 9000], seed=11, bt_mode="permuted")
    d = Dev(inp)
    o1, l1, i1 = d.decode()
    o2, l2, i2 = d.decode()
    import torch

    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert np.array_equal(i1.cpu().numpy(), i2.cpu().numpy())
    assert np.array_equal(l1.cpu().numpy(), l2.cpu().numpy())
    # request 2 alone gives the same bits as inside the batch
    one = gen.make_inputs(4, 1, [5000, 7000, 3000, 9000], seed=11, bt_mode="permuted")
    one.batch = 1
    one.ctx = one.ctx[2:3].copy()
    one.block_table = one.block_table[2:3].copy()
    for f in ("q_idx", "w", "q"):
        setattr(one, f, getattr(one, f)[2:3].copy())
    d1 = Dev(one)
    o3, l3, i3 = d1.decode()
    assert np.array_equal(i3.cpu().numpy()[0], i1.cpu().numpy()[2])
    assert torch.equal(o3.view(torch.int16), o1[2:3].view(torch.int16))
    assert torch.equal(l3, l1[2:3])


def test_device_error_word():
    """Bad block-table entries, context lengths and top-k indices are caught by the
    kernels' own bounds checks: they set the error word and never fault."""
    import torch
    import dsa_sparse_mla_paged_gb300 as dsa

    inp = gen.make_inputs(2, 1, [3000, 3000], seed=12)
    d = Dev(inp)
    assert dsa.get_device_error(d.ws) == 0
    d.decode()
    assert dsa.get_device_error(d.ws) == 0
    d.block_table[1, 3] = inp.num_pages + 5
    d.decode()
    assert dsa.get_device_error(d.ws) & dsa.DSA_DEVERR_BLOCK_TABLE
    assert dsa.get_device_error(d.ws) == 0  # read clears it
    d.block_table[1, 3] = int(inp.block_table[1, 3])
    d.ctx[0] = d.cap + 1
    d.decode()
    assert dsa.get_device_error(d.ws) & dsa.DSA_DEVERR_CTX
    d.ctx[0] = 3000
    idx = torch.full((2, 2048), -1, dtype=torch.int32, device="cuda")
    idx[0, 0] = 3000  # past the visible context
    idx[1, 0] = -2
    d.mla(idx)
    assert dsa.get_device_error(d.ws) & dsa.DSA_DEVERR_TOPK_INDEX


# ----------------------------------------------------------------------------- FP4 formats

SMALL_FP4 = [
    # (batch, n_q, ctx, bt_mode, holes, key_pad, lat_pad, key_fmt, lat_fmt)
    (3, 1, [4096 + 37, 2049, 300], "permuted", True, 0, 0, "mxfp4", "nvfp4"),
    (2, 6, [9000, 700], "permuted", False, 16, 32, "mxfp4", "fp8"),
    (2, 1, [3000, 65], "identity", False, 0, 16, "fp8", "nvfp4"),
]


@functools.lru_cache(maxsize=None)
def _small_fp4(i):
    b, nq, ctx, mode, holes, kp, lp, kf, lf = SMALL_FP4[i]
    return gen.make_inputs(b, nq, ctx, seed=200 + i, bt_mode=mode, holes=holes, key_page_pad=kp,
                           lat_page_pad=lp, key_fmt=kf, lat_fmt=lf, signed_w=i == 1)


def _mx_block_exponent_spread(inp):
    """Largest spread of a token's four E8M0 exponents (the MXFP4 key path is exact up to 14)."""
    e = inp.key_pool[:, 64 * 64:64 * 68].reshape(-1, 4).astype(np.int64)
    return int((e.max(axis=1) - e.min(axis=1)).max())


@pytest.mark.parametrize("case", range(len(SMALL_FP4)))
def test_fp4_indexer_scores_small(case):
    inp = _small_fp4(case)
    if inp.key_fmt == "mxfp4":
        assert _mx_block_exponent_spread(inp) <= 14
    d = Dev(inp)
    sc = d.scores().cpu().numpy()
    es = rows_error_scale(inp)
    for r, rs in rows_scores_oracle(inp).items():
        check_scores(sc[r, :len(rs)], rs, es[r])
        assert np.isnan(sc[r, len(rs):d.cap]).all()


@pytest.mark.parametrize("case", range(len(SMALL_FP4)))
def test_fp4_sparse_mla_over_oracle_indices(case):
    import torch

    inp = _small_fp4(case)
    d = Dev(inp)
    ref = {r: O.topk_select(s, 2048) for r, s in rows_scores_oracle(inp).items()}
    idx = np.stack([ref[r] for r in range(d.rows)])
    out, lse = d.mla(torch.from_numpy(idx).cuda())
    ro, rl = _oracle_mla_all(inp, idx)
    check_attention(bf16_to_np(out), lse.cpu().numpy(), ro, rl)


@pytest.mark.parametrize("case", range(len(SMALL_FP4)))
def test_fp4_decode_end_to_end_small(case):
    inp = _small_fp4(case)
    d = Dev(inp)
    out, lse, idx = d.decode()
    idx = idx.cpu().numpy()
    for (b, t), r in O.decode(inp).items():
        check_selection(idx[b * inp.n_q + t], r["idx"], r["scores"], inp.topk,
                        selection_errscale(inp, score_error_scale(inp, b, t)))
    ro, rl = _oracle_mla_all(inp, idx)
    check_attention(bf16_to_np(out), lse.cpu().numpy(), ro, rl)


def test_mxfp4_exponent_spread_sweep():
    """Tokens whose four block exponents spread by 8..20: scores exact (to fp32
    accumulation) up to 14, within the derived bound
    sum_h |w'_h| sum_{i in blocks 15+ below the largest} |q8_hi| 2^(e_max - 143)
    beyond, and within the 1e-3 score bar everywhere."""
    n = 13 * 200
    inp = gen.make_inputs(1, 1, [n], seed=211, key_fmt="mxfp4", lat_fmt="fp8")
    rng = np.random.default_rng(211)
    pool = inp.key_pool
    tok = np.arange(n)
    pg, sl = inp.block_table[0][tok // 64].astype(np.int64), tok % 64
    spread = 8 + tok % 13
    emax = rng.integers(100, 150, n)
    e = np.empty((n, 4), np.int64)
    for s_ in range(n):
        d = rng.integers(0, spread[s_] + 1, 4)
        d[rng.integers(0, 4)] = 0
        d[(np.argmax(d == 0) + 1 + rng.integers(0, 3)) % 4] = spread[s_]
        e[s_] = emax[s_] - d
    for s_ in range(n):
        off = 64 * 64 + 4 * sl[s_]
        pool[pg[s_], off:off + 4] = e[s_].astype(np.uint8)
    assert _mx_block_exponent_spread(inp) == 20
    d = Dev(inp)
    sc = d.scores().cpu().numpy()[0, :n].astype(np.float64)
    ref = rows_scores_oracle(inp)[0].astype(np.float64)
    es = score_error_scale(inp, 0, 0)
    check_scores(sc.astype(np.float32), ref.astype(np.float32), es)
    # the derived bound, from the oracle's query codes and folded weights
    from oracle.formats import bf16_decode, e4m3_decode
    codes, wp = O.quantize_index_query(bf16_decode(inp.q_idx[0, 0]).astype(np.float32), inp.w[0, 0])
    q8 = np.abs(e4m3_decode(codes)).reshape(32, 4, 32).sum(axis=2)  # [head, block] sum |q8|
    small = (e.max(axis=1, keepdims=True) - e) >= 15                 # [token, block]
    bound = (np.abs(wp.astype(np.float64))[None, :, None] * q8[None] * small[:, None, :]).sum(axis=(1, 2))
    bound *= 2.0 ** (e.max(axis=1) - 143)
    fp32_slack = 2.0 ** -14 * es
    err = np.abs(sc - ref)
    exact = spread <= 14
    assert (err[exact] <= fp32_slack[exact]).all(), float((err - fp32_slack)[exact].max())
    assert (err[~exact] <= bound[~exact] + fp32_slack[~exact]).all()
    assert (bound[exact] == 0).all() and (bound[~exact] > 0).any()


@pytest.mark.slow
def test_workload_fp4_decode():
    """32 requests x 6 causal query rows at 256K context with MXFP4 keys and NVFP4
    latents, in the benchmark's launch configuration, checked on sampled rows."""
    inp = _workload("b32x6_ctx256k_fp4")
    assert _mx_block_exponent_spread(inp) <= 14
    d = Dev(inp)
    out, lse, idx = d.decode()
    sc = d.scores().cpu().numpy()
    idx, out, lse = idx.cpu().numpy(), bf16_to_np(out), lse.cpu().numpy()
    for b in (0, 31):
        res = O.decode(inp, requests=[b])
        for t in (0, 5):
            r = res[(b, t)]
            row = b * inp.n_q + t
            es = score_error_scale(inp, b, t)
            check_scores(sc[row, :len(r["scores"])], r["scores"], es)
            check_selection(idx[row], r["idx"], r["scores"], inp.topk, selection_errscale(inp, es))
            o2, l2 = O.sparse_mla(inp, b, t, idx[row])
            check_attention(out[row][None], lse[row][None], o2[None], l2[None])


# ----------------------------------------------------------------------------- the five workloads

@functools.lru_cache(maxsize=1)
def _workload(name):
    # the tie workload's generator already plants hot tokens and tau ties
    return gen.make_workload(name)


WL_ROWS = {
    "b1_ctx4k": [0],
    "b8_ctx32k": list(range(8)),
    "b64_ctx16k_128k_ties": [0, 31, 63],
    "b4_ctx1m": [1],
}


@pytest.mark.slow
@pytest.mark.parametrize("name", list(WL_ROWS))
def test_workload_decode(name):
    """The full-size workloads in the launch configuration the benchmark times
    (dsa_decode), checked on sampled requests."""
    inp = _workload(name)
    d = Dev(inp)
    out, lse, idx = d.decode()
    sc = d.scores().cpu().numpy()
    idx, out, lse = idx.cpu().numpy(), bf16_to_np(out), lse.cpu().numpy()
    for b in WL_ROWS[name]:
        r = O.decode(inp, requests=[b])[(b, 0)]
        es = score_error_scale(inp, b, 0)
        check_scores(sc[b, :len(r["scores"])], r["scores"], es)
        nd = check_selection(idx[b], r["idx"], r["scores"], inp.topk, selection_errscale(inp, es))
        # top-k alone on the oracle's own scores is bit-exact
        ti, _ = d.topk(np.pad(r["scores"], (0, d.cap - len(r["scores"])))[None].repeat(inp.batch, 0))
        assert np.array_equal(ti.cpu().numpy()[b], r["idx"])
        if nd == 0:
            check_attention(out[b][None], lse[b][None], r["out"][None], r["lse"][None])
        o2, l2 = O.sparse_mla(inp, b, 0, idx[b])
        check_attention(out[b][None], lse[b][None], o2[None], l2[None])
        if name == "b64_ctx16k_128k_ties":
            hot = set(inp.meta["hot_positions"][b].tolist())
            assert hot <= set(idx[b].tolist())
            # the selection boundary lies inside the planted tie cluster
            ties = inp.meta["tau_exact"][b].tolist() + inp.meta["tau_near"][b].tolist() + [inp.meta["tau_token"][b]]
            kth = np.sort(r["scores"])[::-1][inp.topk - 1]
            assert all(abs(r["scores"][t] - kth) <= 1e-5 * abs(kth) for t in ties)
