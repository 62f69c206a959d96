"""Pins of the oracle's DSA decode step against hand-worked values, closed forms,
brute force on tiny inputs and library routines (torch SDPA, scipy logsumexp)."""
import json
import math
import os
import struct

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import gen
from oracle import dsa as O
from oracle import formats as F

GOLD = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- indexer

def test_indexer_hand_example():
    with open(os.path.join(GOLD, "indexer_hand.json")) as f:
        g = json.load(f)
    s = O.indexer_scores_from(np.array(g["q"]), np.array(g["w"]), np.array(g["k"]))
    assert list(s) == g["scores"]
    top = O.topk_select(s.astype(np.float32), 2)
    assert list(top) == g["top2_ascending"]


def test_indexer_negative_weights_and_all_negative_dots():
    q = np.array([[1.0, 0.0], [0.0, 1.0]])
    w = np.array([-1.0, 0.5])
    k = np.array([[2.0, 4.0], [-1.0, -1.0], [3.0, -5.0]])
    # dots h0: 2, -1, 3 ; h1: 4, -1, -5
    assert list(O.indexer_scores_from(q, w, k)) == [-2.0 + 2.0, 0.0, -3.0]


def _brute_scores(inp, b, t):
    """Pure-Python loops through the block table; E4M3 through torch's decoder."""
    L = O.visible_len(inp.ctx[b], inp.n_q, t)
    qf = F.bf16_decode(inp.q_idx[b, t]).astype(np.float32)
    codes, wp = O.quantize_index_query(qf, inp.w[b, t])
    qv = torch.from_numpy(codes.reshape(-1)).view(torch.float8_e4m3fn).to(torch.float64).numpy().reshape(32, 128)
    out = []
    for s in range(L):
        page = int(inp.block_table[b][s // 64])
        slot = s % 64
        raw = inp.key_pool[page]
        kc = raw[slot * 128:(slot + 1) * 128].copy()
        kv = torch.from_numpy(kc).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        (scale,) = struct.unpack("<f", bytes(raw[64 * 128 + 4 * slot: 64 * 128 + 4 * slot + 4]))
        tot = 0.0
        for h in range(32):
            d = math.fsum(float(qv[h, i]) * float(kv[i]) * scale for i in range(128))
            tot += float(wp[h]) * max(0.0, d)
        out.append(tot)
    return np.array(out)


def test_indexer_scores_brute_force_through_pages():
    inp = gen.make_inputs(2, 2, [70, 131], seed=5, bt_mode="permuted", holes=True, key_page_pad=48)
    for b in range(2):
        for t in range(2):
            got = O.indexer_scores(inp, b, t)
            ref = _brute_scores(inp, b, t)
            assert got.shape == ref.shape
            np.testing.assert_allclose(got, ref.astype(np.float32), rtol=2e-7, atol=0)


def test_indexer_block_table_permutation_invariance():
    a = gen.make_inputs(1, 1, 1000, seed=9, bt_mode="identity")
    b = gen.make_inputs(1, 1, 1000, seed=9, bt_mode="identity")
    perm = np.random.default_rng(0).permutation(a.num_pages)
    b.key_pool = np.empty_like(a.key_pool)
    b.key_pool[perm] = a.key_pool
    b.block_table = np.where(a.block_table >= 0, perm[np.maximum(a.block_table, 0)], -1).astype(np.int32)
    assert (O.indexer_scores(a, 0, 0) == O.indexer_scores(b, 0, 0)).all()


def test_index_query_quantisation_recipe():
    rng = np.random.default_rng(1)
    q = F.bf16_decode(gen.f32_to_bf16_bits(rng.standard_normal((32, 128)).astype(np.float32))).astype(np.float32)
    q[3] = 0.0                                     # an all-zero head
    w = rng.uniform(0, 1, 32).astype(np.float32)
    codes, wp = O.quantize_index_query(q, w)
    vals = F.E4M3[codes]
    amax = np.abs(q).max(axis=1)
    # the largest element of each (non-zero) head maps to +-448 exactly
    for h in range(32):
        if h == 3:
            assert (vals[h] == 0).all() and wp[h] == 0
            continue
        j = int(np.argmax(np.abs(q[h])))
        assert abs(vals[h, j]) == 448.0
    # reconstruction within E4M3 precision (relative 2**-4, absolute at the subnormal step)
    rec = vals * (amax[:, None].astype(np.float64) / 448.0)
    err = np.abs(rec - q)
    assert (err <= np.abs(q) * 2.0 ** -4 + amax[:, None] / 448.0 * 2.0 ** -10).all()
    # the same fp32 steps through torch's own E4M3 conversion give the same codes
    qt = torch.from_numpy(q)
    amax_t = qt.abs().amax(dim=1)
    inv_t = torch.where(amax_t > 0, torch.tensor(448.0) / torch.where(amax_t > 0, amax_t, torch.ones_like(amax_t)),
                        torch.ones_like(amax_t))
    ref = (qt * inv_t[:, None]).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert (ref == vals).all()
    wp_t = torch.from_numpy(w) * (amax_t / 448.0)
    assert (wp_t.numpy() == wp).all()


def test_indexer_planted_multiple_of_query_closed_form():
    """Every head holds the same query; a key equal to its E4M3 codes with scale s
    scores s * |q8|^2 * sum_h w'_h (all products exact)."""
    inp = gen.make_inputs(1, 1, 64, seed=2)
    qrow = inp.q_idx[0, 0, 0].copy()
    inp.q_idx[0, 0, :] = qrow
    qf = F.bf16_decode(inp.q_idx[0, 0]).astype(np.float32)
    codes, wp = O.quantize_index_query(qf, inp.w[0, 0])
    pg = inp.block_table[0, 0]
    inp.key_pool[pg, 5 * 128:6 * 128] = codes[0]
    inp.key_pool[pg, 64 * 128 + 20:64 * 128 + 24] = np.frombuffer(struct.pack("<f", 0.75), dtype=np.uint8)
    s = O.indexer_scores(inp, 0, 0)[5]
    v = F.E4M3[codes[0]]
    expect = 0.75 * math.fsum(float(x) * float(x) for x in v) * math.fsum(float(x) for x in wp)
    assert s == np.float32(expect)


# ----------------------------------------------------------------------------- top-k

def _brute_topk(scores, k):
    order = sorted(range(len(scores)), key=lambda i: (-float(scores[i]), i))
    keep = sorted(order[:k])
    return keep + [-1] * (k - len(keep))


@pytest.mark.parametrize("L,k,levels", [(10, 4, 3), (300, 64, 5), (3000, 2048, 40), (5, 8, 2), (2048, 2048, 7)])
def test_topk_brute_force(L, k, levels):
    rng = np.random.default_rng(L + k)
    s = rng.integers(0, levels, L).astype(np.float32) * np.float32(0.25) - np.float32(0.5)
    s[rng.integers(0, L, max(1, L // 10))] = -0.0
    assert list(O.topk_select(s, k)) == _brute_topk(s, k)


def test_topk_all_equal_and_short():
    assert list(O.topk_select(np.ones(5000, np.float32), 2048)) == list(range(2048))
    out = O.topk_select(np.random.default_rng(0).standard_normal(100).astype(np.float32), 2048)
    assert list(out[:100]) == list(range(100)) and (out[100:] == -1).all()


def test_topk_continuous_matches_threshold():
    s = np.random.default_rng(4).standard_normal(50000).astype(np.float32)
    idx = O.topk_select(s, 2048)
    tau = O.kth_score(s, 2048)
    chosen = np.zeros(len(s), bool)
    chosen[idx] = True
    assert (s[chosen] >= tau).all() and (s[~chosen] <= tau).all() and chosen.sum() == 2048


def test_physical_rows():
    bt = np.array([7, 2, 5], dtype=np.int32)
    assert list(O.physical_rows(bt, np.array([0, 63, 64, 130, -1]), 64)) == [448, 511, 128, 322, -1]


# ----------------------------------------------------------------------------- attention

def _sdpa(q, c, scale):
    """torch SDPA (math path, fp64) with the latent as key and its first 512 dims as value."""
    qt = torch.from_numpy(q)[None, :, None, :]                       # [1, H, 1, 576]
    kt = torch.from_numpy(c)[None, None].expand(1, q.shape[0], -1, -1)
    vt = torch.from_numpy(c[:, :512])[None, None].expand(1, q.shape[0], -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return o[0, :, 0, :].numpy()


def test_mla_attention_matches_sdpa_and_logsumexp():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((96, 576))
    c = F.E4M3[rng.integers(0, 126, (300, 576))] * np.where(rng.random((300, 576)) < 0.5, -1, 1)
    sc = 1.0 / math.sqrt(192.0)
    out, lse = O.mla_attention(q, c, sc)
    np.testing.assert_allclose(out, _sdpa(q, c, sc), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, logsumexp(sc * q @ c.T, axis=1), rtol=1e-12)


def test_sparse_equals_dense_when_context_fits():
    inp = gen.make_inputs(1, 1, 1500, seed=8)
    r = O.decode(inp)[(0, 0)]
    assert list(r["idx"][:1500]) == list(range(1500))
    out_d, lse_d = O.dense_mla(inp, 0, 0)
    assert np.array_equal(r["out"], out_d) and np.array_equal(r["lse"], lse_d)


def test_sparse_equals_masked_dense():
    inp = gen.make_inputs(1, 1, 3000, seed=12)
    r = O.decode(inp)[(0, 0)]
    L = 3000
    c = O.dequant_latents(inp, 0, np.arange(L))
    q = F.bf16_decode(inp.q[0, 0])
    mask = np.zeros(L, bool)
    mask[r["idx"][r["idx"] >= 0]] = True
    qt = torch.from_numpy(q)[None, :, None, :]
    kt = torch.from_numpy(c)[None, None].expand(1, 96, -1, -1)
    vt = torch.from_numpy(c[:, :512])[None, None].expand(1, 96, -1, -1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=torch.from_numpy(mask)[None, None, None, :], scale=inp.softmax_scale)
    np.testing.assert_allclose(r["out"], ref[0, :, 0].numpy(), rtol=1e-10, atol=1e-12)


def test_one_token_context_returns_value():
    inp = gen.make_inputs(1, 1, 1, seed=3)
    out, lse = O.sparse_mla(inp, 0, 0, np.array([0]))
    c = O.dequant_latents(inp, 0, np.array([0]))
    assert np.array_equal(out, np.broadcast_to(c[0, :512], (96, 512)))
    q = F.bf16_decode(inp.q[0, 0])
    np.testing.assert_allclose(lse, inp.softmax_scale * q @ c[0], rtol=1e-14)


def test_empty_selection():
    inp = gen.make_inputs(1, 1, 10, seed=3)
    out, lse = O.sparse_mla(inp, 0, 0, np.full(2048, -1))
    assert (out == 0).all() and np.isneginf(lse).all()


def test_lse_combine_split_independence():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((96, 576))
    c = rng.standard_normal((500, 576))
    full_o, full_l = O.mla_attention(q, c, 0.07)
    cuts = [0, 37, 200, 500]
    parts = [O.mla_attention(q, c[a:b], 0.07) for a, b in zip(cuts[:-1], cuts[1:])]
    parts.append(O.mla_attention(q, c[:0], 0.07))            # an empty split
    o, l = O.lse_combine(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    np.testing.assert_allclose(o, full_o, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l, full_l, rtol=1e-13)


def test_causal_visibility_multi_token():
    inp = gen.make_inputs(1, 3, 100, seed=1)
    assert [O.visible_len(100, 3, t) for t in range(3)] == [98, 99, 100]
    r = O.decode(inp)
    for t in range(3):
        assert len(r[(0, t)]["scores"]) == 98 + t


# ----------------------------------------------------------------------------- FP4 formats

def test_mxfp4_key_decode_by_hand():
    pool = np.zeros((1, 64 * 68), dtype=np.uint8)
    pool[0, 0] = 0x72            # elements 0,1 = 1.0, 6.0
    pool[0, 16] = 0x0B           # element 32 = -1.5, element 33 = 0
    pool[0, 64 * 64 + 0] = 128   # block 0 scale 2
    pool[0, 64 * 64 + 1] = 125   # block 1 scale 1/4
    k = O.dequant_mxfp4_keys(pool, np.array([0]), np.array([0]), 64)
    assert k[0, 0] == 2.0 and k[0, 1] == 12.0 and k[0, 32] == -1.5 / 4 and k[0, 33] == 0.0


def test_nvfp4_latent_decode_by_hand():
    pool = np.zeros((1, 64 * 352), dtype=np.uint8)
    row = pool[0, 352:704]       # slot 1
    row[0] = 0x3A                # elements 0,1: -1.0, 1.5
    row[256] = 0x40              # block 0 scale E4M3 0x40 = 2.0
    row[288] = 0x38              # rope[0] = 1.0
    pool[0, 352:704] = row
    c = O.dequant_nvfp4_latents(pool, np.array([0]), np.array([1]), 0.5)
    assert c[0, 0] == -1.0 and c[0, 1] == 1.5 and c[0, 512] == 0.5 and (c[0, 2:512] == 0).all()


def test_generator_fp4_round_trip_error():
    inp = gen.make_inputs(1, 1, 128, seed=4, key_fmt="mxfp4", lat_fmt="nvfp4")
    k = O.dequant_keys(inp, 0, 128)
    c = O.dequant_latents(inp, 0, np.arange(128))
    # E2M1 keeps relative error of a block's largest values within 1/4 of the block scale
    assert np.isfinite(k).all() and np.isfinite(c).all()
    assert 0.5 < np.abs(k).std() < 2.0 and 0.5 < np.abs(c[:, :512]).std() < 2.0


def test_generator_fast_e2m1_encoder_matches_reference():
    rng = np.random.default_rng(5)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    mids = (grid[1:] + grid[:-1]) / 2
    x = np.concatenate([rng.standard_normal(200000) * 3, mids, -mids, grid, -grid,
                        np.nextafter(mids, 0), np.nextafter(mids, 9), [7.0, -7.0, 1e30, -0.0]])
    x = x.astype(np.float32)
    assert np.array_equal(gen.encode_e2m1_fast(x), gen.encode_e2m1(x))


# ----------------------------------------------------------------------------- byte model

def test_byte_model_article_numbers():
    assert O.KEY_BYTES["fp8"] == 128 + 4 and O.LAT_BYTES["fp8"] == 512 + 64
    assert O.LAT_BYTES["nvfp4"] == 512 // 2 + 512 // 16 + 64 and O.KEY_BYTES["mxfp4"] == 128 // 2 + 128 // 32
    # "about 23% of the bytes read by dense MLA" at long context (1M tokens)
    ctx = 1 << 20
    frac = (132 * ctx + 576 * 2048) / (576 * ctx)
    assert abs(frac - 0.23) < 0.005
    # MXFP4 shrinks the index cache by 48.5%
    assert round(1 - 68 / 132, 3) == 0.485
    # capacity ratios of the recipe page: NVFP4 latent ~1.5x, NVFP4 + MXFP4 ~1.7x
    assert round((576 + 132) / (352 + 132), 1) == 1.5
    assert round((576 + 132) / (352 + 68), 1) == 1.7
    assert O.Q_OUT_BYTES == 217216
    assert O.request_bytes(4096, 1, 2048) == 1937536
