"""GPU parity of the fused indexer front end (query norm -> query projection ->
FP8 query with folded head weights, new-token index key written to the cache)
against the oracle, and its hand-off to the scorer through the workspace.

Bars: with inputs whose products and sums are exact in fp32 (small integers
times powers of two, a power-of-two RMS), every output byte equals the
oracle's. With generic inputs: the scorer's effective weighted query
w' * E4M3(q8) is within half an E4M3 step of w * q, nearly every code equals
the oracle's and the others differ by one step (the fp32 and float64 sums may
round to different bf16 values).
"""
import numpy as np
import pytest

import dsa_sparse_mla_paged_gb300 as dsa
import gen
from oracle import dsa as O
from oracle import frontend as F
from oracle.formats import e4m3_decode

from dsa_testlib import Dev, bf16_to_np, check_attention, check_selection, score_error_scale, selection_errscale

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need(lib, cuda_ok):
    yield


def _bf16_tensor(a):
    import torch

    bits = F.bf16_bits(a)
    return torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.bfloat16)


def _exact_inputs(rows, d_c, d_model, seed):
    rng = np.random.default_rng(seed)
    e = -2 + (np.arange(rows) % 3)                      # per-row power-of-two magnitude
    c = np.where(rng.random((rows, d_c)) < 0.5, -1.0, 1.0) * 2.0 ** e[:, None]
    g = rng.integers(-32, 33, d_c) / 16.0
    wq = rng.integers(-8, 9, (4096, d_c)) / 32.0
    x = rng.integers(-16, 17, (rows, d_model)) / 8.0
    wk = rng.integers(-8, 9, (128, d_model)) / 64.0
    w = rng.uniform(0.1, 1.0, (rows, 32)).astype(np.float32)
    return c, g, wq, w, x, wk


def _generic_inputs(rows, d_c, d_model, seed):
    rng = np.random.default_rng(seed)
    c = F.round_bf16(rng.standard_normal((rows, d_c)) * 0.7)
    g = F.round_bf16(rng.uniform(0.5, 1.5, d_c))
    wq = F.round_bf16(rng.standard_normal((4096, d_c)) / np.sqrt(d_c))
    x = F.round_bf16(rng.standard_normal((rows, d_model)))
    wk = F.round_bf16(rng.standard_normal((128, d_model)) / np.sqrt(d_model))
    w = (rng.uniform(-1.0, 1.0, (rows, 32)) / np.sqrt(32)).astype(np.float32)
    return c, g, wq, w, x, wk


def _run(inp, d, fe, eps, flags=0):
    import torch

    c, g, wq, w, x, wk = fe
    dev = Dev(inp, flags=flags)
    rows = dev.rows
    dims = dsa.FrontendDims(d_c=c.shape[1], d_model=x.shape[1], eps=eps)
    q8 = torch.zeros((rows, 32, 128), dtype=torch.uint8, device="cuda")
    wout = torch.zeros((rows, 32), dtype=torch.float32, device="cuda")
    w_t = torch.from_numpy(w).cuda()
    dsa.indexer_frontend(dev.p, dims, _bf16_tensor(c), _bf16_tensor(g), _bf16_tensor(wq), w_t, _bf16_tensor(x),
                         _bf16_tensor(wk), dev.key_pool, dev.block_table, dev.ctx, dev.ws, q8_out=q8, w_out=wout)
    torch.cuda.synchronize()
    return dev, q8.cpu().numpy(), wout.cpu().numpy()


def _oracle(inp, fe, eps):
    c, g, wq, w, x, wk = fe
    return F.frontend(c, g, wq, w, eps, x, wk, inp.key_pool, inp.block_table, inp.ctx, inp.n_q, inp.key_fmt)


@pytest.mark.parametrize("key_fmt", ["fp8", "mxfp4"])
def test_frontend_bit_exact_on_exact_inputs(key_fmt):
    # 3 requests x 4 query rows = 12 rows: two passes of 8; new tokens straddle pages
    inp = gen.make_inputs(3, 4, [130, 64, 4000], seed=70, bt_mode="permuted", key_fmt=key_fmt)
    fe = _exact_inputs(12, 512, 768, 71)
    dev, q8, wp = _run(inp, None, fe, 0.0)
    assert dsa.get_device_error(dev.ws) == 0
    rq8, rwp, keys, pool = _oracle(inp, fe, 0.0)
    assert np.array_equal(q8, rq8)
    assert np.array_equal(wp.view(np.uint32), rwp.view(np.uint32))
    assert np.array_equal(dev.key_pool.cpu().numpy(), pool)


def test_frontend_generic_inputs_decode_shape():
    inp = gen.make_inputs(4, 2, [9000, 70000, 130, 2048], seed=72, bt_mode="permuted", holes=True)
    fe = _generic_inputs(8, 1536, 7168, 73)
    dev, q8, wp = _run(inp, None, fe, 1e-6)
    assert dsa.get_device_error(dev.ws) == 0
    rq8, rwp, keys, pool = _oracle(inp, fe, 1e-6)
    _, _, q = F.frontend_query(*fe[:4], 1e-6)
    eff = wp.astype(np.float64)[:, :, None] * e4m3_decode(q8)
    ref = fe[3].astype(np.float64)[:, :, None] * q
    amax = np.abs(ref).max(axis=2, keepdims=True)
    # half an E4M3 step of the value (2^-4 relative), one bf16 step of amax in the scale
    assert (np.abs(eff - ref) <= 2.0 ** -4 * np.abs(ref) + 2.0 ** -7 * amax).all()
    same = q8 == rq8
    assert same.mean() > 0.99
    steps = np.abs(q8.astype(np.int16) - rq8.astype(np.int16))
    assert (steps[~same] == 1).all()
    assert np.allclose(wp, rwp, rtol=2.0 ** -7, atol=0)
    # the keys read back from the cache are within half an E4M3 step of the oracle's keys
    got = dev.key_pool.cpu().numpy()
    for b in range(4):
        for t in range(2):
            pos = F.new_token_position(inp.ctx[b], 2, t)
            pg, sl = inp.block_table[b][pos // 64], pos % 64
            k = O.dequant_fp8_keys(got, np.array([pg]), np.array([sl]), 64)[0]
            ref_k = keys[b * 2 + t]
            assert (np.abs(k - ref_k) <= 2.0 ** -4 * np.abs(ref_k) + 2.0 ** -6 * np.abs(ref_k).max()).all()
    # every other byte of the pool is untouched
    mask = np.ones_like(got, dtype=bool)
    for b in range(4):
        for t in range(2):
            pos = F.new_token_position(inp.ctx[b], 2, t)
            pg, sl = inp.block_table[b][pos // 64], pos % 64
            mask[pg, sl * 128:(sl + 1) * 128] = False
            mask[pg, 64 * 128 + 4 * sl:64 * 128 + 4 * sl + 4] = False
    assert np.array_equal(got[mask], inp.key_pool[mask])


def test_prepared_query_feeds_the_scorer_and_the_decode():
    """frontend -> dsa_decode(DSA_Q_PREPARED) equals dsa_decode fed the oracle's
    bf16 q and w (same quantised query, same keys), bit for bit."""
    import torch

    inp = gen.make_inputs(2, 2, [5000, 3000], seed=74, bt_mode="permuted")
    fe = _exact_inputs(4, 256, 512, 75)
    dev, _, _ = _run(inp, None, fe, 0.0, flags=dsa.DSA_Q_PREPARED)
    assert dsa.get_device_error(dev.ws) == 0
    out_p, lse_p, idx_p = dev.decode()
    _, _, q = F.frontend_query(*fe[:4], 0.0)
    # the same step the usual way: the oracle's bf16 q, the same key pool
    plain = Dev(inp)
    plain.key_pool.copy_(dev.key_pool)
    plain.q_idx.copy_(_bf16_tensor(q.reshape(2, 2, 32, 128)))
    plain.w.copy_(torch.from_numpy(fe[3].reshape(2, 2, 32)).cuda())
    out_n, lse_n, idx_n = plain.decode()
    torch.cuda.synchronize()
    assert torch.equal(idx_p, idx_n)
    assert torch.equal(out_p.view(torch.int16), out_n.view(torch.int16))
    assert torch.equal(lse_p, lse_n)
    # and the step matches the oracle's on the updated cache
    upd = gen.make_inputs(2, 2, [5000, 3000], seed=74, bt_mode="permuted")
    upd.key_pool = dev.key_pool.cpu().numpy()
    upd.q_idx = F.bf16_bits(q.reshape(2, 2, 32, 128))
    upd.w = fe[3].reshape(2, 2, 32).astype(np.float32)
    idx = idx_p.cpu().numpy()
    for (b, t), r in O.decode(upd).items():
        row = b * 2 + t
        check_selection(idx[row], r["idx"], r["scores"], upd.topk,
                        selection_errscale(upd, score_error_scale(upd, b, t)))
        ro, rl = O.sparse_mla(upd, b, t, idx[row])
        check_attention(bf16_to_np(out_p[row]), lse_p[row].cpu().numpy(), ro, rl)


def test_bad_rows_write_no_key():
    inp = gen.make_inputs(2, 1, [100, 200], seed=76)
    inp.block_table[1][:] = -1          # request 1 has no pages
    fe = _exact_inputs(2, 256, 256, 77)
    dev, q8, _ = _run(inp, None, fe, 0.0)
    assert dsa.get_device_error(dev.ws) & dsa.DSA_DEVERR_BLOCK_TABLE
    got = dev.key_pool.cpu().numpy()
    # request 0's key went in; nothing else changed
    pos = 99
    pg, sl = inp.block_table[0][pos // 64], pos % 64
    changed = np.nonzero((got != inp.key_pool).any(axis=1))[0]
    assert set(changed.tolist()) <= {int(pg)}
    assert np.array_equal(q8, F.frontend_query(*fe[:4], 0.0)[0])
