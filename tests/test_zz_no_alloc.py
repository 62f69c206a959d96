"""dsa_topk_noalloc, the top-k entry point for callers that cannot allocate
device memory (its scratch is a static array inside libdsa), must give exactly
what dsa_topk gives with a workspace and what the oracle's top-k gives -- on two
calls in a row, so that state left in the shared array by one call cannot leak
into the next -- and a warm call must not change the device's free memory.

This file is named to be collected last."""
import ctypes

import numpy as np
import pytest

import dsa_sparse_mla_paged_gb300 as dsa
import gen
from oracle import dsa as O

pytestmark = pytest.mark.gpu


def _case(ctx, seed, levels):
    import torch

    inp = gen.make_inputs(len(ctx), 2, ctx, seed=seed, bt_mode="permuted")
    p = dsa.make_params(batch=inp.batch, n_q=2, max_pages_per_req=inp.max_pages, num_pages=inp.num_pages,
                        key_page_stride=inp.key_page_stride, lat_page_stride=inp.lat_page_stride,
                        flags=dsa.DSA_EMIT_PHYS_ROWS)
    rows, stride = inp.batch * 2, (max(ctx) + 3) // 4 * 4
    rng = np.random.default_rng(seed)
    sc = (rng.integers(0, levels, (rows, stride)) * 0.25 - 3.0).astype(np.float32)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return p, dev(sc), stride, dev(inp.ctx), dev(inp.block_table), rows, (inp, sc)


def _run_both(lib, case):
    import torch

    p, sc, stride, ctx, bt, rows, (inp, sc_np) = case
    ws = torch.zeros(dsa.workspace_size(p), dtype=torch.uint8, device="cuda")
    ref_i = torch.full((rows, 2048), -9, dtype=torch.int32, device="cuda")
    ref_p = torch.full_like(ref_i, -9)
    dsa.topk(p, sc, stride, ctx, bt, ref_i, ref_p, ws)
    got_i = torch.full_like(ref_i, -5)
    got_p = torch.full_like(ref_i, -5)
    # straight through the C ABI
    st = lib.dsa_topk_noalloc(ctypes.byref(p), sc.data_ptr(), stride, ctx.data_ptr(), bt.data_ptr(),
                              got_i.data_ptr(), got_p.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == dsa.DSA_OK, dsa.status_string(st)
    torch.cuda.synchronize()
    assert torch.equal(got_i, ref_i)
    assert torch.equal(got_p, ref_p)
    # and the oracle's selection of the same scores, row by row
    gi, gp = got_i.cpu().numpy(), got_p.cpu().numpy()
    for b in range(inp.batch):
        for t in range(2):
            r = b * 2 + t
            ref = O.topk_select(sc_np[r, :O.visible_len(inp.ctx[b], 2, t)], 2048)
            assert np.array_equal(gi[r], ref), r
            assert np.array_equal(gp[r], O.physical_rows(inp.block_table[b], ref, 64)), r
    # a warm call allocates nothing: the device's free memory is unchanged
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    st = lib.dsa_topk_noalloc(ctypes.byref(p), sc.data_ptr(), stride, ctx.data_ptr(), bt.data_ptr(),
                              got_i.data_ptr(), got_p.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == dsa.DSA_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.equal(got_i, ref_i)


def test_noalloc_topk_matches_workspace_topk_twice(lib, cuda_ok):
    _run_both(lib, _case([70000, 5000, 2049], seed=1, levels=40))   # several chunks, ties
    _run_both(lib, _case([9000, 131072], seed=2, levels=7))         # the second call reuses the array


def test_noalloc_topk_rejects_oversize(lib, cuda_ok):
    p = dsa.make_params(batch=33, n_q=2, max_pages_per_req=10, num_pages=400, key_page_stride=8448,
                        lat_page_stride=36864)
    st = lib.dsa_topk_noalloc(ctypes.byref(p), 0x10000, 640, 0x10000, 0x10000, 0x10000, None, None)
    assert st == dsa.DSA_ERR_UNSUPPORTED
    p = dsa.make_params(batch=1, n_q=1, max_pages_per_req=(1 << 20) // 64 + 1, num_pages=400,
                        key_page_stride=8448, lat_page_stride=36864)
    st = lib.dsa_topk_noalloc(ctypes.byref(p), 0x10000, 640, 0x10000, 0x10000, 0x10000, None, None)
    assert st == dsa.DSA_ERR_UNSUPPORTED
