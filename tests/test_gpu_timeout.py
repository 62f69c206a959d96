"""The bounded-wait abort path on the GPU, in a form that cannot hang: a test
kernel waits on an mbarrier nothing arrives on, with a short poll limit; the
timeout bit must come back through the workspace's error word (status
DSA_ERR_TIMEOUT), and the same context and workspace must then decode exactly."""
import ctypes

import pytest

import gen
from oracle import dsa as O

from dsa_testlib import Dev, bf16_to_np, check_attention, check_selection

import dsa_sparse_mla_paged_gb300 as dsa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need(lib, cuda_ok):
    yield


def test_wait_runs_out_then_decode_is_exact():
    import torch

    inp = gen.make_inputs(2, 1, [6000, 2100], seed=21, bt_mode="permuted")
    d = Dev(inp)
    d.decode()
    assert dsa.get_device_error(d.ws) == 0
    for limit in (1, 1000, 20000):
        dsa.selftest_wait_timeout(d.ws, limit)
        code = ctypes.c_int32(0)
        st = dsa.load().dsa_get_device_error(d.ws.data_ptr(), torch.cuda.current_stream().cuda_stream,
                                             ctypes.byref(code))
        assert st == dsa.DSA_ERR_TIMEOUT and code.value == dsa.DSA_DEVERR_TIMEOUT
        # read and cleared: the next read is clean
        assert dsa.get_device_error(d.ws) == 0
    # the same workspace and context after the aborted wait
    out, lse, idx = d.decode()
    assert dsa.get_device_error(d.ws) == 0
    idx, out, lse = idx.cpu().numpy(), bf16_to_np(out), lse.cpu().numpy()
    for b in range(2):
        r = O.decode(inp, requests=[b])[(b, 0)]
        o2, l2 = O.sparse_mla(inp, b, 0, idx[b])
        check_attention(out[b][None], lse[b][None], o2[None], l2[None])
        check_selection(idx[b], r["idx"], r["scores"], inp.topk)
