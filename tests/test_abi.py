"""The C ABI on the CPU: the library loads, exports every symbol include/dsa.h
declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

import dsa_sparse_mla_paged_gb300 as dsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "dsa.h")).read()
    return sorted(set(re.findall(r"^\s*(?:dsa_status_t|const char\*)\s+(dsa_\w+)\s*\(", src, re.M)))


def test_every_declared_symbol_is_exported(lib):
    decl = _declared()
    assert set(decl) == set(dsa.EXPORTS)
    for name in decl:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for s in range(6):
        assert dsa.status_string(s).startswith("DSA_")
    assert "unknown" in dsa.status_string(99)


def _params(**kw):
    base = dict(batch=2, n_q=1, max_pages_per_req=10, num_pages=20, key_page_stride=8448, lat_page_stride=36864)
    base.update(kw)
    return dsa.make_params(**base)


def test_workspace_size_and_layout(lib):
    n1 = dsa.workspace_size(_params())
    n2 = dsa.workspace_size(_params(batch=4))
    n3 = dsa.workspace_size(_params(max_pages_per_req=20))
    assert n1 > 0 and n2 > n1 and n3 > n1 and n1 % 256 == 0
    # the scores region alone: rows * max_pages * 64 * 4 bytes
    assert n3 - n1 >= 2 * 10 * 64 * 4


@pytest.mark.parametrize("kw,status", [
    (dict(batch=0), dsa.DSA_ERR_INVALID),
    (dict(n_q=0), dsa.DSA_ERR_INVALID),
    (dict(batch=2, n_q=40000), dsa.DSA_ERR_UNSUPPORTED),
    (dict(topk=4096), dsa.DSA_ERR_UNSUPPORTED),
    (dict(topk=0), dsa.DSA_ERR_INVALID),
    (dict(page_size=32), dsa.DSA_ERR_UNSUPPORTED),
    (dict(key_page_stride=8440), dsa.DSA_ERR_INVALID),
    (dict(key_page_stride=8456), dsa.DSA_ERR_INVALID),
    (dict(lat_page_stride=36800), dsa.DSA_ERR_INVALID),
    (dict(num_pages=0), dsa.DSA_ERR_INVALID),
    (dict(key_fmt=7), dsa.DSA_ERR_INVALID),
    (dict(softmax_scale=0.0), dsa.DSA_ERR_INVALID),
    (dict(flags=0x100), dsa.DSA_ERR_INVALID),
])
def test_bad_params_rejected(lib, kw, status):
    with pytest.raises(dsa.DSAError) as e:
        dsa.workspace_size(_params(**kw))
    assert e.value.status == status


FAKE = 0x10000  # never dereferenced: validation fails before any CUDA call


def test_null_and_misaligned_pointers_rejected(lib):
    p = _params()
    need = dsa.workspace_size(p)
    ws = ctypes.c_void_p(FAKE)
    L = lib
    # null q_idx
    st = L.dsa_indexer_scores(ctypes.byref(p), None, FAKE, FAKE, FAKE, FAKE, FAKE, 640, FAKE, need, None)
    assert st == dsa.DSA_ERR_INVALID
    # misaligned key pool
    st = L.dsa_indexer_scores(ctypes.byref(p), FAKE, FAKE, FAKE + 4, FAKE, FAKE, FAKE, 640, FAKE, need, None)
    assert st == dsa.DSA_ERR_INVALID
    # score stride not a multiple of 4
    st = L.dsa_indexer_scores(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 641, FAKE, need, None)
    assert st == dsa.DSA_ERR_INVALID
    # short workspace
    st = L.dsa_indexer_scores(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 640, FAKE, need - 1, None)
    assert st == dsa.DSA_ERR_WORKSPACE
    # phys rows without the flag
    st = L.dsa_topk(ctypes.byref(p), FAKE, 640, FAKE, FAKE, FAKE, FAKE, FAKE, need, None)
    assert st == dsa.DSA_ERR_INVALID
    # null output of the attention
    st = L.dsa_sparse_mla_decode(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, need, None)
    assert st == dsa.DSA_ERR_INVALID
    # null params
    st = L.dsa_decode(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, need, None)
    assert st == dsa.DSA_ERR_INVALID
    st = L.dsa_get_device_error(None, None, None)
    assert st == dsa.DSA_ERR_INVALID


def test_dcp_merge_world_and_arguments_checked(lib):
    p = _params()
    need = dsa.workspace_size(p)
    L = lib
    for world in (0, -1, 17):
        st = L.dsa_dcp_topk_merge(ctypes.byref(p), FAKE, 640, FAKE, world, FAKE, None, FAKE, need, None)
        assert st == dsa.DSA_ERR_INVALID, world
    st = L.dsa_dcp_topk_merge(ctypes.byref(p), FAKE, 640, FAKE, 8, None, None, FAKE, need, None)
    assert st == dsa.DSA_ERR_INVALID
    st = L.dsa_dcp_topk_merge(ctypes.byref(p), FAKE + 4, 640, FAKE, 8, FAKE, None, FAKE, need, None)
    assert st == dsa.DSA_ERR_INVALID
    st = L.dsa_dcp_topk_merge(ctypes.byref(p), FAKE, 640, FAKE, 16, FAKE, None, FAKE, need - 1, None)
    assert st == dsa.DSA_ERR_WORKSPACE


def test_fp4_formats_take_their_own_page_strides(lib):
    """MXFP4 keys are 68 B and NVFP4 latents 352 B per token: a page stride below
    64 rows of the format (or not a multiple of 16 B) is rejected."""
    p = _params(key_fmt=dsa.DSA_KEY_MXFP4_68, key_page_stride=64 * 68,
                lat_fmt=dsa.DSA_LAT_NVFP4_352, lat_page_stride=64 * 352)
    assert dsa.workspace_size(p) > 0
    for kw in (dict(key_page_stride=64 * 68 - 16), dict(lat_page_stride=64 * 352 - 16),
               dict(key_page_stride=64 * 68 + 8)):
        q = _params(**{**dict(key_fmt=dsa.DSA_KEY_MXFP4_68, key_page_stride=64 * 68,
                              lat_fmt=dsa.DSA_LAT_NVFP4_352, lat_page_stride=64 * 352), **kw})
        with pytest.raises(dsa.DSAError) as e:
            dsa.workspace_size(q)
        assert e.value.status == dsa.DSA_ERR_INVALID


def test_library_missing_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(dsa, "_lib", None)
    monkeypatch.setattr(dsa, "library_path", lambda: str(tmp_path / "libdsa.so"))
    with pytest.raises(RuntimeError, match="not built"):
        dsa.load()


def test_lse_combine_arguments_checked(lib):
    p = _params()
    L = lib
    for parts in (0, 17):
        assert L.dsa_lse_combine(ctypes.byref(p), parts, FAKE, FAKE, FAKE, None, None) == dsa.DSA_ERR_INVALID
    assert L.dsa_lse_combine(ctypes.byref(p), 4, None, FAKE, FAKE, None, None) == dsa.DSA_ERR_INVALID
    assert L.dsa_lse_combine(ctypes.byref(p), 4, FAKE + 2, FAKE, FAKE, None, None) == dsa.DSA_ERR_INVALID
    assert L.dsa_lse_combine(ctypes.byref(p), 4, FAKE, FAKE, FAKE + 8, None, None) == dsa.DSA_ERR_INVALID


def test_frontend_arguments_checked(lib):
    p = _params()
    need = dsa.workspace_size(p)
    L = lib
    ok = dsa.FrontendDims(d_c=1536, d_model=7168, eps=1e-6)
    args = lambda dims, cq=FAKE, w=FAKE: (ctypes.byref(p), ctypes.byref(dims), cq, FAKE, FAKE, w, FAKE, FAKE, FAKE,
                                          FAKE, FAKE, None, None, FAKE, need, None)
    for bad in (dsa.FrontendDims(d_c=1000, d_model=7168), dsa.FrontendDims(d_c=1536, d_model=16384),
                dsa.FrontendDims(d_c=0, d_model=256)):
        assert L.dsa_indexer_frontend(*args(bad)) == dsa.DSA_ERR_UNSUPPORTED
    assert L.dsa_indexer_frontend(*args(dsa.FrontendDims(d_c=256, d_model=256, eps=-1.0))) == dsa.DSA_ERR_INVALID
    assert L.dsa_indexer_frontend(*args(ok, cq=None)) == dsa.DSA_ERR_INVALID
    assert L.dsa_indexer_frontend(*args(ok, cq=FAKE + 8)) == dsa.DSA_ERR_INVALID
    assert L.dsa_indexer_frontend(*args(ok, w=FAKE + 2)) == dsa.DSA_ERR_INVALID
    a = list(args(ok))
    a[14] = need - 1
    assert L.dsa_indexer_frontend(*a) == dsa.DSA_ERR_WORKSPACE


def test_prepared_flag_lets_the_query_be_null(lib):
    p = _params(flags=dsa.DSA_Q_PREPARED)
    need = dsa.workspace_size(p)
    # passes validation up to the workspace size check (no launch)
    st = lib.dsa_indexer_scores(ctypes.byref(p), None, None, FAKE, FAKE, FAKE, FAKE, 640, FAKE, need - 1, None)
    assert st == dsa.DSA_ERR_WORKSPACE
    q = _params()
    st = lib.dsa_indexer_scores(ctypes.byref(q), None, None, FAKE, FAKE, FAKE, FAKE, 640, FAKE, need, None)
    assert st == dsa.DSA_ERR_INVALID


def test_frontend_row_limit(lib):
    p = _params(batch=513)
    need = dsa.workspace_size(p)
    dims = dsa.FrontendDims(d_c=1536, d_model=7168, eps=1e-6)
    st = lib.dsa_indexer_frontend(ctypes.byref(p), ctypes.byref(dims), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                  FAKE, FAKE, None, None, FAKE, need, None)
    assert st == dsa.DSA_ERR_UNSUPPORTED


def test_prepared_query_needs_decode_rows(lib):
    p = _params(n_q=16, flags=dsa.DSA_Q_PREPARED)
    need = dsa.workspace_size(p)
    st = lib.dsa_indexer_scores(ctypes.byref(p), None, None, FAKE, FAKE, FAKE, FAKE, 640, FAKE, need, None)
    assert st == dsa.DSA_ERR_UNSUPPORTED


def test_prefill_world_and_rank_checked(lib):
    p = _params(n_q=64)
    need = dsa.workspace_size(p)
    call = lambda world, rank: lib.dsa_indexer_prefill_scores(ctypes.byref(p), world, rank, FAKE, FAKE, FAKE, FAKE,
                                                              FAKE, FAKE, 640, FAKE, need, None)
    assert call(0, 0) == dsa.DSA_ERR_INVALID
    assert call(2, 2) == dsa.DSA_ERR_INVALID
    assert call(2, -1) == dsa.DSA_ERR_INVALID
    assert call(3, 0) == dsa.DSA_ERR_INVALID       # 64 rows are not 6 slices of whole 8-row groups
    a = list((ctypes.byref(p), 4, 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 640, FAKE, need - 1, None))
    assert lib.dsa_indexer_prefill_scores(*a) == dsa.DSA_ERR_WORKSPACE


def test_selftest_wait_timeout_arguments_checked(lib):
    L = lib
    assert L.dsa_selftest_wait_timeout(None, 256, 100, None) == dsa.DSA_ERR_INVALID
    assert L.dsa_selftest_wait_timeout(FAKE + 4, 256, 100, None) == dsa.DSA_ERR_INVALID
    assert L.dsa_selftest_wait_timeout(FAKE, 2, 100, None) == dsa.DSA_ERR_INVALID
    assert L.dsa_selftest_wait_timeout(FAKE, 256, 0, None) == dsa.DSA_ERR_INVALID
    assert L.dsa_selftest_wait_timeout(FAKE, 256, (1 << 20) + 1, None) == dsa.DSA_ERR_INVALID
