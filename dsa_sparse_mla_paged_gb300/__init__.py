"""Python binding of libdsa (ctypes; argument marshalling only).

Every stage of the DSA decode step runs in the CUDA kernels of libdsa.so; this
module only turns tensors into device pointers and status codes into
exceptions. There is no fallback: if libdsa.so is missing, ``load()`` raises.

Entry points mirror include/dsa.h: ``workspace_size``, ``indexer_scores``,
``indexer_frontend``, ``indexer_prefill_scores``, ``topk``, ``topk_noalloc``, ``dcp_topk_merge``, ``lse_combine``, ``sparse_mla_decode``,
``decode``, ``get_device_error``, ``selftest_wait_timeout``, ``status_string``.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))

DSA_OK, DSA_ERR_INVALID, DSA_ERR_UNSUPPORTED, DSA_ERR_WORKSPACE, DSA_ERR_CUDA, DSA_ERR_TIMEOUT = range(6)
DSA_KEY_FP8_132, DSA_KEY_MXFP4_68 = 0, 1
DSA_LAT_FP8_576, DSA_LAT_NVFP4_352 = 0, 1
DSA_EMIT_PHYS_ROWS = 0x1
DSA_Q_PREPARED = 0x2
DSA_DEVERR_BLOCK_TABLE, DSA_DEVERR_CTX, DSA_DEVERR_TOPK_INDEX, DSA_DEVERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8

# Kernels one dsa_decode launches (q quantisation, indexer, top-k, sparse MLA,
# split combine); kept in step with csrc/.
KERNELS_PER_DECODE = 5

EXPORTS = (
    "dsa_workspace_size",
    "dsa_indexer_scores",
    "dsa_indexer_frontend",
    "dsa_indexer_prefill_scores",
    "dsa_topk",
    "dsa_topk_noalloc",
    "dsa_dcp_topk_merge",
    "dsa_lse_combine",
    "dsa_sparse_mla_decode",
    "dsa_decode",
    "dsa_get_device_error",
    "dsa_selftest_wait_timeout",
    "dsa_status_string",
)


class FrontendDims(ctypes.Structure):
    """dsa_frontend_dims_t."""

    _fields_ = [("d_c", ctypes.c_int32), ("d_model", ctypes.c_int32), ("eps", ctypes.c_float)]


class Params(ctypes.Structure):
    """dsa_params_t."""

    _fields_ = [
        ("batch", ctypes.c_int32),
        ("n_q", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("max_pages_per_req", ctypes.c_int32),
        ("idx_heads", ctypes.c_int32),
        ("idx_dim", ctypes.c_int32),
        ("heads", ctypes.c_int32),
        ("d_nope", ctypes.c_int32),
        ("d_rope", ctypes.c_int32),
        ("key_fmt", ctypes.c_int32),
        ("lat_fmt", ctypes.c_int32),
        ("key_page_stride", ctypes.c_int64),
        ("lat_page_stride", ctypes.c_int64),
        ("num_pages", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("latent_scale", ctypes.c_float),
        ("flags", ctypes.c_int32),
    ]


def make_params(*, batch, n_q, max_pages_per_req, num_pages, key_page_stride, lat_page_stride,
                topk=2048, page_size=64, key_fmt=DSA_KEY_FP8_132, lat_fmt=DSA_LAT_FP8_576,
                softmax_scale=1.0 / 192 ** 0.5, latent_scale=1.0, flags=0) -> Params:
    return Params(batch, n_q, topk, page_size, max_pages_per_req, 32, 128, 96, 512, 64, key_fmt, lat_fmt,
                  key_page_stride, lat_page_stride, num_pages, softmax_scale, latent_scale, flags)


class DSAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)}")


_lib = None


def library_path() -> str:
    return os.path.join(_PKG, "libdsa.so")


def load() -> ctypes.CDLL:
    """Load libdsa.so (built by ``__graft_entry__.build()``); raise if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libdsa.so is not built ({path}); run __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(Params)
    vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "dsa_workspace_size": [P, ctypes.POINTER(sz)],
        "dsa_indexer_scores": [P, vp, vp, vp, vp, vp, vp, i64, vp, sz, vp],
        "dsa_topk": [P, vp, i64, vp, vp, vp, vp, vp, sz, vp],
        "dsa_topk_noalloc": [P, vp, i64, vp, vp, vp, vp, vp],
        "dsa_indexer_frontend": [P, ctypes.POINTER(FrontendDims), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                 sz, vp],
        "dsa_indexer_prefill_scores": [P, ctypes.c_int32, ctypes.c_int32, vp, vp, vp, vp, vp, vp, i64, vp, sz, vp],
        "dsa_dcp_topk_merge": [P, vp, i64, vp, ctypes.c_int32, vp, vp, vp, sz, vp],
        "dsa_lse_combine": [P, ctypes.c_int32, vp, vp, vp, vp, vp],
        "dsa_sparse_mla_decode": [P, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp],
        "dsa_decode": [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp],
        "dsa_get_device_error": [vp, vp, ctypes.POINTER(ctypes.c_int32)],
        "dsa_selftest_wait_timeout": [vp, sz, ctypes.c_uint32, vp],
        "dsa_status_string": [ctypes.c_int],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_char_p if name == "dsa_status_string" else ctypes.c_int
    _lib = lib
    return lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _nbytes(ws) -> int:
    return ws.numel() * ws.element_size()


def _check(fn: str, st: int):
    if st != DSA_OK:
        raise DSAError(fn, st)


def status_string(status: int) -> str:
    return load().dsa_status_string(int(status)).decode()


def workspace_size(params: Params) -> int:
    n = ctypes.c_size_t(0)
    _check("dsa_workspace_size", load().dsa_workspace_size(ctypes.byref(params), ctypes.byref(n)))
    return int(n.value)


def indexer_scores(params, q_idx, w, key_pool, block_table, ctx_lens, scores, score_stride, ws, stream=None):
    _check("dsa_indexer_scores", load().dsa_indexer_scores(
        ctypes.byref(params), _ptr(q_idx), _ptr(w), _ptr(key_pool), _ptr(block_table), _ptr(ctx_lens),
        _ptr(scores), int(score_stride), _ptr(ws), _nbytes(ws), _stream(stream)))


def indexer_frontend(params, dims, c_q, gamma_q, w_q, w, x, w_k, key_pool, block_table, ctx_lens, ws,
                     q8_out=None, w_out=None, stream=None):
    """The fused front end: query norm -> projection -> FP8 q with folded weights
    (into the workspace, for a following call with DSA_Q_PREPARED) and the new
    tokens' index keys written into key_pool."""
    _check("dsa_indexer_frontend", load().dsa_indexer_frontend(
        ctypes.byref(params), ctypes.byref(dims), _ptr(c_q), _ptr(gamma_q), _ptr(w_q), _ptr(w), _ptr(x),
        _ptr(w_k), _ptr(key_pool), _ptr(block_table), _ptr(ctx_lens), _ptr(q8_out), _ptr(w_out), _ptr(ws),
        _nbytes(ws), _stream(stream)))


def indexer_prefill_scores(params, world, rank, q_idx, w, key_pool, block_table, ctx_lens, scores, score_stride, ws,
                           stream=None):
    """Scores of rank's two token slices of every request (2 * world slices)."""
    _check("dsa_indexer_prefill_scores", load().dsa_indexer_prefill_scores(
        ctypes.byref(params), int(world), int(rank), _ptr(q_idx), _ptr(w), _ptr(key_pool), _ptr(block_table),
        _ptr(ctx_lens), _ptr(scores), int(score_stride), _ptr(ws), _nbytes(ws), _stream(stream)))


def topk(params, scores, score_stride, ctx_lens, block_table, topk_idx, phys_rows, ws, stream=None):
    _check("dsa_topk", load().dsa_topk(
        ctypes.byref(params), _ptr(scores), int(score_stride), _ptr(ctx_lens), _ptr(block_table),
        _ptr(topk_idx), _ptr(phys_rows), _ptr(ws), _nbytes(ws), _stream(stream)))


def topk_noalloc(params, scores, score_stride, ctx_lens, block_table, topk_idx, phys_rows, stream=None):
    """dsa_topk without a workspace: for callers that cannot allocate device
    memory; its scratch is a static array inside libdsa (limits in include/dsa.h)."""
    _check("dsa_topk_noalloc", load().dsa_topk_noalloc(
        ctypes.byref(params), _ptr(scores), int(score_stride), _ptr(ctx_lens), _ptr(block_table),
        _ptr(topk_idx), _ptr(phys_rows), _stream(stream)))


def dcp_topk_merge(params, scores, score_stride, ctx_lens, world, topk_idx, stats, ws, stream=None):
    """The exact top-k merge of `world` token shards (decode context parallelism,
    emulated on one GPU); `stats` int32 [rows, 2] or None (see include/dsa.h)."""
    _check("dsa_dcp_topk_merge", load().dsa_dcp_topk_merge(
        ctypes.byref(params), _ptr(scores), int(score_stride), _ptr(ctx_lens), int(world), _ptr(topk_idx),
        _ptr(stats), _ptr(ws), _nbytes(ws), _stream(stream)))


def lse_combine(params, parts, part_out, part_lse, out, lse, stream=None):
    """Merge `parts` partial attention results (bf16 out, fp32 lse per shard) by their LSE."""
    _check("dsa_lse_combine", load().dsa_lse_combine(
        ctypes.byref(params), int(parts), _ptr(part_out), _ptr(part_lse), _ptr(out), _ptr(lse), _stream(stream)))


def sparse_mla_decode(params, q, lat_pool, block_table, ctx_lens, topk_idx, out, lse, ws, stream=None):
    _check("dsa_sparse_mla_decode", load().dsa_sparse_mla_decode(
        ctypes.byref(params), _ptr(q), _ptr(lat_pool), _ptr(block_table), _ptr(ctx_lens), _ptr(topk_idx),
        _ptr(out), _ptr(lse), _ptr(ws), _nbytes(ws), _stream(stream)))


def decode(params, q_idx, w, key_pool, q, lat_pool, block_table, ctx_lens, out, lse, topk_idx_out, ws,
           stream=None):
    _check("dsa_decode", load().dsa_decode(
        ctypes.byref(params), _ptr(q_idx), _ptr(w), _ptr(key_pool), _ptr(q), _ptr(lat_pool),
        _ptr(block_table), _ptr(ctx_lens), _ptr(out), _ptr(lse), _ptr(topk_idx_out), _ptr(ws), _nbytes(ws),
        _stream(stream)))


def get_device_error(ws, stream=None) -> int:
    """The workspace's DSA_DEVERR_* bits since the last read (then cleared). A
    timed-out wait (status DSA_ERR_TIMEOUT) is reported through the bits too."""
    code = ctypes.c_int32(0)
    st = load().dsa_get_device_error(_ptr(ws), _stream(stream), ctypes.byref(code))
    if st != DSA_ERR_TIMEOUT:
        _check("dsa_get_device_error", st)
    return int(code.value)


def selftest_wait_timeout(ws, poll_limit=10000, stream=None):
    """Run the bounded-wait abort path on purpose (sets DSA_DEVERR_TIMEOUT in ws)."""
    _check("dsa_selftest_wait_timeout", load().dsa_selftest_wait_timeout(
        _ptr(ws), _nbytes(ws), int(poll_limit), _stream(stream)))
