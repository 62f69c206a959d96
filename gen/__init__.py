"""Seeded synthetic inputs for one DSA decode step over a paged cache.

This module draws the bytes that both sides of every parity check read: the
query tensors, the head weights, the paged index-key and latent caches, the
block tables and the context lengths. It holds no step of the method (no
scoring, no selection, no attention): it only draws random values and stores
them in the cache formats, so that the CUDA library and the CPU oracle start
from identical bytes.

Formats written here (the page layout is this library's, the per-token sizes
are the ones the vLLM Kimi K3.1 Pro article gives in "Sparse attention in
K3.1 Pro" and "A KV cache for three kinds of state"):

* FP8 index key, 132 B/token: a page of ``page_size`` tokens is
  ``[page_size x 128 B E4M3 values][page_size x 4 B fp32 scale]``.
* FP8 latent, 576 B/token: a page is ``page_size`` contiguous rows of
  ``[512 E4M3 nope][64 E4M3 rope]``; one per-tensor ``latent_scale``.
* MXFP4 index key, 68 B/token: ``[page_size x 64 B E2M1 pairs][page_size x 4 B E8M0]``
  (one E8M0 exponent per 32 values; value 2i in the low nibble).
* NVFP4 latent, 352 B/token: rows of ``[256 B E2M1 pairs][32 B E4M3 block
  scales, one per 16 values][64 B E4M3 rope]``.

Value recipe (seeded ``numpy.random.Generator(PCG64(seed))``, draws in this
order: context lengths, block tables, q_idx, w, key values, key scales,
latent values, q, plants):

* q_idx, q: N(0, 1) rounded to bf16 (round to nearest even).
* w: U(0, 1) / sqrt(32) (or U(-1, 1) / sqrt(32) with ``signed_w``).
* FP8 key and latent values: E4M3 codes of N(0, 1), drawn through a 65,536-entry
  inverse-CDF table (each entry is the E4M3 code nearest to the normal quantile
  at the cell's midpoint), so the code histogram is that of E4M3(N(0, 1)) to
  within 2**-16 in probability.
* key scales: U(0.5, 2) in fp32.
* MXFP4 keys and NVFP4 latents: N(0, 1) values quantised block by block (MXFP4
  shared exponent floor(log2 amax) - 2, NVFP4 block scale E4M3(amax / 6), E2M1
  round-half-even, saturating). These pools are drawn in chunks of pages, each
  chunk from its own PCG64 stream seeded by (seed, 1 for keys / 2 for latents,
  chunk index), so that they can be filled by several threads; the main stream
  then skips them.
* tau ties (the 64-request tie workload): after the hot plants, the token the
  oracle ranks K-th in each request (read from a stored table that
  gen/make_tau_ties.py writes with the oracle; the generator itself scores
  nothing) has its key copied into 16 random positions, and into 16 more with
  its scale one fp32 ulp up or down.
"""
from __future__ import annotations

import hashlib
import json
import math
import os
from dataclasses import dataclass, field

import numpy as np

IDX_HEADS = 32
IDX_DIM = 128
HEADS = 96
D_NOPE = 512
D_ROPE = 64
D_QK = D_NOPE + D_ROPE
TOPK = 2048
PAGE_SIZE = 64

KEY_BYTES = {"fp8": IDX_DIM + 4, "mxfp4": IDX_DIM // 2 + IDX_DIM // 32}
LAT_BYTES = {"fp8": D_QK, "nvfp4": D_NOPE // 2 + D_NOPE // 16 + D_ROPE}


# ----------------------------------------------------------------------------
# encoders used only to synthesise inputs
# ----------------------------------------------------------------------------

def _e4m3_positive_values() -> np.ndarray:
    """Magnitudes of E4M3 codes 0..126 (0x7F is NaN), increasing with the code."""
    vals = np.empty(127, dtype=np.float64)
    for c in range(127):
        e, m = c >> 3, c & 7
        vals[c] = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_E4M3_POS = _e4m3_positive_values()


def encode_e4m3(x: np.ndarray) -> np.ndarray:
    """Nearest E4M3 code to each value (ties to the even code, clamped to +-448)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 448.0)
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 1, 126)
    lo = hi - 1
    dlo = a - _E4M3_POS[lo]
    dhi = _E4M3_POS[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(a == 0, 0, code).astype(np.uint8)
    return code | np.where(np.signbit(x) & (code != 0), 0x80, 0).astype(np.uint8)


_E2M1_POS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def encode_e2m1(x: np.ndarray) -> np.ndarray:
    """Nearest E2M1 code (0..15, sign in bit 3), ties to even, clamped to +-6."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 6.0)
    hi = np.clip(np.searchsorted(_E2M1_POS, a, side="left"), 1, 7)
    lo = hi - 1
    dlo = a - _E2M1_POS[lo]
    dhi = _E2M1_POS[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(a == 0, 0, code).astype(np.uint8)
    return code | np.where(np.signbit(x) & (code != 0), 0x8, 0).astype(np.uint8)


def encode_e2m1_fast(x: np.ndarray) -> np.ndarray:
    """``encode_e2m1`` in float32 arithmetic, for the big pools: the E2M1 grid has
    steps of 1/2 below 2, 1 below 4 and 2 up to 6, so the nearest point is a
    round-half-even of the value on that segment's scale (ties go to the even code,
    as in ``encode_e2m1``; the tests compare the two on every midpoint)."""
    x = np.asarray(x, dtype=np.float32)
    a = np.minimum(np.abs(x), np.float32(6.0))
    k1 = np.rint(a * np.float32(2.0))
    k2 = np.rint(a) + np.float32(2.0)
    k3 = np.rint(a * np.float32(0.5)) + np.float32(4.0)
    code = np.where(a < 2, k1, np.where(a < 4, k2, k3)).astype(np.uint8)
    return code | np.where(np.signbit(x) & (code != 0), np.uint8(8), np.uint8(0))


def _chunked(seed: int, tag: int, n: int, step: int, fill) -> None:
    """Call ``fill(rng, lo, hi)`` for every chunk [lo, hi) of range(n), each with
    its own PCG64 stream seeded by (seed, tag, chunk index), on a thread pool (the
    result does not depend on the number of threads)."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    starts = list(range(0, n, step))

    def one(i):
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, i])))
        fill(rng, starts[i], min(n, starts[i] + step))

    with ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1))) as ex:
        list(ex.map(one, range(len(starts))))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest even) and return the 16-bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def _normal_e4m3_lut() -> np.ndarray:
    from scipy.special import ndtri

    u = (np.arange(65536, dtype=np.float64) + 0.5) / 65536.0
    return encode_e4m3(ndtri(u))


_LUT = None


def sample_e4m3_normal(rng: np.random.Generator, n: int, out: np.ndarray | None = None) -> np.ndarray:
    """``n`` E4M3 codes distributed as E4M3(N(0, 1)) (see the module docstring)."""
    global _LUT
    if _LUT is None:
        _LUT = _normal_e4m3_lut()
    if out is None:
        out = np.empty(n, dtype=np.uint8)
    chunk = 1 << 25
    for i in range(0, n, chunk):
        m = min(chunk, n - i)
        u = rng.integers(0, 65536, size=m, dtype=np.uint16)
        out[i:i + m] = _LUT[u]
    return out


# ----------------------------------------------------------------------------
# the input bundle
# ----------------------------------------------------------------------------

@dataclass
class DSAInputs:
    """One decode step's inputs, all as host arrays of raw bytes / plain numbers."""

    name: str
    batch: int
    n_q: int
    ctx: np.ndarray            # int32 [B]; includes the n_q new tokens
    block_table: np.ndarray    # int32 [B, max_pages]; -1 past each request's last page
    num_pages: int
    q_idx: np.ndarray          # uint16 bf16 bits [B, n_q, 32, 128]
    w: np.ndarray              # float32 [B, n_q, 32]
    key_pool: np.ndarray       # uint8 [num_pages, key_page_stride]
    q: np.ndarray              # uint16 bf16 bits [B, n_q, 96, 576]
    lat_pool: np.ndarray       # uint8 [num_pages, lat_page_stride]
    key_fmt: str = "fp8"
    lat_fmt: str = "fp8"
    page_size: int = PAGE_SIZE
    topk: int = TOPK
    softmax_scale: float = 1.0 / math.sqrt(192.0)
    latent_scale: float = 1.0
    meta: dict = field(default_factory=dict)

    @property
    def key_page_stride(self) -> int:
        return int(self.key_pool.shape[1])

    @property
    def lat_page_stride(self) -> int:
        return int(self.lat_pool.shape[1])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])


def _block_tables(rng, ctx, page_size, mode, holes):
    B = len(ctx)
    npg = [(int(c) + page_size - 1) // page_size for c in ctx]
    maxp = max(max(npg), 1)
    total = int(sum(npg))
    if mode == "identity":
        ids = np.arange(total, dtype=np.int32)
    elif mode in ("permuted", "shared_shuffled"):
        ids = rng.permutation(total).astype(np.int32)
    else:
        raise ValueError(mode)
    num_pages = total
    if holes:
        # leave unused physical pages between the used ones
        num_pages = 2 * total + 3
        ids = (2 * ids + 1).astype(np.int32)
    bt = np.full((B, maxp), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        bt[b, :npg[b]] = ids[off:off + npg[b]]
        off += npg[b]
    return bt, num_pages


def _quantise_mxfp4_keys(x: np.ndarray) -> np.ndarray:
    """x float32 [n, 128] -> [n, 64 B E2M1 pairs + 4 B E8M0]."""
    n = x.shape[0]
    blk = x.reshape(n, 4, 32).astype(np.float64)
    amax = np.abs(blk).max(axis=2)
    e = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2, -127)
    e = np.clip(e, -127, 127)
    codes = encode_e2m1_fast((blk / (2.0 ** e)[:, :, None]).astype(np.float32)).reshape(n, 128)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    scales = (e + 127).astype(np.uint8)
    return np.concatenate([packed, scales], axis=1)


def _quantise_nvfp4_latents(x: np.ndarray) -> np.ndarray:
    """x float32 [n, 576] -> [n, 352]: 512 E2M1 with E4M3 scale per 16, 64 E4M3 rope."""
    n = x.shape[0]
    nope = x[:, :D_NOPE].reshape(n, 32, 16).astype(np.float64)
    amax = np.abs(nope).max(axis=2)
    sc_code = encode_e4m3(amax / 6.0)
    sc_val = _E4M3_POS[sc_code & 0x7F]
    safe = np.where(sc_val > 0, sc_val, 1.0)
    codes = encode_e2m1_fast((nope / safe[:, :, None]).astype(np.float32)).reshape(n, D_NOPE)
    codes = np.where(np.repeat(sc_val > 0, 16, axis=1), codes, 0).astype(np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    rope = encode_e4m3(x[:, D_NOPE:])
    return np.concatenate([packed, sc_code.astype(np.uint8), rope], axis=1)


def make_inputs(
    batch: int,
    n_q: int,
    ctx,
    seed: int,
    *,
    name: str = "custom",
    key_fmt: str = "fp8",
    lat_fmt: str = "fp8",
    bt_mode: str = "identity",
    holes: bool = False,
    key_page_pad: int = 0,
    lat_page_pad: int = 0,
    signed_w: bool = False,
    hot_plants: bool = False,
    tau_ties: str | None = None,
    page_size: int = PAGE_SIZE,
    topk: int = TOPK,
) -> DSAInputs:
    """Draw one decode step's inputs.

    ``ctx`` is an int, a list of ints, or ``("uniform", lo, hi)`` for context
    lengths drawn uniformly from [lo, hi]. ``hot_plants`` adds, per request,
    256 tokens in 32 groups of 8 whose index keys are the E4M3 codes of
    ``2 * qbar / rms(qbar)`` with ``qbar = sum_h w_h q_h`` of the request's first
    query token; the 8 keys of a group share bytes and scale (exact ties).
    ``tau_ties`` names a stored table (``gen/tau_ties/<name>.json``) that gives,
    per request, the token ranked K-th by the oracle after the hot plants; its
    key bytes and scale are then copied into 16 other random positions (exact
    ties at tau) and into 16 more with the scale moved by one fp32 ulp, up or
    down (near ties).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    if isinstance(ctx, tuple) and ctx[0] == "uniform":
        ctx_arr = rng.integers(ctx[1], ctx[2], size=batch, endpoint=True).astype(np.int32)
    elif np.isscalar(ctx):
        ctx_arr = np.full(batch, int(ctx), dtype=np.int32)
    else:
        ctx_arr = np.asarray(ctx, dtype=np.int32)
        assert ctx_arr.shape == (batch,)
    assert (ctx_arr >= n_q).all(), "every request holds at least its n_q new tokens"

    bt, num_pages = _block_tables(rng, ctx_arr, page_size, bt_mode, holes)

    q_idx = f32_to_bf16_bits(rng.standard_normal((batch, n_q, IDX_HEADS, IDX_DIM), dtype=np.float32))
    if signed_w:
        w = (rng.uniform(-1.0, 1.0, (batch, n_q, IDX_HEADS)) / math.sqrt(IDX_HEADS)).astype(np.float32)
    else:
        w = (rng.uniform(0.0, 1.0, (batch, n_q, IDX_HEADS)) / math.sqrt(IDX_HEADS)).astype(np.float32)

    kb = KEY_BYTES[key_fmt]
    lb = LAT_BYTES[lat_fmt]
    key_stride = page_size * kb + key_page_pad
    lat_stride = page_size * lb + lat_page_pad
    key_pool = np.zeros((num_pages, key_stride), dtype=np.uint8)
    lat_pool = np.zeros((num_pages, lat_stride), dtype=np.uint8)

    if key_fmt == "fp8":
        vals = sample_e4m3_normal(rng, num_pages * page_size * IDX_DIM)
        key_pool[:, :page_size * IDX_DIM] = vals.reshape(num_pages, page_size * IDX_DIM)
        scales = rng.uniform(0.5, 2.0, (num_pages, page_size)).astype(np.float32)
        key_pool[:, page_size * IDX_DIM:page_size * kb] = scales.view(np.uint8).reshape(num_pages, page_size * 4)
    elif key_fmt == "mxfp4":
        def fill_keys(r, p0, p1):
            x = r.standard_normal(((p1 - p0) * page_size, IDX_DIM), dtype=np.float32)
            enc = _quantise_mxfp4_keys(x).reshape(p1 - p0, page_size, 68)
            key_pool[p0:p1, :page_size * 64] = enc[:, :, :64].reshape(p1 - p0, -1)
            key_pool[p0:p1, page_size * 64:page_size * 68] = enc[:, :, 64:].reshape(p1 - p0, -1)

        _chunked(seed, 1, num_pages, 256, fill_keys)
    else:
        raise ValueError(key_fmt)

    if lat_fmt == "fp8":
        if lat_page_pad == 0:
            sample_e4m3_normal(rng, lat_pool.size, out=lat_pool.reshape(-1))
        else:
            vals = sample_e4m3_normal(rng, num_pages * page_size * D_QK)
            lat_pool[:, :page_size * D_QK] = vals.reshape(num_pages, page_size * D_QK)
    elif lat_fmt == "nvfp4":
        def fill_lat(r, p0, p1):
            x = r.standard_normal(((p1 - p0) * page_size, D_QK), dtype=np.float32)
            lat_pool[p0:p1, :page_size * lb] = _quantise_nvfp4_latents(x).reshape(p1 - p0, -1)

        _chunked(seed, 2, num_pages, 64, fill_lat)
    else:
        raise ValueError(lat_fmt)

    q = f32_to_bf16_bits(rng.standard_normal((batch, n_q, HEADS, D_QK), dtype=np.float32))

    meta = {}
    if hot_plants:
        assert key_fmt == "fp8"
        planted = []
        for b in range(batch):
            qf = (q_idx[b, 0].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            qbar = (w[b, 0].astype(np.float64)[:, None] * qf).sum(axis=0)
            rms = math.sqrt(float((qbar ** 2).mean()))
            codes = encode_e4m3(2.0 * qbar / rms)
            L = int(ctx_arr[b])
            npos = min(256, L)
            pos = np.sort(rng.choice(L, size=npos, replace=False))
            grp_scale = rng.uniform(0.5, 2.0, 32).astype(np.float32)
            for j, s in enumerate(pos):
                pg, sl = bt[b, s // page_size], s % page_size
                key_pool[pg, sl * IDX_DIM:(sl + 1) * IDX_DIM] = codes
                off = page_size * IDX_DIM + 4 * sl
                key_pool[pg, off:off + 4] = grp_scale[j // 8:j // 8 + 1].view(np.uint8)
            planted.append(pos)
        meta["hot_positions"] = planted

    if tau_ties:
        assert key_fmt == "fp8"
        table = load_tau_table(tau_ties)
        assert len(table) == batch, "the tie table was written for another batch"
        exact, near = [], []
        for b in range(batch):
            s_tau = int(table[b]["s_tau"])
            pg, sl = bt[b, s_tau // page_size], s_tau % page_size
            kb = key_pool[pg, sl * IDX_DIM:(sl + 1) * IDX_DIM].copy()
            off = page_size * IDX_DIM + 4 * sl
            sb = key_pool[pg, off:off + 4].copy()
            if _key_digest(kb, sb) != table[b]["key_digest"]:
                raise ValueError(f"tie table {tau_ties!r} does not match the generated keys (request {b}); "
                                 "rewrite it with gen/make_tau_ties.py")
            taken = {s_tau} | set(meta.get("hot_positions", [[]] * batch)[b].tolist())
            draw = rng.choice(int(ctx_arr[b]), size=min(int(ctx_arr[b]), 128), replace=False)
            pos = [int(x) for x in draw if int(x) not in taken][:32]
            scale = sb.view(np.float32)[0]
            for j, s in enumerate(pos):
                p2, l2 = bt[b, s // page_size], s % page_size
                key_pool[p2, l2 * IDX_DIM:(l2 + 1) * IDX_DIM] = kb
                v = scale if j < 16 else np.nextafter(scale, np.float32(np.inf) if j % 2 else np.float32(0))
                o2 = page_size * IDX_DIM + 4 * l2
                key_pool[p2, o2:o2 + 4] = np.array([v], np.float32).view(np.uint8)
            exact.append(np.array(pos[:16]))
            near.append(np.array(pos[16:]))
        meta["tau_token"] = [int(t["s_tau"]) for t in table]
        meta["tau_exact"] = exact
        meta["tau_near"] = near

    return DSAInputs(
        name=name, batch=batch, n_q=n_q, ctx=ctx_arr, block_table=bt, num_pages=num_pages,
        q_idx=q_idx, w=w, key_pool=key_pool, q=q, lat_pool=lat_pool, key_fmt=key_fmt,
        lat_fmt=lat_fmt, page_size=page_size, topk=topk, meta=meta,
    )


TAU_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tau_ties")


def _key_digest(key_bytes: np.ndarray, scale_bytes: np.ndarray) -> str:
    return hashlib.sha256(key_bytes.tobytes() + scale_bytes.tobytes()).hexdigest()[:16]


def load_tau_table(name: str) -> list:
    """Per request {"s_tau": token, "key_digest": ...} from gen/tau_ties/<name>.json."""
    with open(os.path.join(TAU_DIR, name + ".json")) as f:
        return json.load(f)["requests"]


# The five workloads, by what they are. Sizes follow the DSA decode shapes of the
# article (32 indexer heads x 128, 96 query heads x 576, top-2048, 64-token pages).
WORKLOADS = {
    "b1_ctx4k": dict(batch=1, n_q=1, ctx=4096, seed=0, bt_mode="identity"),
    "b8_ctx32k": dict(batch=8, n_q=1, ctx=32768, seed=1, bt_mode="permuted"),
    "b64_ctx16k_128k_ties": dict(batch=64, n_q=1, ctx=("uniform", 16384, 131072), seed=2,
                                 bt_mode="shared_shuffled", hot_plants=True, tau_ties="b64_ctx16k_128k_ties"),
    "b4_ctx1m": dict(batch=4, n_q=1, ctx=1 << 20, seed=3, bt_mode="permuted"),
    "b32x6_ctx256k_fp4": dict(batch=32, n_q=6, ctx=1 << 18, seed=4, bt_mode="permuted",
                              key_fmt="mxfp4", lat_fmt="nvfp4"),
    # a prefill chunk: 2,048 new tokens appended to a 150K-token cached prefix
    "b1_prefill2k_ctx150k": dict(batch=1, n_q=2048, ctx=150 * 1024 + 2048, seed=7, bt_mode="permuted"),
    "b1_prefill512_ctx32k": dict(batch=1, n_q=512, ctx=32768, seed=8, bt_mode="permuted"),
    # small cases for kernel profiles: each kernel's own inputs still exceed the 129 MB L2
    "b4_ctx256k": dict(batch=4, n_q=1, ctx=1 << 18, seed=5, bt_mode="permuted"),
    "b64_ctx16k": dict(batch=64, n_q=1, ctx=1 << 14, seed=6, bt_mode="permuted"),
    # six-row scorer cases (keys above L2): FP8 and MXFP4 keys
    "b8x6_ctx256k": dict(batch=8, n_q=6, ctx=1 << 18, seed=9, bt_mode="permuted"),
    "b8x6_ctx256k_fp4": dict(batch=8, n_q=6, ctx=1 << 18, seed=10, bt_mode="permuted", key_fmt="mxfp4",
                             lat_fmt="nvfp4"),
}
WORKLOAD_ORDER = list(WORKLOADS)


def make_workload(name: str, **overrides) -> DSAInputs:
    kw = dict(WORKLOADS[name])
    kw.update(overrides)
    return make_inputs(name=name, **kw)
