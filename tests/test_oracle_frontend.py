"""Pins of the fused indexer front end's oracle (query norm, query projection,
FP8 quantisation folded into the head weights, new-token index key write) to
closed forms, worked examples of the formats and independent round trips."""
import numpy as np

from oracle import dsa as O
from oracle import frontend as F
from oracle.formats import e4m3_decode


def test_bf16_rounding_ties_to_even_and_matches_the_fp32_bit_formula():
    assert F.round_bf16(1 + 2.0 ** -8) == 1.0                       # midpoint, even mantissa below
    assert F.round_bf16(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6         # midpoint, even mantissa above
    assert F.round_bf16(-1 + 2.0 ** -9) == -1.0
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 6, 20000)).astype(np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    bits = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)   # integer RNE on the fp32 bits
    assert np.array_equal(F.bf16_bits(F.round_bf16(x.astype(np.float64))), bits)


def test_rms_norm_of_a_constant_vector_is_gamma_with_its_sign():
    g = F.round_bf16(np.linspace(-2, 2, 256))
    for a in (3.0, -0.25):
        n = F.rms_norm_bf16(np.full(256, a), g, 0.0)
        assert np.array_equal(n, np.sign(a) * g)
    # eps enters under the root: a = 1, eps = 3 halves the output
    assert np.array_equal(F.rms_norm_bf16(np.ones(256), g, 3.0), F.round_bf16(g / 2))
    # invariance to scaling the input by a power of two (eps = 0)
    c = F.round_bf16(np.random.default_rng(1).standard_normal(512))
    assert np.array_equal(F.rms_norm_bf16(c, np.ones(512), 0.0), F.rms_norm_bf16(c * 8, np.ones(512), 0.0))


def test_projection_selects_and_sums_exactly():
    v = F.round_bf16(np.random.default_rng(2).standard_normal((3, 64)))
    sel = np.zeros((5, 64))
    for i, j in enumerate([0, 7, 63, 5, 7]):
        sel[i, j] = 1.0
    assert np.array_equal(F.project_bf16(v, sel), v[:, [0, 7, 63, 5, 7]])
    ints = np.arange(64, dtype=np.float64)
    assert F.project_bf16(np.ones((1, 64)), ints[None, :])[0, 0] == 2016.0   # sum 0..63, exact in bf16


def test_folded_weights_reproduce_the_weighted_query():
    rng = np.random.default_rng(3)
    d_c = 256
    c = F.round_bf16(rng.standard_normal((2, d_c)))
    g = F.round_bf16(rng.uniform(0.5, 1.5, d_c))
    wq = F.round_bf16(rng.standard_normal((4096, d_c)) / 16)
    w = rng.uniform(0.1, 1.0, (2, 32)).astype(np.float32)
    q8, wp, q = F.frontend_query(c, g, wq, w, 1e-6)
    eff = wp.astype(np.float64)[:, :, None] * e4m3_decode(q8)     # what the scorer multiplies
    ref = w.astype(np.float64)[:, :, None] * q
    amax = np.abs(q).max(axis=2, keepdims=True) * w[:, :, None]
    # E4M3 keeps 3 mantissa bits: error <= half a step, 2^-4 relative, or a subnormal step
    assert (np.abs(eff - ref) <= 2.0 ** -4 * np.abs(ref) + amax * 2.0 ** -9 / 448 * 2 + 1e-12).all()
    # the largest element of each head maps to +-448
    top = np.abs(e4m3_decode(q8)).max(axis=2)
    assert np.allclose(top, 448.0)


def test_fp8_key_round_trip_and_exact_values():
    page_size = 64
    pool = np.zeros((3, page_size * 132), dtype=np.uint8)
    s = 2.0 ** -5
    k = np.zeros(128)
    k[:6] = np.array([448, -224, 1, 0.5, -3.25, 0.0]) * s            # every value an E4M3 code times s
    F.write_key(pool, 2, 17, k, "fp8", page_size)
    back = O.dequant_fp8_keys(pool, np.array([2]), np.array([17]), page_size)[0]
    assert np.array_equal(back, k)
    # only that slot's 132 bytes changed
    touched = np.nonzero(pool.reshape(-1))[0]
    lo, hi = 2 * pool.shape[1] + 17 * 128, 2 * pool.shape[1] + 64 * 128 + 17 * 4 + 4
    assert touched.min() >= lo and touched.max() < hi
    # a general key comes back within half an E4M3 step
    k = F.round_bf16(np.random.default_rng(4).standard_normal(128))
    F.write_key(pool, 0, 63, k, "fp8", page_size)
    back = O.dequant_fp8_keys(pool, np.array([0]), np.array([63]), page_size)[0]
    amax = np.abs(k).max()
    assert (np.abs(back - k) <= 2.0 ** -4 * np.abs(k) + amax / 448 * 2.0 ** -10 + 1e-12).all()


def test_mxfp4_key_worked_blocks():
    k = np.concatenate([[6, -3, 1.5, 0.5] + [0] * 28,        # amax 6: scale 2^0, exact codes
                        np.arange(1, 33),                    # amax 32: scale 2^3
                        [7] + [0] * 31,                      # 7 saturates to 6
                        [0] * 32]).astype(np.float64)        # empty block: scale byte 127, zeros
    packed, e8 = F.quantize_key_mxfp4(k)
    assert e8.tolist() == [127, 130, 127, 127]
    assert packed[0] == (7 | 13 << 4) and packed[1] == (3 | 1 << 4)
    # block 2 (values 1..32 over 8): 1/8 -> 0, 2/8 ties to 0, 3/8 -> 0.5, 6/8 ties to 1.0,
    # 20/8 = 2.5 ties to 2, 28/8 = 3.5 ties to 4, 32/8 = 4
    codes = np.empty(32, dtype=np.uint8)
    codes[0::2], codes[1::2] = packed[16:32] & 0xF, packed[16:32] >> 4
    assert codes[[0, 1, 2, 5, 19, 27, 31]].tolist() == [0, 0, 1, 2, 4, 6, 6]
    assert packed[32] == 7
    pool = np.zeros((1, 64 * 68), dtype=np.uint8)
    F.write_key(pool, 0, 5, k, "mxfp4")
    back = O.dequant_mxfp4_keys(pool, np.array([0]), np.array([5]), 64)[0]
    assert np.array_equal(back[:4], [6, -3, 1.5, 0.5]) and back[32 * 2] == 6.0
    assert back[32 + 31] == 32.0 and back[32 + 19] == 16.0


def test_mxfp4_key_round_trip_error_bound():
    k = F.round_bf16(np.random.default_rng(5).standard_normal(128) * 3)
    pool = np.zeros((1, 64 * 68), dtype=np.uint8)
    F.write_key(pool, 0, 0, k, "mxfp4")
    back = O.dequant_mxfp4_keys(pool, np.array([0]), np.array([0]), 64)[0]
    for blk in range(4):
        v, b = k[32 * blk:32 * blk + 32], back[32 * blk:32 * blk + 32]
        X = 2.0 ** (np.floor(np.log2(np.abs(v).max())) - 2)
        # E2M1 step is at most 2 (between 4 and 6), so error <= X; saturation error <= 2X
        assert (np.abs(b - v) <= 2 * X).all()
        assert (np.abs(b - v)[np.abs(v) <= 4 * X] <= 0.5 * X + 1e-12).all()


def test_frontend_writes_every_new_token_at_its_position():
    rng = np.random.default_rng(6)
    n_q, ctx = 3, [130, 64]
    bt = np.array([[4, 0, 2], [1, 3, 5]])
    x = F.round_bf16(rng.standard_normal((6, 256)))
    wk = F.round_bf16(rng.standard_normal((128, 256)) / 16)
    c = F.round_bf16(rng.standard_normal((6, 256)))
    g = np.ones(256)
    wq = F.round_bf16(rng.standard_normal((4096, 256)) / 16)
    w = np.ones((6, 32), np.float32)
    pool = np.zeros((6, 64 * 132), dtype=np.uint8)
    _, _, keys, out = F.frontend(c, g, wq, w, 1e-6, x, wk, pool, bt, ctx, n_q, "fp8")
    # request 0: tokens 127, 128, 129 -> page bt[0][1] slot 63, page bt[0][2] slots 0, 1
    for t, (pg, sl) in enumerate([(0, 63), (2, 0), (2, 1)]):
        got = O.dequant_fp8_keys(out, np.array([pg]), np.array([sl]), 64)[0]
        assert np.abs(got - keys[t]).max() <= np.abs(keys[t]).max() * 2.0 ** -4
    # request 1: tokens 61..63 -> page bt[1][0] = 1, slots 61..63
    for t in range(3):
        got = O.dequant_fp8_keys(out, np.array([1]), np.array([61 + t]), 64)[0]
        assert np.abs(got - keys[3 + t]).max() <= np.abs(keys[3 + t]).max() * 2.0 ** -4
    assert not out[[3, 4, 5]].any()
