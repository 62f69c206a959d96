"""Pins of the oracle's number formats against the OCP definitions and torch's converters."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_e4m3_spec_points():
    g = _load("e4m3_spec_points.json")
    for code, val in g["points"].items():
        got = F.E4M3[int(code, 16)]
        assert got == val and np.signbit(got) == np.signbit(val), code
    for code in g["nan"]:
        assert np.isnan(F.E4M3[int(code, 16)])


def test_e4m3_table_matches_torch_decoder():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = F.E4M3
    nan = np.isnan(ref)
    assert (nan == np.isnan(ours)).all()
    assert (ref[~nan] == ours[~nan]).all()
    # monotonic over the positive finite codes
    assert (np.diff(ours[:127]) > 0).all()


def test_e4m3_encoder_matches_torch_rne():
    rng = np.random.default_rng(11)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 50,
        rng.standard_normal(2000).astype(np.float32) * 1e-3,
        # exact midpoints between neighbouring codes (ties to even)
        ((F.E4M3[1:126] + F.E4M3[2:127]) / 2).astype(np.float32),
        -((F.E4M3[1:126] + F.E4M3[2:127]) / 2).astype(np.float32),
        np.array([0.0, -0.0, 448.0, -448.0, 447.9, 2.0 ** -10, 2.0 ** -9 * 1.5], dtype=np.float32),
    ])
    ours = F.e4m3_encode_rne_satfinite(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # compare values (torch and we may differ only in the sign of an exact zero)
    assert (F.E4M3[ours] == F.E4M3[ref]).all()


def test_e4m3_encoder_saturates():
    x = np.array([449.0, 464.0, 1e6, -1e30, np.inf, -np.inf], dtype=np.float32)
    v = F.E4M3[F.e4m3_encode_rne_satfinite(x)]
    assert list(v) == [448.0, 448.0, 448.0, -448.0, 448.0, -448.0]
    assert F.e4m3_encode_rne_satfinite(np.array([np.nan], dtype=np.float32))[0] == 0x7F


def test_e2m1_and_e8m0_spec_points():
    g = _load("e2m1_spec_points.json")
    for code, val in g["codes"].items():
        got = F.E2M1[int(code)]
        assert got == val and np.signbit(got) == np.signbit(val)
    for code, val in g["e8m0"].items():
        if code == "source":
            continue
        assert F.e8m0_decode(np.array([int(code)]))[0] == pytest.approx(val, rel=0, abs=0)
    assert np.isnan(F.e8m0_decode(np.array([255]))[0])


def test_e2m1_unpack_nibble_order():
    packed = np.array([0x71, 0xF8], dtype=np.uint8)  # low nibble first
    assert list(F.e2m1_unpack(packed)) == [0.5, 6.0, -0.0, -6.0]


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(3)
    x = torch.from_numpy(rng.standard_normal(5000).astype(np.float32)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    assert (F.bf16_decode(bits) == x.to(torch.float64).numpy()).all()
