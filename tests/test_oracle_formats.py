"""Pins of the oracle's number formats against library routines and the
format specifications (no GPU)."""
import numpy as np
import pytest
import torch

from conftest import read_golden


def _e4m3_table_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_bf16_round_trip_matches_torch(orc):
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        rng.standard_normal(2000).astype(np.float32) * np.float32(1e-30),
        np.array([0.0, -0.0, 1.0, 65504.0, 3.0e38, 1.00390625, 1.01171875], np.float32),
    ])
    # exact ties: bf16 value + half an ulp, both even and odd kept mantissas
    base = rng.standard_normal(2000).astype(np.float32)
    bits = base.view(np.uint32) & np.uint32(0xFFFF0000)
    ties = (bits | np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, ties])
    ours = orc.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = orc.bf16_to_f32(ref)
    assert np.array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16)
                          .to(torch.float32).numpy())


def test_e4m3_decode_matches_torch_table(orc):
    ref = _e4m3_table_torch()
    ours = orc.e4m3_decode(np.arange(256))
    finite = ~np.isnan(ref)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[finite], ref[finite])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x38] == 1.0


def test_e4m3_encode_matches_torch_in_range(orc):
    rng = np.random.default_rng(2)
    x = np.concatenate([
        rng.uniform(-448, 448, 30000),
        rng.standard_normal(10000) * 0.05,
        rng.standard_normal(5000) * 1e-3,
    ]).astype(np.float32)
    table = _e4m3_table_torch()[:127]
    mids = ((table[:-1] + table[1:]) / 2).astype(np.float32)   # exact ties
    assert np.array_equal(mids.astype(np.float64), (table[:-1] + table[1:]) / 2)
    x = np.concatenate([x, mids, -mids, table[:127].astype(np.float32)])
    ours = orc.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_encode_saturates(orc):
    # satfinite: beyond the largest finite value (448) the code clamps to it
    assert list(orc.e4m3_encode([448.0, 460.0, 464.0, 1e6, np.inf, -1e6, -np.inf])) == \
        [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


def test_e2m1_table_and_rounding(orc):
    vals = [float(s) for s in read_golden("e2m1_values.txt")["values"].split(",")]
    dec = orc.e2m1_decode(np.arange(16))
    assert list(dec[:8]) == vals
    assert list(dec[8:]) == [-v for v in vals]
    # every value round-trips; midpoints go to the even code; saturation at 6
    for c, v in enumerate(vals):
        assert orc.e2m1_encode([v])[0] == c
    for c in range(7):
        mid = (vals[c] + vals[c + 1]) / 2
        want = c if c % 2 == 0 else c + 1
        assert orc.e2m1_encode([mid])[0] == want, (c, mid)
        assert orc.e2m1_encode([np.nextafter(np.float32(mid), np.float32(0))])[0] == c
        assert orc.e2m1_encode([np.nextafter(np.float32(mid), np.float32(9))])[0] == c + 1
    assert list(orc.e2m1_encode([7.0, 1e9, -100.0])) == [7, 7, 15]


def test_e2m1_encode_is_nearest(orc):
    vals = np.array([float(s) for s in read_golden("e2m1_values.txt")["values"].split(",")])
    rng = np.random.default_rng(3)
    x = rng.uniform(-7, 7, 5000).astype(np.float32)
    codes = orc.e2m1_encode(x)
    dec = orc.e2m1_decode(codes)
    clipped = np.clip(np.abs(x.astype(np.float64)), 0, 6)
    best = np.min(np.abs(vals[None, :] - clipped[:, None]), axis=1)
    assert np.allclose(np.abs(np.abs(dec) - clipped), best)
    assert np.all((np.sign(dec) == np.sign(x)) | (dec == 0))
