"""Pins of the oracle's QK Hadamard rotation (paper Appx B, §4.1 "Baselines")
against scipy's Hadamard matrix, exact integer inputs and orthogonality, and
of the rotated preparations against torch casts (no GPU)."""
import numpy as np
import pytest
import torch

import synth

scipy_linalg = pytest.importorskip("scipy.linalg")


def _f(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16) \
        .to(torch.float64).numpy()


def _e4m3(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


H = scipy_linalg.hadamard(128).astype(np.float64)


def test_matches_scipy_hadamard(orc):
    x = np.random.default_rng(1).standard_normal((16, 128)).astype(np.float32)
    y = orc.hadamard128(x)
    ref = x.astype(np.float64) @ H / np.sqrt(128)
    assert np.max(np.abs(y - ref)) <= 1e-6 * np.max(np.abs(ref))


def test_integer_rows_round_once(orc):
    """Small integers: every butterfly is exact, so the result is the exact
    integer transform times fp32(1/sqrt(128)), rounded once in fp32."""
    x = np.random.default_rng(2).integers(-8, 9, (8, 128)).astype(np.float32)
    y = orc.hadamard128(x)
    exact = (x.astype(np.int64) @ H.astype(np.int64)).astype(np.float32)
    want = exact * np.float32(1 / np.sqrt(128))
    assert np.array_equal(y, want)
    e0 = np.zeros((1, 128), np.float32)
    e0[0, 0] = 1.0
    assert np.all(orc.hadamard128(e0) == np.float32(1 / np.sqrt(128)))


def test_orthogonal_and_scores_unchanged(orc):
    rng = np.random.default_rng(3)
    q = rng.standard_normal((8, 128)).astype(np.float32)
    k = rng.standard_normal((8, 128)).astype(np.float32)
    back = orc.hadamard128(orc.hadamard128(q))          # H / sqrt(128) is its own inverse
    assert np.max(np.abs(back - q)) <= 1e-5
    s = orc.hadamard128(q).astype(np.float64) @ orc.hadamard128(k).astype(np.float64).T
    assert np.max(np.abs(s - q.astype(np.float64) @ k.T)) <= 1e-4


def test_rotated_preparation8(orc):
    N = 520
    q, k, v = synth.make_qkv(1, 1, N, 128, 8, 61)
    p = orc.prepare8(q[0, 0], k[0, 0], v[0, 0], 8, 3, 61, hadamard=True)
    ref = orc.prepare8(q[0, 0], k[0, 0], v[0, 0], 8, 3, 61)
    for key in ("perm", "labels", "kbar", "rhatT", "sv", "mu", "mutilde"):
        assert np.array_equal(p[key], ref[key]), key
    qr = orc.hadamard128(_f(q[0, 0]).astype(np.float32))
    kp = (_f(k[0, 0])[p["perm"]].astype(np.float32) - _f(p["kbar"]).astype(np.float32))
    kr = orc.hadamard128(kp.astype(np.float32))
    for x, codes, scales in ((qr, p["qhat"], p["sq"]), (kr, p["khat"], p["sk"])):
        for j in range(scales.size):
            blk = x[j * 128:(j + 1) * 128]
            s = np.float32(np.abs(blk).max()) / np.float32(448)
            assert scales[j] == s
            assert np.array_equal(codes[j * 128:j * 128 + len(blk)], _e4m3(blk / s))
    assert not np.array_equal(p["qhat"], ref["qhat"])


def test_rotated_preparation4(orc):
    N = 300
    q, k, v = synth.make_qkv(1, 1, N, 128, 8, 62)
    p = orc.prepare4(q[0, 0], k[0, 0], v[0, 0], 8, 3, 62, hadamard=True)
    ref = orc.prepare4(q[0, 0], k[0, 0], v[0, 0], 8, 3, 62)
    for key in ("perm", "kbar", "r4T", "r4s", "gr", "mu"):
        assert np.array_equal(p[key], ref[key]), key
    qr = orc.hadamard128(_f(q[0, 0]).astype(np.float32))
    assert np.float32(p["gq"][0]) == np.float32(np.abs(qr).max()) / np.float32(2688)


def test_naive_with_rotation(orc):
    """The pages' "8-bit FlashAttention-4 + QK Hadamard" baseline: the naive
    preparation with the rotation, K rotated in sequence order without
    centring."""
    N = 260
    q, k, v = synth.make_qkv(1, 1, N, 128, 8, 63)
    p = orc.prepare8(q[0, 0], k[0, 0], v[0, 0], 8, 2, 63, naive=True, hadamard=True)
    ph = orc.prepare8(q[0, 0], k[0, 0], v[0, 0], 8, 2, 63, hadamard=True)
    pn = orc.prepare8(q[0, 0], k[0, 0], v[0, 0], 8, 2, 63, naive=True)
    assert np.array_equal(p["qhat"], ph["qhat"]) and np.array_equal(p["rhatT"], pn["rhatT"])
    kr = orc.hadamard128(_f(k[0, 0]).astype(np.float32))
    for j in range(p["sk"].size):
        blk = kr[j * 128:(j + 1) * 128]
        s = np.float32(np.abs(blk).max()) / np.float32(448)
        assert p["sk"][j] == s
        assert np.array_equal(p["khat"][j * 128:j * 128 + len(blk)], _e4m3(blk / s))
