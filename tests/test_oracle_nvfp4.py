"""Code-for-code pins of the oracle's NVFP4 quantisers (paper Appx A "Scope of
ExpCast-FP8" and Appx B: E2M1 elements under one E4M3 microscale per 16
elements along the product's reduction dimension, one fp32 global scale per
head and operand).  No GPU.

The quantiser is restated here in numpy from its definitions, independently of
``oracle.cpp``:
  - global scale   g = fp32(amax) / 2688 (1 when amax = 0), 2688 = 448 x 6;
  - block scale    UE4M3_RNE(fp32(amax16) / fp32(6 g)), through torch's
                   float8_e4m3fn cast;
  - element code   E2M1_RNE(x / fp32(scale g)): the nearest entry of the E2M1
                   value table (``golden/e2m1_values.txt``), ties to the even
                   code, saturating at 6, sign bit 8 kept; a block whose scale
                   rounds to 0 gets codes 0.
Every byte of the plain, rotated and after-the-window preparations must match.
Constructed blocks put the block scale on UE4M3 rounding midpoints, the element
quotients on E2M1 midpoints, whole blocks at zero, and block maxima where
(amax16 / 6) / g and amax16 / (6 g) round to different scale codes; the test
shows the misread formulas give other bytes on those blocks."""
import numpy as np
import pytest
import torch

import synth
from conftest import read_golden

E2M1 = np.array([float(x) for x in read_golden("e2m1_values.txt")["values"].split(",")])


def _f32(bits):
    """bf16 bit patterns -> float32 values (exact)."""
    return (np.ascontiguousarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def ue4m3(x):
    x = np.asarray(x, np.float32)
    assert np.all(x >= 0) and np.all(x < 464), "block scales stay below the E4M3 overflow"
    return torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def ue4m3_value(c):
    return torch.from_numpy(np.asarray(c, np.uint8)).view(torch.float8_e4m3fn) \
        .to(torch.float32).numpy()


def e2m1_rne(x, toward_zero=False):
    """E2M1 code of each fp32 value: the nearest table value by brute force over
    all eight, ties to the even code (toward_zero: the misreading that truncates)."""
    x = np.asarray(x, np.float32)
    a = np.abs(x.astype(np.float64))
    dist = np.abs(a[..., None] - E2M1)
    if toward_zero:
        code = np.sum(E2M1 <= a[..., None], -1) - 1
    else:
        best = dist.min(-1, keepdims=True)
        tie_even = (dist == best) & (np.arange(8) % 2 == 0)
        code = np.where(tie_even.any(-1), np.argmax(tie_even, -1), np.argmin(dist, -1))
    return (code + 8 * np.signbit(x)).astype(np.uint8)


def global_scale(x):
    amax = np.float32(np.abs(np.asarray(x, np.float32)).max())
    return np.float32(amax / np.float32(2688)) if amax > 0 else np.float32(1)


def nvfp4(x, g, scale_rule="spec", toward_zero=False):
    """x: fp32 [rows, n] with blocks of 16 along the last axis.  Returns
    (codes [rows, n], scales [rows, n/16])."""
    x = np.asarray(x, np.float32)
    blk = x.reshape(x.shape[0], -1, 16)
    amax = np.abs(blk).max(-1)
    g = np.float32(g)
    if scale_rule == "spec":
        q = amax / np.float32(np.float32(6) * g)
    else:                                         # the misreading (amax16 / 6) / g
        q = (amax / np.float32(6)) / g
    sc = ue4m3(q.astype(np.float32))
    step = (ue4m3_value(sc) * g).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        quot = (blk / step[..., None]).astype(np.float32)
    codes = np.where(step[..., None] > 0, e2m1_rne(quot, toward_zero), 0).astype(np.uint8)
    return codes.reshape(x.shape), sc


# ------------------------------------------------------------------ helpers
def _operands(orc, q, k, v, p, plain=False, hadamard=False):
    """The fp32 operands the quantisers see: Q, K' = K[pi] - kbar (both rotated
    when asked) and R^T = (V[pi] - mu)^T, from the oracle's own pi, kbar and mu
    (each pinned by the V-Smooth tests)."""
    N = q.shape[0]
    nb = (N + 127) // 128
    Q = np.zeros((nb * 128, 128), np.float32)
    Q[:N] = _f32(q)
    Kp = np.zeros_like(Q)
    Kp[:N] = _f32(k)[p["perm"]] - _f32(p["kbar"])
    if hadamard:
        Q[:N] = orc.hadamard128(Q[:N])
        Kp[:N] = orc.hadamard128(Kp[:N])
    R = np.zeros_like(Q)
    mu = np.repeat(_f32(p["mu"]), 128, 0)[:N]
    if plain:
        assert np.all(p["mu"] == 0)
    R[:N] = _f32(v)[p["perm"]] - mu
    return Q, Kp, R


def _check_prepare4(orc, q, k, v, p, **kw):
    Q, Kp, R = _operands(orc, q, k, v, p, **kw)
    N = q.shape[0]
    for name, x, codes, scales, gname in (("Q", Q, "q4", "q4s", "gq"),
                                          ("K'", Kp, "k4", "k4s", "gk")):
        g = global_scale(x[:N])
        assert p[gname][0] == g, f"{name}: global scale"
        c, s = nvfp4(x, g)
        assert np.array_equal(p[codes], c), f"{name}: {np.sum(p[codes] != c)} codes differ"
        assert np.array_equal(p[scales], s), f"{name}: {np.sum(p[scales] != s)} scales differ"
    g = global_scale(R[:N])
    assert p["gr"][0] == g
    c, s = nvfp4(R.T, g)                          # blocks of 16 tokens per channel
    assert np.array_equal(p["r4T"], c), f"R: {np.sum(p['r4T'] != c)} codes differ"
    assert np.array_equal(p["r4s"], s), f"R: {np.sum(p['r4s'] != s)} scales differ"


# ------------------------------------------------------------------ tests
def test_restatement_e2m1_table():
    """The restated E2M1 rounding on the table's own values, midpoints and
    beyond the top (no oracle involved)."""
    x = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, 7, 100,
                  -0.25, -5, -0.1, 0.2600001], np.float32)
    want = [0, 1, 2, 3, 4, 5, 6, 7, 0, 2, 2, 4, 4, 6, 6, 7, 7, 8, 14, 8, 1]
    assert list(e2m1_rne(x)) == want


@pytest.mark.parametrize("N,seed", [(400, 555), (300, 62), (1000, 701)])
def test_plain_preparation_code_for_code(orc, N, seed):
    q, k, v = synth.make_qkv(1, 1, N, 128, 8, seed)
    p = orc.prepare4(q[0, 0], k[0, 0], v[0, 0], 8, 3, seed)
    _check_prepare4(orc, q[0, 0], k[0, 0], v[0, 0], p)


def test_rotated_preparation_code_for_code(orc):
    N, seed = 300, 62
    q, k, v = synth.make_qkv(1, 1, N, 128, 8, seed)
    p = orc.prepare4(q[0, 0], k[0, 0], v[0, 0], 8, 3, seed, hadamard=True)
    _check_prepare4(orc, q[0, 0], k[0, 0], v[0, 0], p, hadamard=True)


def test_after_window_preparation_code_for_code(orc):
    N, seed = 400, 556
    q, k, v = synth.make_qkv(1, 1, N, 128, 8, seed)
    p0 = orc.prepare4(q[0, 0], k[0, 0], v[0, 0], 8, 3, seed)
    p = orc.prepare4(q[0, 0], k[0, 0], v[0, 0], 8, 3, seed, perm=p0["perm"], plain=True)
    _check_prepare4(orc, q[0, 0], k[0, 0], v[0, 0], p, plain=True)
    pr = orc.prepare4(q[0, 0], k[0, 0], v[0, 0], 8, 3, seed, perm=p0["perm"], plain=True,
                      hadamard=True)
    _check_prepare4(orc, q[0, 0], k[0, 0], v[0, 0], pr, plain=True, hadamard=True)


def _constructed_q():
    """Query rows of two heads' worth of blocks (N = 256), values chosen so that
    every rounding the quantiser does is exercised at a boundary:
      head amax 21 (so g = 21 / 2688 = 2^-7 exactly, 6 g = 3 2^-6):
        row 1: block scales exactly on UE4M3 midpoints (1.0625, 1.1875, 3.125,
               0.5625 x 2^-6, 12.5, 200 in units of 6 g) -> ties to the even
               code;
        row 2: block scale exactly 2 (step 2^-6) and elements on every E2M1
               midpoint (0.25, 0.75, ..., 5 steps), positive and negative;
        rows 3-127: zero -> all-zero blocks (scale 0, codes 0)."""
    q = np.zeros((256, 128), np.float32)
    q[0, 0] = 21.0
    d6 = np.float32(3 * 2.0 ** -6)
    for i, m in enumerate([1.0625, 1.1875, 3.125, 0.5625 * 2.0 ** -6, 12.5, 200.0]):
        q[1, 16 * i] = np.float32(m) * d6
        q[1, 16 * i + 1] = -np.float32(m) * d6 / 2
    step = np.float32(2.0 ** -6)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    q[2, 0] = 6 * step                            # the block maximum: scale 2 exactly
    q[2, 1:8] = mids * step
    q[2, 8:15] = -mids * step
    q[2, 16] = 6 * step
    q[2, 17:24] = (mids + np.float32(0.0625)) * step   # just above each midpoint
    q[128 + 5, 0:16] = np.float32(7.25)           # a second block of Q rows
    return q


def test_constructed_boundaries(orc):
    q32 = _constructed_q()
    assert np.array_equal(_f32(_bf16_bits(q32)), q32), "constructed values are bf16-exact"
    N = q32.shape[0]
    _, k, v = synth.make_qkv(1, 1, N, 128, 8, 77)
    q = _bf16_bits(q32)
    p = orc.prepare4(q, k[0, 0], v[0, 0], 8, 2, 77)
    assert p["gq"][0] == np.float32(2.0 ** -7)
    _check_prepare4(orc, q, k[0, 0], v[0, 0], p)
    # the ties of the block scale: 1.0625 -> 1.0 (0x38), 1.1875 -> 1.25 (0x3A),
    # 3.125 -> 3.0 (0x44), the subnormal tie 0.5625 2^-6 -> 0.5 2^-6 (0x04),
    # 12.5 -> 12 (0x54), 200 -> 192 (0x74)
    assert list(p["q4s"][1, :6]) == [0x38, 0x3A, 0x44, 0x04, 0x54, 0x74]
    assert list(p["q4s"][2, :2]) == [0x40, 0x40]                 # scale 2.0
    # E2M1 ties to even: 0.25->0, 0.75->1.0, 1.25->1.0, 1.75->2, 2.5->2, 3.5->4, 5->4
    assert list(p["q4"][2, :8]) == [7, 0, 2, 2, 4, 4, 6, 6]
    assert list(p["q4"][2, 8:15]) == [8, 10, 10, 12, 12, 14, 14]
    assert list(p["q4"][2, 17:24]) == [1, 2, 3, 4, 5, 6, 7]      # just above: rounds up
    assert np.all(p["q4s"][3:128] == 0) and np.all(p["q4"][3:128] == 0)
    # the misreadings change bytes on these blocks
    c_tz, _ = nvfp4(q32, p["gq"][0], toward_zero=True)
    assert not np.array_equal(c_tz, p["q4"])


def _separating_maxima(A, count):
    """bf16 block maxima a < A for which the two scale formulas, amax16 / (6 g)
    and (amax16 / 6) / g with g = A / 2688, round to different UE4M3 codes."""
    u = np.arange(0x3000, 0x7F80, dtype=np.uint32) << 16
    a = u.view(np.float32)
    a = a[(a <= np.float32(A)) & (a >= np.float32(A) / 400)]
    g = np.float32(np.float32(A) / np.float32(2688))
    good = ue4m3(a / np.float32(np.float32(6) * g))
    bad = ue4m3((a / np.float32(6)) / g)
    return a[good != bad][:count]


def test_scale_formula_separating_blocks(orc):
    """Blocks whose maximum separates amax16 / (6 g) from (amax16 / 6) / g: the
    oracle gives the first formula's scale code on each of them."""
    A = 0.875
    sep = _separating_maxima(A, 12)
    assert sep.size >= 6
    q32 = np.zeros((128, 128), np.float32)
    q32[0, 0] = A
    for i, a in enumerate(sep):
        q32[1 + i // 8, 16 * (i % 8)] = a
        q32[1 + i // 8, 16 * (i % 8) + 3] = -a / 2
    N = 128
    _, k, v = synth.make_qkv(1, 1, N, 128, 8, 78)
    q = _bf16_bits(q32)
    assert np.array_equal(_f32(q), q32)
    p = orc.prepare4(q, k[0, 0], v[0, 0], 8, 2, 78)
    _check_prepare4(orc, q, k[0, 0], v[0, 0], p)
    _, s_bad = nvfp4(q32, p["gq"][0], scale_rule="twice")
    _, s_good = nvfp4(q32, p["gq"][0])
    rows = slice(1, 1 + (sep.size + 7) // 8)
    assert np.sum(s_bad[rows] != s_good[rows]) == sep.size
    assert np.array_equal(p["q4s"][rows], s_good[rows])


def test_zero_key_and_value_blocks(orc):
    """Key channels 0-15 constant (so K' = K[pi] - kbar is exactly zero there:
    every key's first scale block is 0) and value channel 5 zero (every R block
    of that channel is 0)."""
    N = 300
    q, k, v = synth.make_qkv(1, 1, N, 128, 8, 79)
    k = k[0, 0].copy()
    v = v[0, 0].copy()
    k[:, :16] = _bf16_bits(np.full(16, 1.5, np.float32))
    v[:, 5] = 0
    p = orc.prepare4(q[0, 0], k, v, 8, 2, 79)
    assert np.all(_f32(p["kbar"][:16]) == 1.5)
    assert np.all(p["k4s"][:, 0] == 0) and np.all(p["k4"][:, :16] == 0)
    assert np.all(p["r4s"][5] == 0) and np.all(p["r4T"][5] == 0)
    _check_prepare4(orc, q[0, 0], k, v, p)
