"""Pins of the oracle's ExpCast-FP8 (paper §3.3 Eq 7, Appx C/D) against the
numbers the paper prints and against torch's exp-then-cast (no GPU)."""
import math

import numpy as np
import torch

from conftest import read_golden

G = read_golden("expcast_constants.txt")


def _e4m3_cast_torch(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy().astype(np.int32)


def _decode(codes):
    c = torch.from_numpy(np.asarray(codes, np.uint8))
    return c.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_worked_example(orc):
    g = read_golden("expcast_worked_example.txt")
    u = float(g["u"])
    beta = float(g["beta"])
    assert abs(8 * (u + 8) + 56 + beta - float(g["eq7_value"])) < 1e-9
    c = orc.expcast_code(u)
    assert c == int(g["byte"]) == 8 * int(g["byte_exponent_field"]) + int(g["byte_mantissa_field"])
    assert _decode([c])[0] == float(g["decoded_value"])
    assert abs(2 ** (u + 8) - float(g["exp_path_value"])) < 0.05
    # the conventional path (exp, then an E4M3 cast) writes the same byte
    assert _e4m3_cast_torch([2 ** (u + 8)])[0] == c


def test_agreement_over_a_doubling(orc):
    # Fig 5: same byte as exp-then-cast on 79.6% of a doubling, else 1 code.
    u = np.linspace(-1.0, 0.0, 200001)[:-1]
    ours = orc.expcast_codes(u)
    ref = _e4m3_cast_torch(np.exp2(u + 8.0))
    same = np.mean(ours == ref)
    assert abs(same - float(G["agreement"])) < 0.001, same
    assert np.max(np.abs(ours - ref)) == int(G["max_code_gap"])
    # "every unit interval of z looks the same": a deeper doubling agrees too
    u2 = u - 7.0
    same2 = np.mean(orc.expcast_codes(u2) == _e4m3_cast_torch(np.exp2(u2 + 8.0)))
    assert abs(same2 - same) < 1e-9


def test_ratio_range_eq11(orc):
    u = np.linspace(-3.0, 0.0, 300001)
    ratio = _decode(orc.expcast_codes(u)) / np.exp2(u + 8.0)
    lo, hi = float(G["ratio_min"]), float(G["ratio_max"])
    assert ratio.min() >= lo - 1e-4 and ratio.max() <= hi + 1e-4
    assert ratio.min() <= lo + 1e-3 and ratio.max() >= hi - 1e-3
    assert np.max(np.abs(ratio - 1)) <= float(G["max_rel_error"]) + 1e-4


def test_mitchell_constants():
    # Eq 9: e(f) = 8 [f - (2^f - 1)] on [0, 1): range [0, 0.6886]; minimax shift -0.3443
    f = np.linspace(0, 1, 1000001)
    e = 8 * (f - (np.exp2(f) - 1))
    assert abs(e.min()) < 1e-12 and abs(e.max() - float(G["e_max"])) < 1e-4
    assert abs(-e.max() / 2 - float(G["beta_minimax"])) < 1e-4
    a, b = float(G["ratio_min"]), float(G["ratio_max"])
    assert (math.sqrt(b) - math.sqrt(a)) / (math.sqrt(b) + math.sqrt(a)) < float(G["tv_bound"])


def _row_probs(orc, u):
    p = np.exp2(u)
    p /= p.sum()
    w = _decode(orc.expcast_codes(u))
    return p, w / w.sum()


def test_tv_bound_random_rows(orc):
    rng = np.random.default_rng(4)
    bound = float(G["tv_bound"])
    for _ in range(300):
        n = int(rng.integers(2, 600))
        u = -rng.uniform(0, 13.9, n)
        u[rng.integers(n)] = 0.0                 # the row maximum sits at u = 0
        p, ph = _row_probs(orc, u)
        assert 0.5 * np.abs(p - ph).sum() < bound


def test_tv_bound_adversarial_row(orc):
    # Eq 12: the worst row puts mass q at the largest ratio and the rest at the
    # smallest; build it from the extreme cells found on a grid.
    f = np.linspace(-1.0, 0.0, 100001)[:-1]
    ratio = _decode(orc.expcast_codes(f)) / np.exp2(f + 8.0)
    u_hi, u_lo = f[np.argmax(ratio)], f[np.argmin(ratio)]
    a, b = ratio.min(), ratio.max()
    q = math.sqrt(a) / (math.sqrt(a) + math.sqrt(b))
    n = 1000
    n_hi = int(round(q * n))
    u = np.concatenate([np.full(n_hi, u_hi), np.full(n - n_hi, u_lo)])
    p, ph = _row_probs(orc, u)
    tv = 0.5 * np.abs(p - ph).sum()
    assert 0.03 < tv < float(G["tv_bound"])


def test_tv_bound_with_underflow_tail(orc):
    rng = np.random.default_rng(5)
    for _ in range(200):
        n = int(rng.integers(2, 400))
        u = -rng.exponential(6.0, n)
        u[0] = 0.0
        p, ph = _row_probs(orc, u)
        tail = u < float(G["u_normal_min"])
        tau = max(p[tail].sum(), ph[tail].sum())
        assert 0.5 * np.abs(p - ph).sum() < float(G["tv_bound"]) + tau + 1e-12


def test_output_bound_eq15(orc):
    rng = np.random.default_rng(6)
    for _ in range(100):
        n, d = int(rng.integers(2, 300)), 16
        u = -rng.uniform(0, 16, n)
        u[0] = 0.0
        V = rng.standard_normal((n, d)) * rng.uniform(0.1, 10)
        p, ph = _row_probs(orc, u)
        tail = u < -14
        tau = max(p[tail].sum(), ph[tail].sum())
        diam = max(np.linalg.norm(V[a] - V[b]) for a in range(n) for b in range(a + 1, n)) \
            if n < 60 else np.linalg.norm(V.max(0) - V.min(0))
        assert np.linalg.norm(ph @ V - p @ V) <= (float(G["tv_bound"]) + tau) * diam + 1e-12


def test_single_fma_form_matches_eq7(orc):
    # The fp32 form clip(RNE(fmaf(a, acc, b))) with b = 120 + beta - M is Eq 7
    # with u = (a acc - M) / 8, away from rounding ties.
    rng = np.random.default_rng(7)
    n = 20000
    a = rng.uniform(0.01, 2.0, n).astype(np.float32)
    acc = rng.uniform(-300, 300, n).astype(np.float32)
    M = (a.astype(np.float64) * 300).astype(np.float32)
    b = (np.float32(119.65) - M).astype(np.float32)
    ours = orc.expcast_f32(acc, a, b).astype(np.int32)
    u = (a.astype(np.float64) * acc - M.astype(np.float64)) / 8.0
    ref = orc.expcast_codes(u)
    v = 8 * (u + 8) + 56 - 0.35
    away = np.abs(v - np.floor(v) - 0.5) > 1e-3
    assert np.array_equal(ours[away], ref[away])
    assert np.max(np.abs(ours - ref)) <= 1
    assert orc.expcast_f32([np.nan, -np.inf, 0.0], [1, 1, 1], [0, 0, 119.65]).tolist() == [0, 0, 120]
