"""Pins of the oracle's attention (paper §3.1 Eq 1, §3.2 Eq 3 and Eq 6,
§3.3 Eq 7) against numpy's softmax, exact identities and bounds (no GPU)."""
import numpy as np
import pytest
import torch

import synth


def _f(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16) \
        .to(torch.float64).numpy()


def _e4m3_val(c):
    return torch.from_numpy(np.ascontiguousarray(c, np.uint8)).view(torch.float8_e4m3fn) \
        .to(torch.float64).numpy()


def _softmax_attention(q, k, v):
    s = q @ k.T / np.sqrt(q.shape[1])
    s -= s.max(1, keepdims=True)
    p = np.exp(s)
    return (p / p.sum(1, keepdims=True)) @ v


@pytest.fixture(scope="module")
def small():
    q, k, v = synth.make_qkv(1, 1, 333, 128, 6, 2024)   # 333 keys: three tiles, ragged
    return q[0, 0], k[0, 0], v[0, 0]


def test_exact_matches_numpy_softmax(orc, small):
    q, k, v = small
    rows = np.arange(0, 333, 7)
    ours = orc.attention_exact(q, k, v, rows)
    ref = _softmax_attention(_f(q)[rows], _f(k), _f(v))
    assert np.allclose(ours, ref, rtol=1e-12, atol=1e-12)


def test_permutation_invariance_eq3(orc, small):
    q, k, v = small
    perm = np.random.default_rng(1).permutation(333)
    rows = np.arange(333)
    a = orc.attention_exact(q, k, v, rows)
    b = orc.attention_exact(q, k[perm], v[perm], rows)
    assert np.max(np.abs(a - b)) < 1e-12


@pytest.mark.parametrize("Bv", [128, 16, 100 - 36])
def test_mean_restoration_eq6(orc, small, Bv):
    """Eq 6 with exact exp and unquantised residual equals Eq 1 exactly."""
    q, k, v = small
    N = 333
    perm = np.random.default_rng(2).permutation(N)
    kp, vp = _f(k)[perm], _f(v)[perm]
    nb = (N + Bv - 1) // Bv
    mu = np.stack([vp[j * Bv:(j + 1) * Bv].mean(0) for j in range(nb)])
    r = vp - np.repeat(mu, Bv, 0)[:N]
    rows = np.arange(0, N, 5)
    got = orc.attention_recurrence(_f(q), kp, r, mu, Bv, 0, rows)
    ref = orc.attention_exact(q, k, v, rows)
    assert np.max(np.abs(got - ref)) < 1e-12


def test_expcast_recurrence_output_bound(orc, small):
    """Prop 3.1 / Eq 15 on the running-max recurrence: rows whose scores stay in
    the normal range move by at most 3.64% of diam(V')."""
    q, k, v = small
    qf, kf, vf = _f(q) * 0.25, _f(k), _f(v)     # mild scores: no underflow tail
    N, Bv = 333, 128
    mu = np.zeros(((N + Bv - 1) // Bv, 128))
    rows = np.arange(N)
    exact = orc.attention_recurrence(qf, kf, vf, mu, Bv, 0, rows)
    fast = orc.attention_recurrence(qf, kf, vf, mu, Bv, 1, rows)
    s = qf @ kf.T / np.sqrt(128) * np.log2(np.e)
    assert np.all(s - s.max(1, keepdims=True) >= -14)
    lo, hi = vf.min(0), vf.max(0)
    diam = np.linalg.norm(hi - lo)           # >= the largest row distance
    err = np.linalg.norm(fast - exact, axis=1)
    assert np.all(err <= 0.0364 * diam)
    assert err.max() > 0                     # ExpCast does perturb


@pytest.fixture(scope="module")
def prep8(orc):
    q, k, v = synth.make_qkv(1, 1, 700, 128, 8, 99)
    p = orc.prepare8(q[0, 0], k[0, 0], v[0, 0], 8, 5, 99)
    return q[0, 0], k[0, 0], v[0, 0], p


def test_attention8_is_the_recurrence_on_dequantised_operands(orc, prep8):
    q, k, v, p = prep8
    N, d = 700, 128
    qd = _e4m3_val(p["qhat"][:N]) * np.repeat(p["sq"], 128)[:N, None]
    kd = _e4m3_val(p["khat"][:N]) * np.repeat(p["sk"], 128)[:N, None]
    rd = _e4m3_val(p["rhatT"][:, :N]).T * p["sv"][None, :]
    mu = _f(p["mu"])
    rows = np.arange(0, N, 3)
    ref = orc.attention_recurrence(qd, kd, rd, mu, 128, 1, rows)
    bits, got = orc.attention8(p, rows)
    # mu enters attention8 as fp32(mu / sv) * sv: a relative 2^-24 rounding
    assert np.max(np.abs(got - ref)) < 1e-6 * np.max(np.abs(ref))
    gotb = _f(bits)
    assert np.all(np.abs(gotb - got) <= np.abs(got) * 2.0 ** -8)


def test_plain_attention8_is_the_recurrence_without_means(orc, prep8):
    """After the grouping window the value operand is V[pi] itself: attention8
    on the plain preparation is the ExpCast recurrence on the dequantised
    operands with every mean zero."""
    q, k, v, p0 = prep8
    N = 700
    p = orc.prepare8(q, k, v, 8, 5, 99, perm=p0["perm"], plain=True)
    qd = _e4m3_val(p["qhat"][:N]) * np.repeat(p["sq"], 128)[:N, None]
    kd = _e4m3_val(p["khat"][:N]) * np.repeat(p["sk"], 128)[:N, None]
    rd = _e4m3_val(p["rhatT"][:, :N]).T * p["sv"][None, :]
    rows = np.arange(1, N, 5)
    ref = orc.attention_recurrence(qd, kd, rd, np.zeros_like(_f(p["mu"])), 128, 1, rows)
    _, got = orc.attention8(p, rows)
    assert np.max(np.abs(got - ref)) < 1e-9 * np.max(np.abs(ref))


def _e4m3(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def test_recurrence_exp_then_cast_single_tile(orc, small):
    """pmode 2 on one tile (every u relative to the row maximum): the weights
    are torch's E4M3 cast of 2^(u + 8), and the output their weighted mean."""
    q, k, v = (_f(x) for x in small)
    N, d = k.shape
    rows = np.arange(0, N, 7)
    got = orc.attention_recurrence(q, k, v, np.zeros((1, d)), 512, 2, rows)
    t = q[rows] @ k.T / np.sqrt(d) * np.log2(np.e)
    u = t - t.max(1, keepdims=True)
    w = _e4m3_val(_e4m3(np.exp2(u + 8.0)))
    want = (w @ v) / w.sum(1, keepdims=True)
    assert np.max(np.abs(got - want)) < 1e-9 * np.max(np.abs(want))


def test_attention8_exp_is_the_recurrence_on_dequantised_operands(orc, prep8):
    q, k, v, p = prep8
    N = 700
    qd = _e4m3_val(p["qhat"][:N]) * np.repeat(p["sq"], 128)[:N, None]
    kd = _e4m3_val(p["khat"][:N]) * np.repeat(p["sk"], 128)[:N, None]
    rd = _e4m3_val(p["rhatT"][:, :N]).T * p["sv"][None, :]
    rows = np.arange(2, N, 7)
    ref = orc.attention_recurrence(qd, kd, rd, _f(p["mu"]), 128, 2, rows)
    _, got = orc.attention8(p, rows, expcast=False)
    assert np.max(np.abs(got - ref)) < 1e-6 * np.max(np.abs(ref))
    _, got_ec = orc.attention8(p, rows)
    assert np.max(np.abs(got_ec - got)) > 0          # the two byte rules differ


def test_naive_preparation(orc):
    """Naive FP8: sequence order, no key centring, no demeaning; Q and K per
    128-token block, V per channel (torch E4M3 casts of the same divisions)."""
    N = 600
    q, k, v = synth.make_qkv(1, 1, N, 128, 8, 77)
    p = orc.prepare8(q[0, 0], k[0, 0], v[0, 0], 8, 2, 77, naive=True)
    ref = orc.prepare8(q[0, 0], k[0, 0], v[0, 0], 8, 2, 77)
    assert np.array_equal(p["perm"], np.arange(N)) and np.all(p["labels"] == -1)
    assert np.all(p["kbar"] == 0) and np.all(p["mu"] == 0) and np.all(p["mutilde"] == 0)
    assert np.array_equal(p["qhat"], ref["qhat"]) and np.array_equal(p["sq"], ref["sq"])
    kf = _f(k[0, 0]).astype(np.float32)
    for j in range(p["sk"].size):
        blk = kf[j * 128:(j + 1) * 128]
        s = np.float32(np.abs(blk).max()) / np.float32(448)
        assert p["sk"][j] == s
        assert np.array_equal(p["khat"][j * 128:j * 128 + len(blk)], _e4m3(blk / s))
    vf = _f(v[0, 0]).astype(np.float32)
    sv = np.abs(vf).max(0).astype(np.float32) / np.float32(448)
    assert np.array_equal(p["sv"], sv)
    assert np.array_equal(p["rhatT"][:, :N], _e4m3((vf / sv).T))


def test_attention8_value_path_with_flat_scores(orc):
    """q = 0: every score is 0, every byte is 120 (value 256), so the output is
    the mean of the dequantised residual plus the restored block means."""
    N = 500
    q, k, v = synth.make_qkv(1, 1, N, 128, 8, 3)
    q0 = np.zeros_like(q[0, 0])
    p = orc.prepare8(q0, k[0, 0], v[0, 0], 8, 3, 3)
    _, got = orc.attention8(p, np.arange(0, N, 50))
    vf = _f(v[0, 0])
    R = vf[p["perm"]] - np.repeat(_f(p["mu"]), 128, 0)[:N]
    tol = np.abs(R).mean(0) / 16 + p["sv"] * 2.0 ** -9
    assert np.all(np.abs(got - vf.mean(0)[None, :]) <= tol[None, :] + 1e-9)


def test_attention4_value_path_with_flat_scores(orc):
    N = 500
    q, k, v = synth.make_qkv(1, 1, N, 128, 8, 4)
    q0 = np.zeros_like(q[0, 0])
    p = orc.prepare4(q0, k[0, 0], v[0, 0], 8, 3, 4)
    _, got = orc.attention4(p, np.arange(0, N, 50))
    vf = _f(v[0, 0])
    gr = float(p["gr"][0])
    scale = np.repeat(_e4m3_val(p["r4s"]), 16, 1)[:, :N] * gr        # per element step unit
    tol = scale.mean(1)                                               # one E2M1 unit
    assert np.all(np.abs(got - vf.mean(0)[None, :]) <= tol[None, :] + 1e-9)


def test_quantised_attention_against_exact_report(orc, prep8):
    q, k, v, p = prep8
    rows = np.arange(0, 700, 11)
    ex = orc.attention_exact(q, k, v, rows)
    _, o8 = orc.attention8(p, rows)
    p4 = orc.prepare4(q, k, v, 8, 5, 99)
    _, o4 = orc.attention4(p4, rows)
    e8 = np.linalg.norm(o8 - ex) / np.linalg.norm(ex)
    e4 = np.linalg.norm(o4 - ex) / np.linalg.norm(ex)
    print(f"rel L2 vs exact fp64: 8-bit {e8:.4f}, 4-bit {e4:.4f}")
    assert e8 < 0.1 and e4 < 0.4


# E2M1 from its definition (1 sign, 2 exponent, 1 mantissa bit, no inf or NaN):
# the eight magnitudes, code 8 + c the negative of code c
_E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e2m1_val(c):
    c = np.asarray(c, np.int64)
    return np.where(c & 8, -1.0, 1.0) * _E2M1[c & 7]


def _e2m1_rne(x):
    """Round non-negative fp32 values to E2M1 magnitudes, nearest with ties to
    the even code, saturating at 6."""
    x = np.asarray(x, np.float64)
    codes = np.zeros(x.shape, np.int64)
    for i in range(len(_E2M1) - 1):  # choose between code i and i + 1 on [E2M1[i], E2M1[i+1]]
        lo, hi = _E2M1[i], _E2M1[i + 1]
        mid = (lo + hi) / 2
        up = (x > mid) | ((x == mid) & (i % 2 == 1))
        codes = np.where((x >= lo) & (x <= hi), np.where(up, i + 1, i), codes)
    return np.where(x > 6.0, 7, codes)


@pytest.mark.parametrize("N", [100, 700])
def test_attention4_single_pass_when_block0_holds_every_row_max(orc, N):
    """When key block 0 holds each sampled row's largest score, the running
    maximum of the online recurrence never rises after block 0 (alpha = 1
    from then on), so the 4-bit output must equal one pass over all keys at
    the row's global maximum: p = 2^(t - max), P = NVFP4 of 2688 p per 16 keys
    (UE4M3 scale of the block maximum / 6, E2M1 codes of the quotients),
    O = (sum_k Pq_k R_k + sum_j r_j mu_j) / sum_k p_k, with r_j and the
    denominator from the unquantised p (Eq 6 with Appx B's 4-bit operands).
    The formats are restated here (E2M1 table, UE4M3 through torch's
    float8_e4m3fn); the permutation is chosen so that block 0 holds the
    maxima (a K' row's codes do not depend on the order)."""
    q, k, v = synth.make_qkv(1, 1, N, 128, 8, 77)
    q, k, v = q[0, 0], k[0, 0], v[0, 0]
    rows = np.arange(0, N, 11)
    log2e = 1.4426950408889634

    def scores(p):
        d = 128
        qd = _e2m1_val(p["q4"][rows]) * np.repeat(_e4m3_val(p["q4s"][rows]), 16, 1) * \
            np.float64(p["gq"][0])
        kd = _e2m1_val(p["k4"][:N]) * np.repeat(_e4m3_val(p["k4s"][:N]), 16, 1) * \
            np.float64(p["gk"][0])
        return qd @ kd.T * (1.0 / np.sqrt(d)) * log2e

    p0 = orc.prepare4(q, k, v, 8, 3, 77)
    best = p0["perm"][np.argmax(scores(p0), 1)]          # the token holding each row's max
    first = list(dict.fromkeys(best.tolist()))
    assert len(first) <= 128
    perm = np.array(first + [t for t in p0["perm"].tolist() if t not in set(first)], np.int32)
    p = orc.prepare4(q, k, v, 8, 3, 77, perm=perm)
    t = scores(p)
    assert np.all(np.argmax(t, 1) < 128)
    m = t.max(1, keepdims=True)
    pr = np.exp2(t - m)                                   # unquantised, max 1
    npad = (N + 15) // 16 * 16
    pp = np.zeros((len(rows), npad))
    pp[:, :N] = pr
    blocks = pp.reshape(len(rows), -1, 16)
    amax = (2688.0 * blocks).max(2)
    scv = _e4m3_val(torch.from_numpy((amax / 6.0).astype(np.float32)).to(torch.float8_e4m3fn)
                    .view(torch.uint8).numpy())
    with np.errstate(divide="ignore", invalid="ignore"):
        x = (2688.0 * blocks / scv[:, :, None]).astype(np.float32)
    pq = np.where(scv[:, :, None] > 0, _E2M1[_e2m1_rne(x)] * scv[:, :, None] / 2688.0, 0.0)
    pq = pq.reshape(len(rows), npad)[:, :N]
    rd = (_e2m1_val(p["r4T"][:, :N]) * np.repeat(_e4m3_val(p["r4s"]), 16, 1)[:, :N] *
          np.float64(p["gr"][0])).T
    mu = _f(p["mu"])                                      # [nb][d]
    nb = mu.shape[0]
    rj = np.stack([pr[:, j * 128:(j + 1) * 128].sum(1) for j in range(nb)], 1)
    want = (pq @ rd + rj @ mu) / pr.sum(1, keepdims=True)
    _, got = orc.attention4(p, rows)
    assert np.max(np.abs(got - want)) <= 1e-9 * np.max(np.abs(want))


def test_attention4_unrolled_recurrence(orc):
    """The general case: unrolling the online rescaling (the alpha factors
    telescope), block j's probabilities are taken, and quantised, at the prefix
    maximum m_j = max of the scores of blocks 0..j, and enter the output with
    weight 2^(m_j - M), M the row maximum:
    O = sum_j 2^(m_j - M) (Pq_j R_j + r_j mu_j) / sum_j 2^(m_j - M) r_j."""
    N = 900
    q, k, v = synth.make_qkv(1, 1, N, 128, 8, 91)
    p = orc.prepare4(q[0, 0], k[0, 0], v[0, 0], 8, 3, 91)
    rows = np.arange(0, N, 7)
    log2e = 1.4426950408889634
    qd = _e2m1_val(p["q4"][rows]) * np.repeat(_e4m3_val(p["q4s"][rows]), 16, 1) * \
        np.float64(p["gq"][0])
    kd = _e2m1_val(p["k4"][:N]) * np.repeat(_e4m3_val(p["k4s"][:N]), 16, 1) * \
        np.float64(p["gk"][0])
    t = qd @ kd.T * (1.0 / np.sqrt(128)) * log2e
    rd = (_e2m1_val(p["r4T"][:, :N]) * np.repeat(_e4m3_val(p["r4s"]), 16, 1)[:, :N] *
          np.float64(p["gr"][0])).T
    mu = _f(p["mu"])
    nb = mu.shape[0]
    bmax = np.stack([t[:, j * 128:(j + 1) * 128].max(1) for j in range(nb)], 1)
    mj = np.maximum.accumulate(bmax, 1)                     # running maximum after block j
    M = mj[:, -1:]
    num = np.zeros((len(rows), 128))
    den = np.zeros((len(rows), 1))
    rises = 0
    for j in range(nb):
        k0, k1 = j * 128, min(N, (j + 1) * 128)
        pj = np.exp2(t[:, k0:k1] - mj[:, j:j + 1])
        pad = np.zeros((len(rows), 128))
        pad[:, :k1 - k0] = pj
        blocks = pad.reshape(len(rows), 8, 16)
        amax = (2688.0 * blocks).max(2)
        scv = _e4m3_val(torch.from_numpy((amax / 6.0).astype(np.float32)).to(torch.float8_e4m3fn)
                        .view(torch.uint8).numpy())
        with np.errstate(divide="ignore", invalid="ignore"):
            x = (2688.0 * blocks / scv[:, :, None]).astype(np.float32)
        pq = np.where(scv[:, :, None] > 0, _E2M1[_e2m1_rne(x)] * scv[:, :, None] / 2688.0, 0.0)
        pq = pq.reshape(len(rows), 128)[:, :k1 - k0]
        w = np.exp2(mj[:, j:j + 1] - M)
        rj = pj.sum(1, keepdims=True)
        num += w * (pq @ rd[k0:k1] + rj * mu[j][None, :])
        den += w * rj
        if j > 0:
            rises += int(np.sum(mj[:, j] > mj[:, j - 1]))
    assert rises > 0                                         # the rescaling path is exercised
    want = num / den
    _, got = orc.attention4(p, rows)
    assert np.max(np.abs(got - want)) <= 1e-9 * np.max(np.abs(want))


@pytest.mark.parametrize("expcast", [True, False])
def test_attention8_unrolled_recurrence(orc, expcast):
    """The 8-bit recurrence unrolled, as for 4 bits: block j's probability
    bytes are taken at its prefix maximum m_j (Eq 7's ExpCast code
    clip_[0,120](RNE(8(u+8)+56+beta)), beta = -0.35, or the E4M3 cast of
    2^(u+8)), and block j enters with weight 2^(m_j - M):
    O = sv * sum_j 2^(m_j - M) (P_j R^_j + r_j mutilde_j) / sum_j 2^(m_j - M) r_j.
    The scores are exact (products of E4M3 codes summed in fp64, then the
    block scales), so the bytes match the oracle's one for one."""
    N = 900
    q, k, v = synth.make_qkv(1, 1, N, 128, 8, 92)
    p = orc.prepare8(q[0, 0], k[0, 0], v[0, 0], 8, 3, 92)
    rows = np.arange(0, N, 7)
    log2e, inv = 1.4426950408889634, 1.0 / np.sqrt(128.0)
    qd = _e4m3_val(p["qhat"][rows])
    kd = _e4m3_val(p["khat"][:N])
    rd = _e4m3_val(p["rhatT"][:, :N]).T
    nb = (N + 127) // 128
    acc = qd @ kd.T                                          # exact: integers times powers of two
    sq = p["sq"][rows // 128].astype(np.float64)[:, None]
    sk = np.repeat(p["sk"].astype(np.float64), 128)[:N][None, :]
    t = acc * sq * sk * inv * log2e
    bmax = np.stack([t[:, j * 128:(j + 1) * 128].max(1) for j in range(nb)], 1)
    mj = np.maximum.accumulate(bmax, 1)
    M = mj[:, -1:]
    num = np.zeros((len(rows), 128))
    den = np.zeros((len(rows), 1))
    mt = p["mutilde"].astype(np.float64)
    for j in range(nb):
        k0, k1 = j * 128, min(N, (j + 1) * 128)
        u = t[:, k0:k1] - mj[:, j:j + 1]
        if expcast:
            code = np.clip(np.rint(8.0 * (u + 8.0) + 56.0 + (-0.35)), 0, 120).astype(np.uint8)
            w8 = _e4m3_val(code)
        else:
            w8 = _e4m3_val(torch.from_numpy(np.exp2(u + 8.0).astype(np.float32))
                           .to(torch.float8_e4m3fn).view(torch.uint8).numpy())
        w = np.exp2(mj[:, j:j + 1] - M)
        rj = w8.sum(1, keepdims=True)
        num += w * (w8 @ rd[k0:k1] + rj * mt[j][None, :])
        den += w * rj
    want = p["sv"].astype(np.float64)[None, :] * num / den
    _, got = orc.attention8(p, rows, expcast=expcast)
    assert np.max(np.abs(got - want)) <= 1e-9 * np.max(np.abs(want))
