"""Pins of the oracle's V-Smooth preprocessing (paper §3.2 Eq 3-5, §3.4,
Appx B) against the pages' toy example, published SplitMix64 values, numpy /
torch library routines and brute force on tiny inputs (no GPU)."""
import numpy as np
import pytest
import torch

import synth
from conftest import read_golden


def _vec(s):
    return np.array([float(x) for x in s.split(",")])


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def _f(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16) \
        .to(torch.float64).numpy()


def _e4m3(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def _e4m3_val(c):
    return torch.from_numpy(np.asarray(c, np.uint8)).view(torch.float8_e4m3fn) \
        .to(torch.float64).numpy()


# ------------------------------------------------------------ toy example
def test_toy_example_permutation_and_means(orc):
    g = read_golden("vsmooth_toy.txt")
    V = np.stack([_vec(g[t]) for t in ("t0", "t1", "t2", "t3")])
    labels = np.array([int(x) for x in g["labels"].split(",")], np.int32)
    pi = np.array([int(x) for x in g["pi"].split(",")], np.int32)
    Bv = int(g["block_rows"])
    assert np.array_equal(orc.stable_argsort(labels, 2), pi)        # pi = argsort(z)
    vb = _bf16(V)
    # sequence order: blocks {t0,t1},{t2,t3}
    mu_seq, _ = orc.block_demean(vb, Bv)
    assert np.allclose(_f(mu_seq[0]), _vec(g["seq_mean_t0t1"]), atol=0.01)
    # sorted order: V' = V[pi], blocks {t0,t2},{t1,t3}
    mu, r = orc.block_demean(vb[pi], Bv)
    assert np.allclose(_f(mu[1]), _vec(g["sorted_mean_t1t3"]), atol=0.01)
    assert np.allclose(r[2], _vec(g["residual_t1"]), atol=0.01)     # row 2 of V' is t1
    assert np.max(np.abs(r[2:4])) <= 0.2 + 0.01


def test_block_mean_is_rounded_mean_and_energy_identity(orc):
    rng = np.random.default_rng(8)
    N, d, Bv = 300, 32, 64          # ragged last block (300 = 4*64 + 44)
    vb = _bf16(rng.standard_normal((N, d)) * 2 + rng.standard_normal(d))
    mu, r = orc.block_demean(vb, Bv)
    V = _f(vb)
    for j in range(mu.shape[0]):
        blk = V[j * Bv:(j + 1) * Bv]
        exact = blk.mean(0)
        m16 = _f(mu[j])
        ulp = np.abs(exact) * 2.0 ** -8 + 1e-30
        assert np.all(np.abs(m16 - exact) <= ulp)                  # bf16 of the mean
        R = r[j * Bv:j * Bv + len(blk)].astype(np.float64)
        assert np.allclose(R, blk - m16, atol=1e-5, rtol=0)          # R = V' - 1 mu^T
        # Eq 5 with the exact mean: ||V'-1c^T||^2 = ||V'-1mu^T||^2 + n ||c-mu||^2
        c = rng.standard_normal(d)
        lhs = np.sum((blk - c) ** 2)
        rhs = np.sum((blk - exact) ** 2) + len(blk) * np.sum((c - exact) ** 2)
        assert abs(lhs - rhs) <= 1e-9 * lhs
        share = len(blk) * np.sum(exact ** 2) / np.sum(blk ** 2)
        assert 0 <= share <= 1
    assert np.all(r[N:] == 0)


# ------------------------------------------------------------ SplitMix64 / k-means
def test_splitmix64_published_values(orc):
    g = read_golden("splitmix64.txt")
    gold = [int(g[f"out{i}"], 16) for i in range(3)]
    N = 2 ** 31 - 1
    # with b=0, h=0, H=1 the generator state is seed ^ 0x9E3779B97F4A7C15
    idx = orc.kmeans_init_indices(0x9E3779B97F4A7C15, 0, 0, 1, N, 3)
    assert list(idx) == [x % N for x in gold]


def test_kmeans_init_distinct(orc):
    idx = orc.kmeans_init_indices(12345, 0, 3, 8, 70, 64)
    assert len(set(idx.tolist())) == 64 and idx.min() >= 0 and idx.max() < 70


def test_stable_argsort_matches_numpy(orc):
    rng = np.random.default_rng(9)
    for k in (1, 3, 64, 200):
        z = rng.integers(0, k, 5000).astype(np.int32)
        assert np.array_equal(orc.stable_argsort(z, k), np.argsort(z, kind="stable"))


def test_k1_gives_identity(orc):
    q, k, v = synth.make_qkv(1, 1, 300, 128, 4, 77)
    x, s, labels, cent = orc.kmeans(v[0, 0], 1, 3, 5)
    assert np.all(labels == 0)
    assert np.array_equal(orc.stable_argsort(labels, 1), np.arange(300))


def test_kmeans_features_match_numpy(orc):
    q, k, v = synth.make_qkv(1, 1, 256, 128, 8, 78)
    x, s, _, _ = orc.kmeans(v[0, 0], 8, 1, 0)
    vf = _f(v[0, 0]).astype(np.float32)
    amax = np.abs(vf).max()
    assert s == np.float32(amax) / np.float32(127)
    ref = np.clip(np.rint(vf / np.float32(s)), -127, 127)
    assert np.array_equal(x.astype(np.float32), ref)


@pytest.mark.parametrize("iters", [1, 2, 5])
def test_kmeans_brute_force_fixed_point(orc, iters):
    """Tiny inputs: the oracle's labels after T+1 iterations are the argmin
    against its centroids after T; those centroids are the round-half-even
    integer means of the iteration-T members (empty clusters keep theirs)."""
    rng = np.random.default_rng(10 + iters)
    N, d, k = 48, 16, 5
    vb = _bf16(rng.standard_normal((N, d)) + np.repeat(rng.standard_normal((4, d)) * 3, 12, 0))
    x, s, lab_t, cent_t = orc.kmeans(vb, k, iters, 99)
    _, _, lab_t1, cent_t1 = orc.kmeans(vb, k, iters + 1, 99)
    X = x.astype(np.int64)
    C = cent_t.astype(np.int64)
    dist = ((X[:, None, :] - C[None, :, :]) ** 2).sum(-1)
    assert np.array_equal(lab_t1, np.argmin(dist, axis=1))          # lowest index on ties
    for m in range(k):
        mem = X[lab_t1 == m]
        if len(mem) == 0:
            assert np.array_equal(cent_t1[m], cent_t[m])
        else:
            assert np.array_equal(cent_t1[m], np.rint(mem.sum(0) / len(mem)).astype(np.int8))
    # the initial centroids are the features of the SplitMix64-drawn tokens
    _, _, lab1, _ = orc.kmeans(vb, k, 1, 99)
    idx = orc.kmeans_init_indices(99, 0, 0, 1, N, k)
    d0 = ((X[:, None, :] - X[idx][None, :, :]) ** 2).sum(-1)
    assert np.array_equal(lab1, np.argmin(d0, axis=1))


def _doubled_amax_copy(vb, base=None):
    """`base` (default vb) with one element set to exactly twice the largest
    |vb|: when every other |element| stays below that, the feature grid scale
    is exactly twice vb's (scaling by 2 commutes with fp32 rounding)."""
    vf = _f(vb)
    amax = np.abs(vf).max()
    v2 = np.array(vb if base is None else base, copy=True)
    assert np.abs(_f(v2)).max() < 2 * amax
    r, c = np.unravel_index(np.argmax(np.abs(vf)), vf.shape)
    v2[(r + 1) % vf.shape[0], c] = _bf16(np.float32(2 * amax))[()]
    return v2


def test_kmeans_warm_moves_centroids_to_the_new_grid(orc):
    """Warm start: when the grid scale doubles exactly, the previous centroids
    land on the new grid at exactly half their integer value, rounded half to
    even (numpy rint); an unchanged grid leaves them untouched."""
    rng = np.random.default_rng(7)
    N, d, k = 96, 16, 6
    vb = _bf16(rng.standard_normal((N, d)) * 2 + np.repeat(rng.standard_normal((6, d)) * 4, 16, 0))
    _, s1, _, c1 = orc.kmeans(vb, k, 4, 5)
    assert (np.abs(c1) % 2 == 1).any()      # odd codes exercise the tie rule
    v2 = _doubled_amax_copy(vb)
    _, s2, lab, c2 = orc.kmeans_warm(v2, c1, s1, 0)
    assert s2 == 2 * s1
    assert np.array_equal(c2, np.rint(c1.astype(np.float64) / 2).astype(np.int8))
    assert (lab == -1).all()
    _, s3, _, c3 = orc.kmeans_warm(vb, c1, s1, 0)
    assert s3 == s1 and np.array_equal(c3, c1)


@pytest.mark.parametrize("iters", [1, 3])
def test_kmeans_warm_brute_force(orc, iters):
    """Warm-started Lloyd: the first assignment is the brute-force argmin
    (lowest index on ties) against the moved centroids; after the last update
    the centroids are the rounded integer means of the last members."""
    rng = np.random.default_rng(20 + iters)
    N, d, k = 64, 16, 5
    vb = _bf16(rng.standard_normal((N, d)) + np.repeat(rng.standard_normal((4, d)) * 3, 16, 0))
    _, s1, _, c1 = orc.kmeans(vb, k, 3, 11)
    v2 = _doubled_amax_copy(vb, _bf16(_f(vb) + rng.standard_normal((N, d)) * 0.5))
    x2, s2, lab1, _ = orc.kmeans_warm(v2, c1, s1, 1)
    assert s2 == 2 * s1
    X = x2.astype(np.int64)
    C0 = np.rint(c1.astype(np.float64) / 2).astype(np.int64)
    assert np.array_equal(lab1, np.argmin(((X[:, None] - C0[None]) ** 2).sum(-1), axis=1))
    _, _, lab_t, cent_t = orc.kmeans_warm(v2, c1, s1, iters)
    _, _, lab_t1, cent_t1 = orc.kmeans_warm(v2, c1, s1, iters + 1)
    C = cent_t.astype(np.int64)
    assert np.array_equal(lab_t1, np.argmin(((X[:, None] - C[None]) ** 2).sum(-1), axis=1))
    for m in range(k):
        mem = X[lab_t1 == m]
        want = cent_t[m] if len(mem) == 0 else np.rint(mem.sum(0) / len(mem)).astype(np.int8)
        assert np.array_equal(cent_t1[m], want)


def test_kmeans_warm_from_a_converged_run_is_a_fixed_point(orc):
    """Started from the centroids of a converged run on the same values, warm
    k-means changes nothing: one iteration returns the same labels and
    centroids."""
    q, k, v = synth.make_qkv(1, 1, 512, 128, 8, 44)
    vb = v[0, 0]
    _, s, lab, cent = orc.kmeans(vb, 8, 40, 3)
    _, _, lab41, cent41 = orc.kmeans(vb, 8, 41, 3)
    assert np.array_equal(lab, lab41) and np.array_equal(cent, cent41)   # converged
    _, s_w, lab_w, cent_w = orc.kmeans_warm(vb, cent, s, 1)
    assert s_w == s and np.array_equal(lab_w, lab) and np.array_equal(cent_w, cent)


def test_kmeans_objective_nonincreasing_and_clusters_found(orc):
    # Lloyd on the integer grid: the rounded mean is the best integer centre per
    # coordinate, so the within-cluster sum of squares never increases.
    B, H, N, C = 1, 1, 2048, 8
    q, k, v = synth.make_qkv(B, H, N, 128, C, 31)
    prev = None
    for it in range(1, 7):
        x, _, labels, cent = orc.kmeans(v[0, 0], 16, it, 1)
        X = x.astype(np.int64)
        obj = int(((X - cent.astype(np.int64)[labels]) ** 2).sum())  # centroids after update it
        if prev is not None:
            assert obj <= prev
        prev = obj
    truth, outl = synth.v_labels(B, H, N, C, 31, 0, 0)
    keep = ~outl
    pure = sum(np.bincount(truth[keep][labels[keep] == m]).max()
               for m in np.unique(labels[keep]))
    assert pure / keep.sum() > 0.8


# ------------------------------------------------------------ quantizers
@pytest.fixture(scope="module")
def head(orc):
    N, d = 1000, 128                                               # ragged: 8 blocks, last has 104
    q, k, v = synth.make_qkv(1, 2, N, d, 16, 4242)
    b, h = 0, 1
    p = orc.prepare8(q[b, h], k[b, h], v[b, h], 16, 4, 4242, b=b, h=h, H=2)
    return dict(q=q[b, h], k=k[b, h], v=v[b, h], p=p, N=N, d=d)


def test_q_quantizer_matches_torch(head):
    p, N, d = head["p"], head["N"], head["d"]
    qf = _f(head["q"]).astype(np.float32)
    for j in range(p["sq"].size):
        blk = qf[j * 128:(j + 1) * 128]
        s = np.float32(np.abs(blk).max()) / np.float32(448)
        assert p["sq"][j] == s
        assert np.array_equal(p["qhat"][j * 128:j * 128 + len(blk)], _e4m3(blk / s))
    assert np.all(p["qhat"][N:] == 0)


def test_k_centering_and_quantizer(head):
    p, N, d = head["p"], head["N"], head["d"]
    kf = _f(head["k"])
    exact_mean = kf.mean(0)
    kbar = _f(p["kbar"])
    assert np.all(np.abs(kbar - exact_mean) <= np.abs(exact_mean) * 2.0 ** -8 + 1e-6)
    kp = (kf[p["perm"]].astype(np.float32) - kbar.astype(np.float32)).astype(np.float32)
    for j in range(p["sk"].size):
        blk = kp[j * 128:(j + 1) * 128]
        s = np.float32(np.abs(blk).max()) / np.float32(448)
        assert p["sk"][j] == s
        assert np.array_equal(p["khat"][j * 128:j * 128 + len(blk)], _e4m3(blk / s))


def test_v_residual_quantizer_and_means(head):
    p, N, d = head["p"], head["N"], head["d"]
    assert np.array_equal(np.sort(p["perm"]), np.arange(N))
    assert np.array_equal(p["perm"], np.argsort(p["labels"], kind="stable"))
    vp = _f(head["v"])[p["perm"]].astype(np.float32)
    mu = _f(p["mu"]).astype(np.float32)
    R = vp - np.repeat(mu, 128, 0)[:N]
    sv = np.abs(R).max(0).astype(np.float32) / np.float32(448)
    assert np.array_equal(p["sv"], sv)
    Npad = p["rhatT"].shape[1]
    assert np.array_equal(p["rhatT"][:, :N], _e4m3((R / sv).T))
    assert np.all(p["rhatT"][:, N:] == 0)
    assert np.array_equal(p["mutilde"], mu / sv)
    # dequantised residual + mean reconstructs V' within half an E4M3 step
    deq = _e4m3_val(p["rhatT"][:, :N]).T * sv + np.repeat(mu, 128, 0)[:N]
    assert np.all(np.abs(deq - vp) <= np.abs(R) / 16 + sv * 2.0 ** -10 + 1e-6)


def test_reuse_permutation(orc, head):
    p2 = orc.prepare8(head["q"], head["k"], head["v"], 16, 4, 4242, perm=head["p"]["perm"])
    for key in ("qhat", "khat", "rhatT", "sq", "sk", "sv", "mu", "mutilde", "kbar"):
        assert np.array_equal(p2[key], head["p"][key]), key


def test_plain_preparation_after_the_window(orc, head):
    """After the grouping window: the same permutation, no block demeaning.
    Every mean is zero, the value codes are per-channel E4M3 of V[pi] itself
    (torch casts), and the Q and K operands equal the demeaned preparation's."""
    p, N = head["p"], head["N"]
    pp = orc.prepare8(head["q"], head["k"], head["v"], 16, 4, 4242, perm=p["perm"], plain=True)
    assert np.array_equal(pp["perm"], p["perm"])
    assert np.all(pp["mu"] == 0) and np.all(pp["mutilde"] == 0)
    vp = _f(head["v"])[p["perm"]].astype(np.float32)
    sv = np.abs(vp).max(0).astype(np.float32) / np.float32(448)
    assert np.array_equal(pp["sv"], sv)
    assert np.array_equal(pp["rhatT"][:, :N], _e4m3((vp / sv).T))
    assert np.all(pp["rhatT"][:, N:] == 0)
    for key in ("qhat", "sq", "khat", "sk", "kbar"):
        assert np.array_equal(pp[key], p[key]), key
    with pytest.raises(ValueError):
        orc.prepare8(head["q"], head["k"], head["v"], 16, 4, 4242, plain=True)


def test_plain_nvfp4_preparation(orc):
    N, d = 400, 128
    q, k, v = synth.make_qkv(1, 1, N, d, 8, 556)
    p = orc.prepare4(q[0, 0], k[0, 0], v[0, 0], 8, 3, 556)
    pp = orc.prepare4(q[0, 0], k[0, 0], v[0, 0], 8, 3, 556, perm=p["perm"], plain=True)
    assert np.all(pp["mu"] == 0)
    for key in ("q4", "q4s", "gq", "k4", "k4s", "gk", "kbar"):
        assert np.array_equal(pp[key], p[key]), key
    vp = _f(v[0, 0])[p["perm"]]
    assert np.float32(pp["gr"][0]) == np.float32(np.abs(vp).max().astype(np.float32)) / \
        np.float32(2688)
    gr = float(pp["gr"][0])
    scale = np.repeat(_e4m3_val(pp["r4s"]), 16, 1)[:, :N] * gr
    dq = orc.e2m1_decode(pp["r4T"][:, :N].ravel()).reshape(d, N) * scale
    assert np.all(np.abs(dq - vp.T) <= scale + 1e-6)


def test_nvfp4_quantizers(orc):
    N, d = 400, 128
    q, k, v = synth.make_qkv(1, 1, N, d, 8, 555)
    p = orc.prepare4(q[0, 0], k[0, 0], v[0, 0], 8, 3, 555)
    p8 = orc.prepare8(q[0, 0], k[0, 0], v[0, 0], 8, 3, 555)
    assert np.array_equal(p["perm"], p8["perm"]) and np.array_equal(p["mu"], p8["mu"])
    qf = _f(q[0, 0])
    gq = float(p["gq"][0])
    assert np.float32(gq) == np.float32(np.abs(qf).max().astype(np.float32)) / np.float32(2688)
    dq = orc.e2m1_decode(p["q4"][:N].ravel()).reshape(N, d) * \
        np.repeat(_e4m3_val(p["q4s"][:N]), 16, 1) * gq
    scale = np.repeat(_e4m3_val(p["q4s"][:N]), 16, 1) * gq
    # within one E2M1 step of the block (half a step from rounding, up to the
    # saturation at 6 x scale caused by rounding the block scale down)
    assert np.all(np.abs(dq - qf) <= scale * 1.0 + 1e-6)
    assert np.all(p["q4s"] <= 126) and np.max(_e4m3_val(p["q4s"])) <= 448
    # the largest block of the head gets the largest block scale
    assert _e4m3_val(p["q4s"]).max() >= 416
    # residual blocks run along tokens: reconstruct and compare with V' - mu
    vp = _f(v[0, 0])[p["perm"]]
    R = vp - np.repeat(_f(p["mu"]), 128, 0)[:N]
    gr = float(p["gr"][0])
    rs = np.repeat(_e4m3_val(p["r4s"]), 16, 1) * gr                   # [d, Npad]
    rd = orc.e2m1_decode(p["r4T"].ravel()).reshape(d, -1) * rs
    assert np.all(np.abs(rd[:, :N].T - R) <= rs[:, :N].T * 1.0 + 1e-6)
