"""GPU: V-Smooth preparation (k-means labels, permutation, centroids, every
quantised code, scale and mean) is bit-exact with the CPU oracle."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import to_dev

pytestmark = pytest.mark.gpu


def gpu_prepare(q, k, v, kc, iters, seed, bits=8, reuse=False, state=None):
    from bit_attention_video_gb300 import vca
    B, H, N, d = q.shape
    if state is None:
        state = vca.alloc_state(B, H, N, d, kc, bits)
    vca.vsmooth_prepare(to_dev(q), to_dev(k), to_dev(v), kc, state, reuse, bits, iters, seed)
    st = vca.get_status(state)
    views = vca.state_view(state, (B, H, N, d), kc, bits)
    return state, st, {n: t.cpu().numpy() for n, t in views.items()}


def check_head8(g, p, bh, N, what=("labels", "perm", "centroids")):
    for key in what:
        assert np.array_equal(g[key][bh], p[key]), f"head {bh}: {key} differs"
    pairs = [("qhat", "qhat"), ("sq", "sq"), ("khat", "khat"), ("sk", "sk"), ("rhatT", "rhatT"),
             ("sv", "sv"), ("mutilde", "mutilde")]
    for gk, pk in pairs:
        a, b = g[gk][bh], p[pk]
        if not np.array_equal(a, b):
            bad = np.argwhere(a != b)
            pytest.fail(f"head {bh}: {gk} differs at {len(bad)} places, first {bad[:3].tolist()}: "
                        f"{a[tuple(bad[0])]} vs {b[tuple(bad[0])]}")
    assert np.array_equal(g["kbar"][bh].view(np.uint16), p["kbar"]), f"head {bh}: kbar"
    assert np.array_equal(g["mu"][bh].view(np.uint16), p["mu"]), f"head {bh}: mu"
    # mean operand of the restoration MMA: per group of 8 blocks (aligned to
    # the last block) chunk 0 = bf16(mutilde), chunk 1 = bf16 remainder, K
    # columns 8..15 zero
    mt = torch.from_numpy(p["mutilde"])
    hi = mt.to(torch.bfloat16)
    lo = (mt - hi.float()).to(torch.bfloat16)
    hi = hi.view(torch.int16).numpy().view(np.uint16)
    lo = lo.view(torch.int16).numpy().view(np.uint16)
    nb = p["mutilde"].shape[0]
    ng = (nb + 7) // 8
    gpad = ng * 8 - nb
    tiles = g["mside"][bh].view(np.uint16).reshape(ng, 2, 2048)
    c = np.arange(128)
    for slot_j in range(-gpad, nb):
        gi, k = divmod(slot_j + gpad, 8)
        idx = (c // 8) * 128 + (k // 8) * 64 + (c % 8) * 8 + (k % 8)   # in bf16 elements
        want_hi = hi[slot_j] if slot_j >= 0 else 0
        want_lo = lo[slot_j] if slot_j >= 0 else 0
        assert np.array_equal(tiles[gi, 0, idx], np.broadcast_to(want_hi, (128,))), slot_j
        assert np.array_equal(tiles[gi, 1, idx], np.broadcast_to(want_lo, (128,))), slot_j
    upper = (c[:, None] // 8) * 128 + 64 + (c[:, None] % 8) * 8 + np.arange(8)[None, :]
    assert np.all(tiles[:, :, upper.ravel()] == 0)


@pytest.mark.parametrize("B,H,N,C,kc,iters", [
    (1, 1, 1024, 16, 16, 10),    # the small parity configuration
    (1, 2, 1000, 16, 16, 4),     # ragged last block
    (2, 1, 300, 4, 8, 3),        # B > 1, three blocks
    (1, 1, 128, 4, 4, 2),        # exactly one block
    (1, 3, 1, 1, 1, 1),          # one token
    (1, 1, 2500, 64, 200, 2),    # k > 96 (single accumulator group), several sort chunks
    (1, 2, 1300, 64, 96, 3),     # 64 < k <= 128: the tensor-core Lloyd step, two D_a chunks
    (1, 1, 700, 24, 24, 3),      # 16 < k <= 32: one 32-column D_a load
    (1, 1, 1100, 64, 256, 2),    # the largest k (CUDA-core assignment, one accumulator group)
])
def test_prepare8_bit_exact(orc, B, H, N, C, kc, iters):
    seed = 0xC0FFEE + N
    q, k, v = synth.make_qkv(B, H, N, 128, C, seed)
    _, st, g = gpu_prepare(q, k, v, kc, iters, seed)
    assert st == 0
    for b in range(B):
        for h in range(H):
            p = orc.prepare8(q[b, h], k[b, h], v[b, h], kc, iters, seed, b=b, h=h, H=H)
            check_head8(g, p, b * H + h, N)


@pytest.mark.parametrize("kc", [3, 33])
def test_kmeans_extreme_distances(orc, kc):
    """Value tokens on the vertices of the feature cube (every channel
    +-amax, so every feature is +-127), half of them at the two all-equal
    corners: the squared-distance offsets
    ||c||^2 - 2 x.c reach both ends of their range, -128 * 127^2 and
    3 * 128 * 127^2, and the labels, permutation and operands must still be
    bit-exact with the oracle's."""
    B, H, N = 1, 2, 900
    q, k, v = synth.make_qkv(B, H, N, 128, 8, 31)
    rng = np.random.default_rng(31)
    amax = 2.5
    signs = rng.choice([-1.0, 1.0], size=(B, H, N, 1))
    mixed = np.where(rng.random((B, H, N, 128)) < 0.8, signs, -signs)
    corner = np.where(rng.random((B, H, N, 1)) < 0.5, signs, mixed)  # half of them pure corners
    vals = (amax * corner).astype(np.float32)
    v = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    v = np.ascontiguousarray(v)
    _, st, g = gpu_prepare(q, k, v, kc, 4, 17)
    assert st == 0
    for h in range(H):
        p = orc.prepare8(q[0, h], k[0, h], v[0, h], kc, 4, 17, b=0, h=h, H=H)
        check_head8(g, p, h, N)


def test_prepare8_h8_sampled_heads(orc):
    w = synth.CONFIGS["h8"]
    q, k, v = synth.make(w)
    _, st, g = gpu_prepare(q, k, v, w.k, 10, w.seed)
    assert st == 0
    for h in (0, 5):
        p = orc.prepare8(q[0, h], k[0, h], v[0, h], w.k, 10, w.seed, b=0, h=h, H=w.H)
        check_head8(g, p, h, w.N)


def test_reuse_permutation(orc):
    B, H, N, kc = 1, 2, 900, 8
    q, k, v = synth.make_qkv(B, H, N, 128, 8, 5)
    q2, k2, v2 = synth.make_qkv(B, H, N, 128, 8, 6)      # the next "denoising step"
    state, st, g1 = gpu_prepare(q, k, v, kc, 3, 9)
    assert st == 0
    state, st, g2 = gpu_prepare(q2, k2, v2, kc, 3, 9, reuse=True, state=state)
    assert st == 0
    assert np.array_equal(g1["perm"], g2["perm"])
    for h in range(H):
        p = orc.prepare8(q2[0, h], k2[0, h], v2[0, h], kc, 3, 9, perm=g1["perm"][h])
        check_head8(g2, p, h, N, what=("perm",))


@pytest.mark.parametrize("bits,B,H,N,C,kc,it0,it1", [
    (8, 1, 2, 1000, 16, 16, 4, 2),     # ragged last block
    (8, 2, 1, 2500, 64, 40, 3, 1),     # B > 1, several sort chunks
    (8, 1, 1, 700, 32, 144, 2, 2),     # k > 128 (the CUDA-core assignment)
    (4, 1, 2, 640, 16, 16, 3, 2),      # the 4-bit preparation shares the grouping
])
def test_warm_start_matches_oracle(orc, bits, B, H, N, C, kc, it0, it1):
    """A fresh grouping of one step, then a warm start on the next step's
    values: labels, permutation, centroids and feature grid scale are
    bit-exact with the oracle's warm k-means, and so is every operand."""
    from bit_attention_video_gb300 import vca
    q, k, v = synth.make_qkv(B, H, N, 128, C, 21)
    q2, k2, v2 = synth.make_qkv(B, H, N, 128, C, 22)     # the next "denoising step"
    v2[0, 0, 3, 5] = 0x4300                              # 128.0: the grid scale changes
    state, st, g1 = gpu_prepare(q, k, v, kc, it0, 13, bits=bits)
    assert st == 0
    state, st, g2 = gpu_prepare(q2, k2, v2, kc, it1, 13, bits=bits, reuse=vca.PERM_WARM,
                                state=state)
    assert st == 0
    for b in range(B):
        for h in range(H):
            bh = b * H + h
            _, s1, _, c1 = orc.kmeans(v[b, h], kc, it0, 13, b=b, h=h, H=H)
            assert np.array_equal(g1["centroids"][bh], c1) and g1["grid_scale"][bh] == s1
            _, s2, lab, cent = orc.kmeans_warm(v2[b, h], c1, s1, it1)
            assert g2["grid_scale"][bh] == s2
            assert np.array_equal(g2["labels"][bh], lab), f"head {bh}: labels"
            assert np.array_equal(g2["centroids"][bh], cent), f"head {bh}: centroids"
            perm = orc.stable_argsort(lab, kc)
            assert np.array_equal(g2["perm"][bh], perm), f"head {bh}: perm"
            if bits == 8:
                p = orc.prepare8(q2[b, h], k2[b, h], v2[b, h], kc, it1, 13, perm=perm)
                check_head8(g2, p, bh, N, what=("perm",))
    # a reuse after the warm start keeps the warm permutation
    state, st, g3 = gpu_prepare(q, k, v, kc, it1, 13, bits=bits, reuse=vca.PERM_REUSE,
                                state=state)
    assert st == 0 and np.array_equal(g3["perm"], g2["perm"])


def test_warm_start_without_cached_grouping_is_reported(orc):
    from bit_attention_video_gb300 import vca
    B, H, N, kc = 1, 1, 300, 4
    q, k, v = synth.make_qkv(B, H, N, 128, 4, 5)
    state = vca.alloc_state(B, H, N, 128, kc, 8)
    state.zero_()
    vca.vsmooth_prepare(to_dev(q), to_dev(k), to_dev(v), kc, state, vca.PERM_WARM, 8, 2, 0)
    assert vca.get_status(state) == -5


def test_reuse_without_cached_permutation_is_reported(orc):
    from bit_attention_video_gb300 import vca
    B, H, N, kc = 1, 1, 300, 4
    q, k, v = synth.make_qkv(B, H, N, 128, 4, 5)
    state = vca.alloc_state(B, H, N, 128, kc, 8)
    state.zero_()
    vca.vsmooth_prepare(to_dev(q), to_dev(k), to_dev(v), kc, state, True, 8, 2, 0)
    assert vca.get_status(state) == -5
    # a blob prepared with another k is refused as well
    state2 = vca.alloc_state(B, H, N, 128, 8, 8)
    vca.vsmooth_prepare(to_dev(q), to_dev(k), to_dev(v), 8, state2, False, 8, 2, 0)
    assert vca.get_status(state2) == 0
    big = torch.zeros(max(state.numel(), state2.numel()), dtype=torch.uint8, device="cuda")
    big[:state2.numel()].copy_(state2)
    vca.vsmooth_prepare(to_dev(q), to_dev(k), to_dev(v), 4, big, True, 8, 2, 0)
    assert vca.get_status(big) == -5


def test_quantiser_rounding_boundaries(orc):
    """Quotients on E4M3 rounding midpoints: every 128-row block of Q holds
    448 (so its scale is exactly 1) and values halfway between two E4M3 codes,
    which the quantiser must round to even exactly as the oracle's division
    does (the reciprocal shortcut cannot decide them)."""
    B, H, N, kc = 1, 1, 512, 4
    q, k, v = synth.make_qkv(B, H, N, 128, 4, 77)
    rng = np.random.default_rng(5)
    mids = np.array([1 + (2 * m + 1) / 16 for m in range(8)] +
                    [2 * (1 + (2 * m + 1) / 16) for m in range(8)], np.float32)
    vals = rng.choice(np.concatenate([mids, -mids]), size=(N, 128)).astype(np.float32)
    vals[::128, 0] = 448.0
    q = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    q = np.ascontiguousarray(q.reshape(B, H, N, 128))
    _, st, g = gpu_prepare(q, k, v, kc, 2, 3)
    assert st == 0
    p = orc.prepare8(q[0, 0], k[0, 0], v[0, 0], kc, 2, 3)
    assert np.all(p["sq"] == 1.0)
    assert np.array_equal(g["qhat"][0], p["qhat"])
    assert np.array_equal(g["sq"][0], p["sq"])
