"""GPU: the 4-bit (NVFP4) path.  The preparation (codes, UE4M3 scales, global
scales, block means and the mean operand) is bit-exact with the CPU oracle;
the attention output is within the 4-bit parity bound of the oracle's."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import rel_l2, to_dev
from test_gpu_prep import gpu_prepare

pytestmark = pytest.mark.gpu

REL_L2_4BIT = 1e-2   # GPU vs oracle relative L2 bound of the 4-bit path


def unpack_e2m1(b: np.ndarray) -> np.ndarray:
    """Packed E2M1 bytes (element 2i in the low nibble) -> one code per byte."""
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), np.uint8)
    out[..., 0::2] = b & 0x0F
    out[..., 1::2] = b >> 4
    return out


def tile_rows(t: np.ndarray) -> np.ndarray:
    from bit_attention_video_gb300 import vca
    return vca.scale_tile_to_rows(torch.from_numpy(np.ascontiguousarray(t))).numpy()


def _same(name, a, b):
    if not np.array_equal(a, b):
        bad = np.argwhere(a != b)
        pytest.fail(f"{name} differs at {len(bad)} places, first {bad[:3].tolist()}: "
                    f"{a[tuple(bad[0])]} vs {b[tuple(bad[0])]}")


def check_head4(g, p, bh, N, what=("labels", "perm", "centroids")):
    nb = (N + 127) // 128
    for key in what:
        _same(f"head {bh}: {key}", g[key][bh], p[key])
    _same("kbar", g["kbar"][bh].view(np.uint16), p["kbar"])
    _same("mu", g["mu"][bh].view(np.uint16), p["mu"])
    _same("q4", unpack_e2m1(g["q4"][bh]), p["q4"])
    _same("k4", unpack_e2m1(g["k4"][bh]), p["k4"])
    _same("r4T", unpack_e2m1(g["r4T"][bh]), p["r4T"])
    _same("q4s", tile_rows(g["q4s"][bh]).reshape(nb * 128, 8), p["q4s"])
    kr = g["kr4s"][bh]                                        # [nb][2][1024]
    _same("k4s", tile_rows(kr[:, 0]).reshape(nb * 128, 8), p["k4s"])
    rs = tile_rows(kr[:, 1])                                  # [nb][channel][8 token blocks]
    _same("r4s", rs.transpose(1, 0, 2).reshape(128, nb * 8), p["r4s"])
    _same("g4", g["g4"][bh][:3], np.array([p["gq"][0], p["gk"][0], p["gr"][0]], np.float32))
    # mean operand: groups of 4 blocks aligned to the last block; K rows 2u,
    # 2u+1, 8+2u, 9+2u of slot u hold that block's mean, empty slots are 0
    ng = (nb + 3) // 4
    gpad = ng * 4 - nb
    tiles = g["mside"][bh].view(np.uint16).reshape(ng, 2048)
    c = np.arange(128)
    for slot_j in range(-gpad, nb):
        gi, u = divmod(slot_j + gpad, 4)
        want = p["mu"][slot_j] if slot_j >= 0 else np.zeros(128, np.uint16)
        for k in (2 * u, 2 * u + 1, 8 + 2 * u, 9 + 2 * u):
            idx = (c // 8) * 128 + (k // 8) * 64 + (c % 8) * 8 + (k % 8)
            _same(f"mside group {gi} row {k}", tiles[gi, idx], want)


@pytest.mark.parametrize("B,H,N,C,kc,iters", [
    (1, 1, 1024, 16, 16, 10),    # the small parity configuration
    (1, 2, 1000, 16, 16, 4),     # ragged last block
    (2, 1, 300, 4, 8, 3),        # B > 1, three blocks
    (1, 1, 128, 4, 4, 2),        # exactly one block
    (1, 3, 1, 1, 1, 1),          # one token
    (1, 1, 700, 32, 96, 2),      # 64 < k <= 128 at 4 bits
])
def test_prepare4_bit_exact(orc, B, H, N, C, kc, iters):
    seed = 0xC0FFEE + N
    q, k, v = synth.make_qkv(B, H, N, 128, C, seed)
    _, st, g = gpu_prepare(q, k, v, kc, iters, seed, bits=4)
    assert st == 0
    for b in range(B):
        for h in range(H):
            p = orc.prepare4(q[b, h], k[b, h], v[b, h], kc, iters, seed, b=b, h=h, H=H)
            check_head4(g, p, b * H + h, N)


def test_prepare4_reuse_permutation(orc):
    B, H, N, kc = 1, 2, 900, 8
    q, k, v = synth.make_qkv(B, H, N, 128, 8, 5)
    q2, k2, v2 = synth.make_qkv(B, H, N, 128, 8, 6)
    state, st, g1 = gpu_prepare(q, k, v, kc, 3, 9, bits=4)
    assert st == 0
    state, st, g2 = gpu_prepare(q2, k2, v2, kc, 3, 9, bits=4, reuse=True, state=state)
    assert st == 0
    for h in range(H):
        p = orc.prepare4(q2[0, h], k2[0, h], v2[0, h], kc, 3, 9, perm=g1["perm"][h])
        check_head4(g2, p, h, N, what=("perm",))


def run_nvfp4(q, k, v, kc, iters, seed):
    from bit_attention_video_gb300 import vca
    from gpu_util import to_np_u16
    B, H, N, d = q.shape
    att = vca.VCAttention(B, H, N, d, k_clusters=kc, bits=4, iters=iters, seed=seed)
    out = att(to_dev(q), to_dev(k), to_dev(v))
    return to_np_u16(out), att.status()


@pytest.mark.parametrize("B,H,N,C,kc,iters", [
    (1, 1, 1024, 16, 16, 10),
    (1, 2, 1000, 16, 16, 4),     # ragged last block, two groups of four blocks
    (2, 1, 300, 4, 8, 3),
    (1, 1, 129, 4, 4, 2),        # a one-token last block
    (1, 1, 1, 1, 1, 1),
    (1, 1, 2200, 8, 8, 2),       # 18 blocks: a partial first mean group, several stage wraps
])
def test_nvfp4_attention_matches_oracle(orc, B, H, N, C, kc, iters):
    from gpu_util import bf16_f64
    seed = 0xFACE + N
    q, k, v = synth.make_qkv(B, H, N, 128, C, seed)
    got, st = run_nvfp4(q, k, v, kc, iters, seed)
    assert st == 0
    rows = np.arange(N)
    for b in range(B):
        for h in range(H):
            p = orc.prepare4(q[b, h], k[b, h], v[b, h], kc, iters, seed, b=b, h=h, H=H)
            _, ref = orc.attention4(p, rows)
            err = rel_l2(bf16_f64(got[b, h]), ref)
            assert err <= REL_L2_4BIT, f"(b={b},h={h}) relative L2 {err:.3e}"


def test_nvfp4_attention_h8_sampled_rows(orc):
    from gpu_util import bf16_f64
    w = synth.CONFIGS["h8"]
    q, k, v = synth.make(w)
    got, st = run_nvfp4(q, k, v, w.k, 10, w.seed)
    assert st == 0
    rng = np.random.default_rng(4)
    for h in (2, 7):
        rows = np.sort(rng.choice(w.N, 64, replace=False))
        p = orc.prepare4(q[0, h], k[0, h], v[0, h], w.k, 10, w.seed, b=0, h=h, H=w.H)
        _, ref = orc.attention4(p, rows)
        err = rel_l2(bf16_f64(got[0, h][rows]), ref)
        print(f"h{h}: 4-bit relative L2 vs oracle {err:.2e}")
        assert err <= REL_L2_4BIT


def test_nvfp4_attention_rejects_8bit_state():
    from bit_attention_video_gb300 import vca
    q, k, v = synth.make_qkv(1, 1, 300, 128, 4, 1)
    att = vca.VCAttention(1, 1, 300, 128, k_clusters=4, bits=8, iters=2)
    att.prepare(to_dev(q), to_dev(k), to_dev(v))
    assert att.status() == 0
    out = torch.empty(1, 1, 300, 128, dtype=torch.bfloat16, device="cuda")
    big = torch.zeros(vca.state_bytes(1, 1, 300, 128, 4, 4) + att.state.numel(),
                      dtype=torch.uint8, device="cuda")
    big[:att.state.numel()].copy_(att.state)
    vca.attention_nvfp4(big, (1, 1, 300, 128), out)           # an 8-bit preparation
    assert vca.get_status(big) == -7
