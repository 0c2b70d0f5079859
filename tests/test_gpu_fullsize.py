"""GPU: the full Wan2.2-like 720p workload (B=1, H=40, N=75600, k=64, 10
iterations) in the launch configuration the benchmark times, at 8 and 4 bits;
preparation of three sampled heads (first, middle, last) is bit-exact with the
oracle, and sampled attention rows (including rows of the last full query-tile
pair, of the lone last tile and the last 8 rows) are within relative L2 2e-3
(8-bit) and 1e-2 (4-bit) of the oracle over the sample, every row within 5x
that; their error against exact fp64 attention is reported and bounded loosely
(0.1 and 0.4, the bounds of the oracle's own report)."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import bf16_f64, rel_l2, to_np_u16

pytestmark = pytest.mark.gpu


def _sample_rows(N, rng):
    """24 random rows, 4 of the last full query-tile pair (tiles nb-3, nb-2),
    4 of the last tile (alone in its CTA when nb is odd) and the last 8."""
    nb = (N + 127) // 128
    tail = (nb - 3) * 128
    return np.sort(np.concatenate([rng.choice(tail, 24, replace=False),
                                   rng.choice(np.arange(tail, (nb - 1) * 128), 4, replace=False),
                                   rng.choice(np.arange((nb - 1) * 128, N - 8), 4, replace=False),
                                   np.arange(N - 8, N)]))


def _errors(got, ref):
    """Relative L2 over the sample and of the worst row."""
    per_row = np.linalg.norm(got - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    return rel_l2(got, ref), float(per_row.max())


def test_wan720p_sampled_parity(orc):
    from bit_attention_video_gb300 import vca
    w = synth.CONFIGS["wan720p"]
    shape = (w.B, w.H, w.N, w.d)
    host = [torch.empty(shape, dtype=torch.bfloat16) for _ in range(3)]
    q, k, v = synth.make_qkv(w.B, w.H, w.N, w.d, w.clusters, w.seed,
                             out=tuple(h.view(torch.int16).numpy().view(np.uint16) for h in host))
    dq, dk, dv = (h.cuda() for h in host)
    att = vca.VCAttention(*shape, k_clusters=w.k, bits=8, iters=10, seed=0)
    out = att(dq, dk, dv)
    assert att.status() == 0
    views = vca.state_view(att.state, shape, w.k, 8)
    rng = np.random.default_rng(20)
    for h in (0, w.H // 2, w.H - 1):
        p = orc.prepare8(q[0, h], k[0, h], v[0, h], w.k, 10, 0, b=0, h=h, H=w.H)
        for key in ("labels", "perm", "qhat", "sq", "khat", "sk", "rhatT", "sv", "mutilde"):
            g = views[key][h].cpu().numpy()
            assert np.array_equal(g, p[key]), f"head {h}: {key}"
        assert np.array_equal(views["mu"][h].cpu().numpy().view(np.uint16), p["mu"])
        rows = _sample_rows(w.N, rng)
        _, ref = orc.attention8(p, rows)
        got = bf16_f64(to_np_u16(out[0, h][torch.from_numpy(rows).cuda()]))
        err, worst = _errors(got, ref)
        ex = orc.attention_exact(q[0, h], k[0, h], v[0, h], rows)
        ex_err = rel_l2(got, ex)
        print(f"head {h}: relative L2 vs oracle {err:.2e} (worst row {worst:.2e}), "
              f"vs exact fp64 attention {ex_err:.3f}")
        assert err <= 2e-3 and worst <= 1e-2
        assert ex_err < 0.1


def test_wan720p_nvfp4_sampled_parity(orc):
    from bit_attention_video_gb300 import vca
    from test_gpu_nvfp4 import check_head4
    w = synth.CONFIGS["wan720p_fp4"]
    shape = (w.B, w.H, w.N, w.d)
    host = [torch.empty(shape, dtype=torch.bfloat16) for _ in range(3)]
    q, k, v = synth.make_qkv(w.B, w.H, w.N, w.d, w.clusters, w.seed,
                             out=tuple(h.view(torch.int16).numpy().view(np.uint16) for h in host))
    dq, dk, dv = (h.cuda() for h in host)
    att = vca.VCAttention(*shape, k_clusters=w.k, bits=4, iters=10, seed=0)
    out = att(dq, dk, dv)
    assert att.status() == 0
    views = {n: t.cpu().numpy() for n, t in vca.state_view(att.state, shape, w.k, 4).items()}
    rng = np.random.default_rng(21)
    for h in (1, w.H // 2 + 1, w.H - 2):
        p = orc.prepare4(q[0, h], k[0, h], v[0, h], w.k, 10, 0, b=0, h=h, H=w.H)
        check_head4(views, p, h, w.N, what=("labels", "perm"))
        rows = _sample_rows(w.N, rng)
        _, ref = orc.attention4(p, rows)
        got = bf16_f64(to_np_u16(out[0, h][torch.from_numpy(rows).cuda()]))
        err, worst = _errors(got, ref)
        ex = orc.attention_exact(q[0, h], k[0, h], v[0, h], rows)
        ex_err = rel_l2(got, ex)
        print(f"head {h}: 4-bit relative L2 vs oracle {err:.2e} (worst row {worst:.2e}), "
              f"vs exact fp64 attention {ex_err:.3f}")
        assert err <= 1e-2 and worst <= 5e-2
        assert ex_err < 0.4
