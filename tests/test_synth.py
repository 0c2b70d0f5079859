"""The seeded generators follow their stated recipe (no GPU)."""
import numpy as np
import torch

import synth


def _f(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16) \
        .to(torch.float64).numpy()


def test_deterministic_and_index_addressable():
    a = synth.make_qkv(1, 2, 512, 128, 8, 7)
    b = synth.make_qkv(1, 2, 512, 128, 8, 7)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    # a longer sequence extends the shorter one head by head (values depend on the
    # global index, so only head 0's prefix coincides)
    c = synth.make_qkv(1, 1, 1024, 128, 8, 7)
    assert np.array_equal(c[1][0, 0, :512], a[1][0, 0])


def test_recipe_statistics():
    B, H, N, C = 1, 4, 8192, 16
    q, k, v = synth.make_qkv(B, H, N, 128, C, 11)
    qf = _f(q[0])
    off = qf.mean(1)                                   # per-(h, channel) offset estimate
    assert abs(off.var() - 2.0) < 0.4                  # offsets ~ N(0, 2)
    assert abs((qf - off[:, None, :]).std() - 1.0) < 0.02
    lab, outl = synth.v_labels(B, H, N, C, 11, 0, 2)
    assert abs(outl.mean() - 0.01) < 0.004
    assert np.bincount(lab, minlength=C).min() > N / C * 0.8
    vf = _f(v[0, 2])
    normal = vf[~outl]
    for m in range(C):
        rows = normal[lab[~outl] == m]
        assert abs(rows.std(0).mean() - 0.3) < 0.03     # spread 0.3 around the centre
    big = np.abs(vf[outl]) > 8 * np.abs(vf[~outl]).max(0).mean()
    assert np.all(big.sum(1) <= 4)
