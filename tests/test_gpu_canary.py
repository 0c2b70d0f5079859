"""GPU: guard bands around every buffer the library writes (the state blob, the
attention output, the allocation-free call's labels and permutation), in place
of a memory checker.  Each buffer sits between two 4 KB bands of a known byte
pattern; after the calls of each preparation mode and bit width, on ragged
shapes, the bands must be intact and the inputs unchanged."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import to_dev

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


class Guarded:
    """A device buffer of `nbytes` between two guard bands."""

    def __init__(self, nbytes):
        self.n = nbytes
        self.raw = torch.full((2 * GUARD + nbytes,), PATTERN, dtype=torch.uint8, device="cuda")
        self.inner = self.raw[GUARD:GUARD + nbytes]

    def view(self, dtype, shape):
        return self.inner.view(dtype).view(*shape)

    def check(self, what):
        torch.cuda.synchronize()
        lo, hi = self.raw[:GUARD], self.raw[GUARD + self.n:]
        for name, band in (("before", lo), ("after", hi)):
            bad = torch.nonzero(band != PATTERN)
            assert bad.numel() == 0, f"{what}: guard band {name} overwritten at {bad[:4].tolist()}"


def _inputs(B, H, N, seed):
    q, k, v = synth.make_qkv(B, H, N, 128, 8, seed)
    dev = [to_dev(x) for x in (q, k, v)]
    return dev, [x.clone() for x in dev]


CASES = [
    # bits, B, H, N, k, modes in order, QK rotation
    (8, 2, 3, 700, 8, ("fresh", "reuse", "warm", "plain", "naive"), False),
    (8, 1, 2, 129, 4, ("fresh", "reuse"), True),
    (8, 1, 1, 1000, 144, ("fresh", "warm"), False),
    (8, 1, 1, 1, 1, ("fresh",), False),
    (4, 2, 3, 700, 8, ("fresh", "reuse", "warm", "plain"), False),
    (4, 1, 2, 300, 16, ("fresh", "reuse"), True),
]


@pytest.mark.parametrize("bits,B,H,N,kc,modes,rot", CASES)
def test_guard_bands_intact(bits, B, H, N, kc, modes, rot):
    from bit_attention_video_gb300 import vca
    mode_id = {"fresh": vca.PERM_FRESH, "reuse": vca.PERM_REUSE, "warm": vca.PERM_WARM,
               "plain": vca.PERM_PLAIN, "naive": vca.PERM_NAIVE}
    shape = (B, H, N, 128)
    state = Guarded(vca.state_bytes(B, H, N, 128, kc, bits))
    out = Guarded(B * H * N * 128 * 2)
    o = out.view(torch.bfloat16, shape)
    st = state.inner
    flags = vca.PREP_QK_HADAMARD if rot else 0
    for i, mode in enumerate(modes):
        (q, k, v), orig = _inputs(B, H, N, 900 + i)
        vca.vsmooth_prepare(q, k, v, kc, st, mode_id[mode], bits, 3, 5, flags=flags)
        assert vca.get_status(st) == 0, mode
        state.check(f"{mode} preparation: state")
        calls = [vca.attention_nvfp4] if bits == 4 else [vca.attention_fp8, vca.attention_fp8_exp]
        for call in calls:
            call(st, shape, o)
            assert vca.get_status(st) == 0
            out.check(f"{mode} {call.__name__}: output")
            state.check(f"{mode} {call.__name__}: state")
        for a, b in zip((q, k, v), orig):
            assert torch.equal(a, b), "an input was modified"


def test_guard_bands_reference_and_noalloc():
    from bit_attention_video_gb300 import vca
    B, H, N = 1, 2, 300
    (q, k, v), orig = _inputs(B, H, N, 77)
    out = Guarded(B * H * N * 128 * 2)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    vca.attention_bf16_ref(q, k, v, out.view(torch.bfloat16, (B, H, N, 128)), status)
    assert vca.get_status(None, status) == 0
    out.check("bf16 reference: output")
    labels, perm = Guarded(4 * N), Guarded(4 * N)
    vca.kmeans_permutation_noalloc(v[0, 1].contiguous(), 8, labels.view(torch.int32, (N,)),
                                   perm.view(torch.int32, (N,)), 3, 1, b=0, h=1, H=H)
    assert vca.noalloc_status() == 0
    labels.check("noalloc labels")
    perm.check("noalloc perm")
    assert sorted(perm.view(torch.int32, (N,)).cpu().tolist()) == list(range(N))
    for a, b in zip((q, k, v), orig):
        assert torch.equal(a, b)
