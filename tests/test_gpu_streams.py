"""GPU: the library keeps no state outside the caller's buffers, so two
problems prepared and attended on two streams at once, their calls
interleaved, give exactly the outputs of the same calls made one problem at a
time on the default stream (an 8-bit and a 4-bit problem, a fresh step then a
step reusing the cached permutation)."""
import pytest
import torch

import synth
from gpu_util import to_dev

pytestmark = pytest.mark.gpu

PROBLEMS = [  # B, H, N, kc, bits, seed
    (1, 2, 700, 8, 8, 901),
    (1, 3, 1000, 16, 4, 902),
]


def _setup(vca):
    out = []
    for B, H, N, kc, bits, seed in PROBLEMS:
        steps = [tuple(to_dev(x) for x in synth.make_qkv(B, H, N, 128, 8, seed + i)) for i in range(2)]
        att = vca.VCAttention(B, H, N, 128, k_clusters=kc, bits=bits, iters=3, seed=7)
        outs = [torch.empty(B, H, N, 128, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        out.append((att, steps, outs))
    torch.cuda.synchronize()
    return out


def test_two_streams_match_one_at_a_time():
    from bit_attention_video_gb300 import vca
    modes = [vca.PERM_FRESH, vca.PERM_REUSE]
    # one problem at a time, default stream
    ref = _setup(vca)
    for att, steps, outs in ref:
        for (q, k, v), m, o in zip(steps, modes, outs):
            att.prepare(q, k, v, reuse_perm=m)
            att.attention(o)
        assert att.status() == 0
    # both problems at once on two streams, calls interleaved
    run = _setup(vca)
    streams = [torch.cuda.Stream() for _ in run]
    for i, m in enumerate(modes):
        for (att, steps, outs), s in zip(run, streams):
            q, k, v = steps[i]
            att.prepare(q, k, v, reuse_perm=m, stream=s)
        for (att, steps, outs), s in zip(run, streams):
            att.attention(outs[i], stream=s)
    for (att, _, _), s in zip(run, streams):
        assert att.status(stream=s) == 0
    torch.cuda.synchronize()
    for (_, _, o_ref), (_, _, o_run) in zip(ref, run):
        for a, b in zip(o_ref, o_run):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
