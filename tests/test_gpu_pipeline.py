"""The host-buffer pipeline (vca_pipeline_*): every step's O, read back into
host memory, is bit-identical with the device-buffer calls made in the same
order on the same inputs, for several slot counts, both bit widths and a mix
of grouping modes; a refused submit leaves the pipeline usable."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _host(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).pin_memory()


def _direct(steps, B, H, N, kc, bits, iters, modes):
    from bit_attention_video_gb300 import vca
    att = vca.VCAttention(B, H, N, 128, k_clusters=kc, bits=bits, iters=iters)
    outs = []
    for (q, k, v), m in zip(steps, modes):
        o = torch.empty(B, H, N, 128, dtype=torch.bfloat16, device="cuda")
        att.prepare(q.cuda(), k.cuda(), v.cuda(), reuse_perm=m)
        att.attention(o)
        outs.append(o.cpu())
    assert att.status() == 0
    return outs


@pytest.mark.parametrize("bits,slots,modes", [
    (8, 2, [0, 1, 3, 0, 2, 1, 0]),
    (8, 3, [0, 0, 1, 2, 0]),
    (8, 1, [0, 1, 0]),
    (4, 2, [0, 1, 2, 0]),
])
def test_pipeline_matches_device_calls(bits, slots, modes, B=1, H=2, N=700):
    from bit_attention_video_gb300 import vca
    kc, iters = 8, 3
    steps = [tuple(_host(x) for x in synth.make_qkv(B, H, N, 128, 8, 100 + i))
             for i in range(len(modes))]
    want = _direct(steps, B, H, N, kc, bits, iters, modes)
    pipe = vca.HostPipeline(B, H, N, 128, k_clusters=kc, bits=bits, slots=slots, iters=iters)
    outs = [torch.empty(B, H, N, 128, dtype=torch.bfloat16).pin_memory() for _ in modes]
    ids = [pipe.submit(*s, o, reuse_perm=m) for s, o, m in zip(steps, outs, modes)]
    assert ids == list(range(len(modes)))
    pipe.wait(ids[1])                      # an early step, while later ones may still run
    assert torch.equal(outs[1].view(torch.int16), want[1].view(torch.int16))
    pipe.flush()
    for i, (o, w) in enumerate(zip(outs, want)):
        assert torch.equal(o.view(torch.int16), w.view(torch.int16)), i
    pipe.close()


def test_pipeline_batch_of_two_ragged_length():
    """B = 2 and a length that is not a multiple of 128."""
    test_pipeline_matches_device_calls(8, 3, [0, 1, 0, 2], B=2, H=1, N=333)


def test_pipeline_refused_submit_and_pageable_memory():
    from bit_attention_video_gb300 import vca
    B, H, N, kc = 1, 1, 300, 4
    q, k, v = (_host(x) for x in synth.make_qkv(B, H, N, 128, 4, 7))
    pipe = vca.HostPipeline(B, H, N, 128, k_clusters=kc, bits=8, slots=2, iters=2)
    o = torch.empty(B, H, N, 128, dtype=torch.bfloat16)       # pageable: correct, not overlapped
    with pytest.raises(vca.VcaError) as e:
        pipe.submit(q, k, v, o, reuse_perm=7)
    assert e.value.code == -1
    with pytest.raises(vca.VcaError):
        pipe.wait(0)                                           # nothing was submitted
    assert pipe.submit(q, k, v, o) == 0
    assert pipe.submit(q, k, v, o, reuse_perm=vca.PERM_REUSE) == 1
    pipe.flush()
    want = _direct([(q, k, v)] * 2, B, H, N, kc, 8, 2, [0, 1])
    assert torch.equal(o.view(torch.int16), want[1].view(torch.int16))
    pipe.close()
    pipe.close()                                               # idempotent


@pytest.mark.parametrize("qk_hadamard,fp8_exp", [(True, False), (False, True), (True, True)])
def test_pipeline_flags_match_device_calls(qk_hadamard, fp8_exp):
    """The pipeline's option bits reach the calls they name: the QK rotation
    in the preparation, and the conventional exp-then-cast product."""
    from bit_attention_video_gb300 import vca
    B, H, N, kc, iters = 1, 2, 600, 8, 2
    steps = [tuple(_host(x) for x in synth.make_qkv(B, H, N, 128, 8, 300 + i)) for i in range(3)]
    modes = [0, 1, 0]
    flags = vca.PREP_QK_HADAMARD if qk_hadamard else 0
    state = vca.alloc_state(B, H, N, 128, kc, 8)
    want = []
    for (q, k, v), m in zip(steps, modes):
        o = torch.empty(B, H, N, 128, dtype=torch.bfloat16, device="cuda")
        vca.vsmooth_prepare(q.cuda(), k.cuda(), v.cuda(), kc, state, m, 8, iters, 0, None, flags)
        (vca.attention_fp8_exp if fp8_exp else vca.attention_fp8)(state, (B, H, N, 128), o)
        want.append(o.cpu())
    assert vca.get_status(state) == 0
    pipe = vca.HostPipeline(B, H, N, 128, k_clusters=kc, bits=8, slots=2, iters=iters,
                            qk_hadamard=qk_hadamard, fp8_exp=fp8_exp)
    outs = [torch.empty(B, H, N, 128, dtype=torch.bfloat16).pin_memory() for _ in modes]
    for s, o, m in zip(steps, outs, modes):
        pipe.submit(*s, o, reuse_perm=m)
    pipe.flush()
    for i, (o, w) in enumerate(zip(outs, want)):
        assert torch.equal(o.view(torch.int16), w.view(torch.int16)), i
    pipe.close()


def test_pipeline_rejects_exp_product_at_4_bits():
    from bit_attention_video_gb300 import vca
    B, H, N = 1, 1, 256
    q, k, v = (_host(x) for x in synth.make_qkv(B, H, N, 128, 4, 9))
    o = torch.empty(B, H, N, 128, dtype=torch.bfloat16).pin_memory()
    pipe = vca.HostPipeline(B, H, N, 128, k_clusters=4, bits=4, slots=2, iters=2, fp8_exp=True)
    with pytest.raises(vca.VcaError) as e:
        pipe.submit(q, k, v, o)
    assert e.value.code == -1
    pipe.close()
