"""GPU: checkpoint and resume of the cached grouping.  The only state carried
across calls is the permutation, centroids and grid scale in the caller's
state blob, which holds no device addresses, so a blob saved to host memory
and restored into a fresh allocation resumes exactly: a reuse (and a
warm-start) step on the restored blob gives the same operands and output as
on the original."""
import pytest
import torch

import synth
from gpu_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bits,mode_name", [(8, "PERM_REUSE"), (8, "PERM_WARM"), (4, "PERM_REUSE")])
def test_saved_blob_resumes_exactly(bits, mode_name):
    from bit_attention_video_gb300 import vca
    B, H, N, kc = 1, 2, 900, 16
    shape = (B, H, N, 128)
    mode = getattr(vca, mode_name)
    att = (vca.attention_nvfp4 if bits == 4 else vca.attention_fp8)
    q0, k0, v0 = (to_dev(x) for x in synth.make_qkv(B, H, N, 128, 8, 31))
    q1, k1, v1 = (to_dev(x) for x in synth.make_qkv(B, H, N, 128, 8, 32))
    a = vca.alloc_state(B, H, N, 128, kc, bits)
    vca.vsmooth_prepare(q0, k0, v0, kc, a, vca.PERM_FRESH, bits, 3, 5)
    assert vca.get_status(a) == 0
    saved = a.cpu()                          # the checkpoint: plain bytes
    b = vca.alloc_state(B, H, N, 128, kc, bits)
    b.fill_(0xA5)
    b.copy_(saved.cuda())                    # resumed into a fresh allocation
    outs = []
    for blob in (a, b):
        vca.vsmooth_prepare(q1, k1, v1, kc, blob, mode, bits, 3, 5)
        assert vca.get_status(blob) == 0
        o = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
        att(blob, shape, o)
        assert vca.get_status(blob) == 0
        outs.append((o, vca.state_view(blob, shape, kc, bits)))
    (oa, va), (ob, vb) = outs
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    for name in va:
        if name != "status":
            assert torch.equal(va[name], vb[name]), name
