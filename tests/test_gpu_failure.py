"""GPU: the failure path of the kernels' bounded waits, without a fault.  A CTA
whose barriers are never arrived at gives up after its limit, records the
timeout in the status word and leaves; its other warp leaves through the CTA's
abort flag long before its own one-second limit; the host reads
VCA_ERR_TIMEOUT; and the context stays usable (an attention call right after
runs and matches the oracle)."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import bf16_f64, rel_l2, to_dev, to_np_u16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", [0, 1, 2], ids=["suspending", "spinning", "polled"])
def test_wait_gives_up_and_reports_timeout(orc, mode):
    from bit_attention_video_gb300 import vca
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros(4, dtype=torch.int64, device="cuda")
    limit_ns = 1_000_000                                  # 1 ms
    vca.debug_wait_timeout(mode, limit_ns, status, out)
    rc = vca.get_status(None, status)
    assert rc == -6, vca.STATUS_NAMES.get(rc, rc)        # VCA_ERR_TIMEOUT
    gave_up, waited = out.cpu().numpy()[:2], out.cpu().numpy()[2:]
    assert list(gave_up) == [1, 1]
    assert limit_ns <= waited[0] < 200 * limit_ns
    assert waited[1] < 200 * limit_ns, "the second warp left through the abort flag"
    assert vca.get_status(None, status) == 0             # read and cleared
    # the context is intact: a small attention call runs and is right
    B, H, N, kc = 1, 1, 300, 8
    q, k, v = synth.make_qkv(B, H, N, 128, 8, 4242)
    att = vca.VCAttention(B, H, N, 128, k_clusters=kc, bits=8, iters=3, seed=1)
    o = att(to_dev(q), to_dev(k), to_dev(v))
    assert att.status() == 0
    p = orc.prepare8(q[0, 0], k[0, 0], v[0, 0], kc, 3, 1)
    _, ref = orc.attention8(p)
    assert rel_l2(bf16_f64(to_np_u16(o[0, 0])), ref) <= 2e-3


def test_wait_limit_arguments():
    from bit_attention_video_gb300 import vca
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros(4, dtype=torch.int64, device="cuda")
    for mode, limit in ((3, 1000), (-1, 1000), (0, 0), (0, 10 ** 9)):
        with pytest.raises(vca.VcaError):
            vca.debug_wait_timeout(mode, limit, status, out)
    assert np.all(out.cpu().numpy() == 0)
