"""GPU: the allocation-free grouping entry point (for callers that cannot
allocate device memory) gives the same k-means labels and permutation as the
state-blob preparation, on two calls in a row with different inputs, so the
contents its shared scratch keeps from the previous call do not matter; at
the largest size it accepts; and its device status word reads 0 after every
call."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import to_dev

pytestmark = pytest.mark.gpu


def _compare_with_prepare(B, H, N, kc, iters, seed, data_seeds):
    from bit_attention_video_gb300 import vca
    for call, data_seed in enumerate(data_seeds):
        q, k, v = synth.make_qkv(B, H, N, 128, 12, data_seed)
        dq, dk, dv = to_dev(q), to_dev(k), to_dev(v)
        state = vca.alloc_state(B, H, N, 128, kc, 8)
        vca.vsmooth_prepare(dq, dk, dv, kc, state, False, 8, iters, seed)
        assert vca.get_status(state) == 0
        view = vca.state_view(state, (B, H, N, 128), kc, 8)
        for h in range(H):
            labels = torch.full((N,), -1, dtype=torch.int32, device="cuda")
            perm = torch.full((N,), -1, dtype=torch.int32, device="cuda")
            vca.kmeans_permutation_noalloc(dv[0, h].contiguous(), kc, labels, perm, iters, seed,
                                           b=0, h=h, H=H)
            assert vca.noalloc_status() == 0, f"call {call} head {h}: device status"
            assert torch.equal(labels, view["labels"][h]), f"call {call} head {h}: labels"
            assert torch.equal(perm, view["perm"][h]), f"call {call} head {h}: perm"


def test_noalloc_grouping_matches_prepare_twice():
    _compare_with_prepare(1, 2, 5000, 16, 5, 12345, (101, 202))


def test_noalloc_largest_size_and_cluster_count():
    """N at the maximum and k = 256: the sort histogram fills the end of the
    fixed array (16 chunks x 256 clusters), and k > 128 takes the other
    assignment kernel."""
    from bit_attention_video_gb300 import vca
    _compare_with_prepare(1, 1, vca.NOALLOC_MAX_TOKENS, 256, 3, 99, (303,))


def test_noalloc_refuses_short_outputs():
    from bit_attention_video_gb300 import vca
    v = torch.zeros(300, 128, dtype=torch.bfloat16, device="cuda")
    ok = torch.empty(300, dtype=torch.int32, device="cuda")
    short = torch.empty(299, dtype=torch.int32, device="cuda")
    for labels, perm in ((short, ok), (ok, short)):
        with pytest.raises(vca.VcaError):
            vca.kmeans_permutation_noalloc(v, 8, labels, perm)


def test_noalloc_rejects_sizes_beyond_its_maximum():
    from bit_attention_video_gb300 import vca
    n = vca.NOALLOC_MAX_TOKENS + 1
    v = torch.zeros(n, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(n, dtype=torch.int32, device="cuda")
    with pytest.raises(vca.VcaError) as e:
        vca.kmeans_permutation_noalloc(v, 8, out, out.clone())
    assert e.value.code == -2
