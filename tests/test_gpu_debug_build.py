"""GPU: the VCA_DEBUG build of the library, whose kernels check every
data-dependent index they address memory with (the cached permutation in the
gathers, labels in the sort, the sort's scatter position) and record an error
instead of an out-of-bounds access.  On the small cases every call leaves the
status word clear and gives the release build's outputs bit for bit; a reuse
step on a blob whose cached permutation was corrupted (entries past N, in head
0 of 2, so that even an unchecked read would stay inside the value tensor) is
stopped by the checks and reported as VCA_ERR_INVALID_ARG."""
import pytest
import torch

import synth
from gpu_util import to_dev

pytestmark = pytest.mark.gpu

MODES = ("fresh", "reuse", "warm", "plain", "naive")


def _run(vca, bits, B, H, N, kc, modes, rot):
    mode_id = {"fresh": vca.PERM_FRESH, "reuse": vca.PERM_REUSE, "warm": vca.PERM_WARM,
               "plain": vca.PERM_PLAIN, "naive": vca.PERM_NAIVE}
    shape = (B, H, N, 128)
    state = vca.alloc_state(B, H, N, 128, kc, bits)
    o = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    results = []
    for i, mode in enumerate(modes):
        q, k, v = (to_dev(x) for x in synth.make_qkv(B, H, N, 128, 8, 500 + i))
        vca.vsmooth_prepare(q, k, v, kc, state, mode_id[mode], bits, 3, 9,
                            flags=vca.PREP_QK_HADAMARD if rot else 0)
        assert vca.get_status(state) == 0, mode
        (vca.attention_nvfp4 if bits == 4 else vca.attention_fp8)(state, shape, o)
        assert vca.get_status(state) == 0, mode
        view = vca.state_view(state, shape, kc, bits)
        results.append((mode, o.clone(), {n: t.clone() for n, t in view.items()}))
    return results


@pytest.mark.parametrize("bits,B,H,N,kc,modes,rot", [
    (8, 2, 3, 700, 8, MODES, False),
    (8, 1, 1, 1000, 144, ("fresh", "warm"), False),
    (8, 1, 2, 300, 8, ("fresh", "naive"), True),
    (4, 2, 3, 700, 8, MODES[:4], False),
    (4, 1, 2, 300, 16, ("fresh", "reuse"), True),
])
def test_debug_build_matches_release(bits, B, H, N, kc, modes, rot):
    from bit_attention_video_gb300 import vca
    rel = _run(vca, bits, B, H, N, kc, modes, rot)
    with vca.debug_build():
        dbg = _run(vca, bits, B, H, N, kc, modes, rot)
    for (mode, o_r, v_r), (_, o_d, v_d) in zip(rel, dbg):
        assert torch.equal(o_r.view(torch.int16), o_d.view(torch.int16)), f"{mode}: output"
        for name in v_r:
            if name != "status":
                assert torch.equal(v_r[name], v_d[name]), f"{mode}: {name}"


@pytest.mark.parametrize("bits", [8, 4])
def test_debug_build_stops_a_corrupted_permutation(bits):
    from bit_attention_video_gb300 import vca
    B, H, N, kc = 1, 2, 300, 8
    shape = (B, H, N, 128)
    q, k, v = (to_dev(x) for x in synth.make_qkv(B, H, N, 128, 8, 61))
    with vca.debug_build():
        state = vca.alloc_state(B, H, N, 128, kc, bits)
        vca.vsmooth_prepare(q, k, v, kc, state, vca.PERM_FRESH, bits, 3, 0)
        assert vca.get_status(state) == 0
        perm = vca.state_view(state, shape, kc, bits)["perm"]
        perm[0, 5:9] = N + 3        # past head 0's tokens, still inside the tensors
        vca.vsmooth_prepare(q, k, v, kc, state, vca.PERM_REUSE, bits, 3, 0)
        assert vca.get_status(state) == -1        # VCA_ERR_INVALID_ARG: kStatBadArg
        # a fresh grouping rewrites the permutation and clears the word
        vca.vsmooth_prepare(q, k, v, kc, state, vca.PERM_FRESH, bits, 3, 0)
        assert vca.get_status(state) == 0
