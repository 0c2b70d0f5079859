"""The C ABI library loads, exports every declared entry point and rejects bad
arguments synchronously, before any launch (no GPU needed)."""
import ctypes as C
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def L():
    from bit_attention_video_gb300 import build, vca
    build.build()
    return vca.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "vca.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(vca_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert "vca_vsmooth_prepare" in names and "vca_attention_fp8" in names
    assert "vca_attention_nvfp4" in names and "vca_attention_bf16_ref" in names
    for n in names:
        assert hasattr(L, n), n


def test_state_bytes_and_layout(L):
    from bit_attention_video_gb300 import vca
    n = vca.state_bytes(1, 40, 75600, 128, 64, 8)
    assert n > 3 * 40 * 75648 * 128
    assert vca.state_bytes(1, 1, 100, 64, 8, 8) == 0       # d != 128
    assert vca.state_bytes(1, 1, 100, 128, 101, 8) == 0    # k > N
    assert vca.state_bytes(1, 1, 100, 128, 8, 5) == 0      # bits
    assert vca.state_bytes(1, 65535, 128, 128, 8, 8) > 0   # B*H up to the grids' y extent
    assert vca.state_bytes(256, 256, 128, 128, 8, 8) == 0  # B*H = 65536
    assert vca.state_bytes(1, 128, 1 << 24, 128, 8, 8) == 0  # B*H*Npad = 2^31
    a = vca.state_layout(2, 3, 1000, 128, 16, 8)
    b = vca.state_layout(2, 3, 1000, 128, 64, 8)
    # what the attention reads does not depend on k
    for f in ("qhat", "sq", "khat", "sk", "rhatT", "sv", "mutilde", "mside", "status", "header"):
        assert getattr(a, f) == getattr(b, f), f
    offs = sorted((getattr(a, f), f) for f, _ in vca.StateLayout._fields_
                  if f != "total_bytes" and getattr(a, f))
    assert all(o % 1024 == 0 for o, _ in offs)
    assert offs[-1][0] < a.total_bytes
    c = vca.state_layout(1, 2, 700, 128, 8, 4)
    assert c.q4 and c.kr4s and not c.qhat


def test_prepare_rejects_bad_arguments(L):
    fake = C.c_void_p(1 << 20)       # aligned, never dereferenced: calls fail before launching
    mis = C.c_void_p((1 << 20) + 8)
    nb = L.vca_state_bytes(1, 1, 256, 128, 4, 8)
    P = L.vca_vsmooth_prepare
    ok = dict(q=fake, k=fake, v=fake, B=1, H=1, N=256, d=128, kc=4, reuse=0, bits=8, iters=3,
              seed=0, state=fake, sb=nb, st=None)

    def call(**kw):
        a = dict(ok, **kw)
        return P(a["q"], a["k"], a["v"], a["B"], a["H"], a["N"], a["d"], a["kc"], a["reuse"],
                 a["bits"], a["iters"], a["seed"], a["state"], a["sb"], a["st"])
    assert call(q=None) == -1
    assert call(state=None) == -1
    assert call(v=mis) == -1
    assert call(iters=0) == -1
    assert call(reuse=5) == -1       # 0 fresh, 1 reuse, 2 warm, 3 plain, 4 naive
    assert call(reuse=-1) == -1
    assert call(N=0) == -1
    assert call(d=64) == -2
    assert call(bits=6) == -2
    assert call(kc=300) == -2
    assert call(kc=257 - 1, N=100) == -2
    assert call(sb=nb - 1) == -4
    a = dict(ok)
    X = L.vca_vsmooth_prepare_ex
    assert X(a["q"], a["k"], a["v"], 1, 1, 256, 128, 4, 0, 8, 3, 0, 2, a["state"], nb, None) == -1


def test_attention_rejects_bad_arguments(L):
    fake = C.c_void_p(1 << 20)
    nb = L.vca_state_bytes(1, 2, 300, 128, 1, 8)
    assert L.vca_attention_fp8(None, nb, 1, 2, 300, 128, fake, None) == -1
    assert L.vca_attention_fp8(fake, nb, 1, 2, 300, 128, None, None) == -1
    assert L.vca_attention_fp8_exp(fake, nb, 1, 2, 300, 128, None, None) == -1
    assert L.vca_attention_fp8_exp(fake, nb, 1, 2, 300, 64, fake, None) == -2
    assert L.vca_attention_fp8(fake, nb, 1, 2, 300, 64, fake, None) == -2
    assert L.vca_attention_fp8(fake, 1024, 1, 2, 300, 128, fake, None) == -4
    assert L.vca_attention_fp8(C.c_void_p((1 << 20) + 64), nb, 1, 2, 300, 128, fake, None) == -1
    assert L.vca_attention_bf16_ref(fake, fake, None, 1, 1, 10, 128, fake, None, None) == -1
    assert L.vca_attention_bf16_ref(fake, fake, fake, 1, 1, 10, 96, fake, None, None) == -2
    assert L.vca_debug_mma(9, fake, fake, fake, None) == -1


def test_status_strings(L):
    for code in range(0, -8, -1):
        s = L.vca_status_string(code)
        assert s and s != b"unknown status"
    assert L.vca_status_string(5) == b"unknown status"


def test_pipeline_sizes_and_argument_errors(L):
    """The host-buffer pipeline's workspace size is the state blob plus
    slots x 4 staging tensors (each rounded to 256 bytes), and create refuses
    bad arguments before it creates any CUDA resource."""
    from bit_attention_video_gb300 import vca
    sb = L.vca_state_bytes(1, 2, 300, 128, 8, 8)
    t = (1 * 2 * 300 * 128 * 2 + 255) // 256 * 256
    want = (sb + 255) // 256 * 256 + 3 * 4 * t
    assert vca.pipeline_workspace_bytes(1, 2, 300, 128, 8, 8, 3) == want
    assert vca.pipeline_workspace_bytes(1, 2, 300, 128, 8, 8, 0) == 0
    assert vca.pipeline_workspace_bytes(1, 2, 300, 128, 8, 8, 9) == 0
    assert vca.pipeline_workspace_bytes(1, 2, 300, 64, 8, 8, 2) == 0
    fake = C.c_void_p(1 << 20)
    out = C.c_void_p()
    create = L.vca_pipeline_create
    assert create(1, 2, 300, 128, 8, 8, 3, fake, want, None, None) == -1
    assert create(1, 2, 300, 128, 8, 8, 0, fake, want, None, C.byref(out)) == -1
    assert create(1, 2, 300, 128, 8, 8, 9, fake, want, None, C.byref(out)) == -1
    assert create(1, 2, 300, 64, 8, 8, 3, fake, want, None, C.byref(out)) == -2
    assert create(1, 2, 300, 128, 8, 5, 3, fake, want, None, C.byref(out)) == -2
    assert create(1, 2, 300, 128, 8, 8, 3, None, want, None, C.byref(out)) == -1
    assert create(1, 2, 300, 128, 8, 8, 3, C.c_void_p((1 << 20) + 16), want, None,
                  C.byref(out)) == -1
    assert create(1, 2, 300, 128, 8, 8, 3, fake, want - 1, None, C.byref(out)) == -4
    assert not out.value
    assert L.vca_pipeline_submit(None, fake, fake, fake, fake, 0, 3, 0, 0, None) == -1
    assert L.vca_pipeline_wait(None, 0) == -1
    assert L.vca_pipeline_flush(None) == -1
    assert L.vca_pipeline_destroy(None) == 0
    assert L.vca_pipeline_state(None) is None
