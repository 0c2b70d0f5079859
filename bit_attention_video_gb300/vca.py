"""Thin Python binding of the VC-Attention C ABI (``include/vca.h``).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libvca.so``.  PyTorch supplies device memory and streams.  There
is no fallback: if the library is missing the import of a function fails
loudly.
"""
from __future__ import annotations

import contextlib
import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libvca.so")
# the -DVCA_DEBUG build (index checks that record an error instead of an
# out-of-bounds access), loaded beside the release build for tests
LIB_DEBUG_PATH = os.path.join(_HERE, "_build_debug", "libvca.so")
_lib = None
_lib_debug = None
_override = None

VCA_OK = 0
STATUS_NAMES = {0: "VCA_OK", -1: "VCA_ERR_INVALID_ARG", -2: "VCA_ERR_UNSUPPORTED",
                -3: "VCA_ERR_CUDA", -4: "VCA_ERR_BUFFER_TOO_SMALL",
                -5: "VCA_ERR_NO_CACHED_PERM", -6: "VCA_ERR_TIMEOUT",
                -7: "VCA_ERR_STATE_MISMATCH"}
DEFAULT_ITERS = 10
DEFAULT_SEED = 0
# reuse_perm modes of vsmooth_prepare (False / True map to FRESH / REUSE)
PERM_FRESH, PERM_REUSE, PERM_WARM, PERM_PLAIN, PERM_NAIVE = 0, 1, 2, 3, 4
# option bits of vsmooth_prepare
PREP_QK_HADAMARD = 1
# option bit of HostPipeline (vca_pipeline_submit): the conventional exp-then-cast FP8 product
PIPELINE_FP8_EXP = 0x100


class VcaError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} returned {STATUS_NAMES.get(code, code)}")
        self.code = code


class StateLayout(C.Structure):
    _fields_ = [(n, C.c_uint64) for n in (
        "total_bytes", "header", "status", "labels", "perm", "centroids", "grid", "features",
        "sums", "qhat", "sq", "khat", "sk", "kbar", "ksum", "rhatT", "sv", "mu", "mutilde",
        "mside", "vamax", "q4", "q4s", "k4", "kr4s", "r4T", "g4")]


def lib():
    """Load libvca.so (raises if it has not been built).  Inside
    ``debug_build()`` this is the VCA_DEBUG build instead."""
    global _lib
    if _override is not None:
        return _override
    if _lib is None:
        _lib = _load(LIB_PATH)
    return _lib


def lib_debug():
    """Load the VCA_DEBUG build (raises if it has not been built)."""
    global _lib_debug
    if _lib_debug is None:
        _lib_debug = _load(LIB_DEBUG_PATH, "build(debug=True)")
    return _lib_debug


@contextlib.contextmanager
def debug_build():
    """Route every call of this module through the VCA_DEBUG build."""
    global _override
    prev, _override = _override, lib_debug()
    try:
        yield _override
    finally:
        _override = prev


def _load(path, how="build()"):
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: run bit_attention_video_gb300.build.{how}")
    L = C.CDLL(path)
    P, I, S, U64 = C.c_void_p, C.c_int, C.c_size_t, C.c_uint64
    L.vca_state_bytes.restype = S
    L.vca_state_bytes.argtypes = [I] * 6
    L.vca_state_layout_get.restype = I
    L.vca_state_layout_get.argtypes = [I] * 6 + [C.POINTER(StateLayout)]
    L.vca_vsmooth_prepare.restype = I
    L.vca_vsmooth_prepare.argtypes = [P, P, P, I, I, I, I, I, I, I, I, U64, P, S, P]
    L.vca_vsmooth_prepare_ex.restype = I
    L.vca_vsmooth_prepare_ex.argtypes = [P, P, P, I, I, I, I, I, I, I, I, U64, C.c_uint, P,
                                         S, P]
    for fn in ("vca_attention_fp8", "vca_attention_fp8_exp", "vca_attention_nvfp4"):
        getattr(L, fn).restype = I
        getattr(L, fn).argtypes = [P, S, I, I, I, I, P, P]
    L.vca_attention_bf16_ref.restype = I
    L.vca_attention_bf16_ref.argtypes = [P, P, P, I, I, I, I, P, P, P]
    L.vca_get_status.restype = I
    L.vca_get_status.argtypes = [P, P, P]
    L.vca_status_string.restype = C.c_char_p
    L.vca_status_string.argtypes = [I]
    L.vca_debug_expcast.restype = I
    L.vca_debug_expcast.argtypes = [P, P, P, P, S, P]
    L.vca_debug_expcast_rows.restype = I
    L.vca_debug_expcast_rows.argtypes = [P, P, P, P, P, P, S, P]
    L.vca_debug_encode.restype = I
    L.vca_debug_encode.argtypes = [P, P, P, S, P]
    L.vca_debug_mma.restype = I
    L.vca_debug_mma.argtypes = [I, P, P, P, P]
    L.vca_kmeans_permutation_noalloc.restype = I
    L.vca_kmeans_permutation_noalloc.argtypes = [P, I, I, I, I, U64, I, I, I, P, P, P]
    L.vca_pipeline_workspace_bytes.restype = S
    L.vca_pipeline_workspace_bytes.argtypes = [I] * 7
    L.vca_pipeline_create.restype = I
    L.vca_pipeline_create.argtypes = [I] * 7 + [P, S, P, C.POINTER(C.c_void_p)]
    L.vca_pipeline_submit.restype = I
    L.vca_pipeline_submit.argtypes = [P, P, P, P, P, I, I, U64, C.c_uint,
                                      C.POINTER(C.c_int64)]
    L.vca_pipeline_wait.restype = I
    L.vca_pipeline_wait.argtypes = [P, C.c_int64]
    L.vca_pipeline_flush.restype = I
    L.vca_pipeline_flush.argtypes = [P]
    L.vca_pipeline_state.restype = P
    L.vca_pipeline_state.argtypes = [P]
    L.vca_pipeline_destroy.restype = I
    L.vca_pipeline_destroy.argtypes = [P]
    L.vca_debug_wait_timeout.restype = I
    L.vca_debug_wait_timeout.argtypes = [I, U64, P, P, P]
    return L


def _check(fn, rc):
    if rc != VCA_OK:
        raise VcaError(fn, rc)


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, dtype=None):
    assert t.is_cuda and t.is_contiguous(), "expected a contiguous CUDA tensor"
    if dtype is not None:
        assert t.dtype == dtype, f"expected {dtype}, got {t.dtype}"
    return C.c_void_p(t.data_ptr())


# ----------------------------------------------------------------------------
def state_bytes(B, H, N, d, k_clusters, bits) -> int:
    return lib().vca_state_bytes(B, H, N, d, k_clusters, bits)


def state_layout(B, H, N, d, k_clusters, bits) -> StateLayout:
    L = StateLayout()
    _check("vca_state_layout_get", lib().vca_state_layout_get(B, H, N, d, k_clusters, bits,
                                                              C.byref(L)))
    return L


def alloc_state(B, H, N, d, k_clusters, bits, device="cuda") -> torch.Tensor:
    n = state_bytes(B, H, N, d, k_clusters, bits)
    if n == 0:
        raise VcaError("vca_state_bytes", -1)
    return torch.empty(n, dtype=torch.uint8, device=device)


def vsmooth_prepare(q, k, v, k_clusters, state, reuse_perm=False, bits=8,
                    iters=DEFAULT_ITERS, seed=DEFAULT_SEED, stream=None, flags=0):
    """flags: 0 or PREP_QK_HADAMARD."""
    B, H, N, d = q.shape
    _check("vca_vsmooth_prepare_ex", lib().vca_vsmooth_prepare_ex(
        _dev(q, torch.bfloat16), _dev(k, torch.bfloat16), _dev(v, torch.bfloat16), B, H, N, d,
        k_clusters, int(reuse_perm), bits, iters, seed, flags, _dev(state, torch.uint8),
        state.numel(), _stream(stream)))


def attention_fp8(state, shape, out, stream=None):
    B, H, N, d = shape
    _check("vca_attention_fp8", lib().vca_attention_fp8(
        _dev(state, torch.uint8), state.numel(), B, H, N, d, _dev(out, torch.bfloat16),
        _stream(stream)))


def attention_fp8_exp(state, shape, out, stream=None):
    """The FP8 product with the conventional exp-then-E4M3 probability bytes."""
    B, H, N, d = shape
    _check("vca_attention_fp8_exp", lib().vca_attention_fp8_exp(
        _dev(state, torch.uint8), state.numel(), B, H, N, d, _dev(out, torch.bfloat16),
        _stream(stream)))


def attention_nvfp4(state, shape, out, stream=None):
    B, H, N, d = shape
    _check("vca_attention_nvfp4", lib().vca_attention_nvfp4(
        _dev(state, torch.uint8), state.numel(), B, H, N, d, _dev(out, torch.bfloat16),
        _stream(stream)))


def attention_bf16_ref(q, k, v, out, status=None, stream=None):
    B, H, N, d = q.shape
    _check("vca_attention_bf16_ref", lib().vca_attention_bf16_ref(
        _dev(q, torch.bfloat16), _dev(k, torch.bfloat16), _dev(v, torch.bfloat16), B, H, N, d,
        _dev(out, torch.bfloat16), _dev(status, torch.int32) if status is not None else None,
        _stream(stream)))


def get_status(state=None, status_word=None, stream=None) -> int:
    """Synchronise the stream and read-and-clear the device status word."""
    return lib().vca_get_status(_dev(state) if state is not None else None,
                                _dev(status_word) if status_word is not None else None,
                                _stream(stream))


NOALLOC_MAX_TOKENS = 32768


def kmeans_permutation_noalloc(v_head, k_clusters, labels, perm, iters=DEFAULT_ITERS,
                               seed=DEFAULT_SEED, b=0, h=0, H=1, stream=None):
    """Grouping of one head without a state blob (scratch inside the library).
    Its device status word is read with noalloc_status()."""
    N, d = v_head.shape
    if d != 128 or labels.numel() < N or perm.numel() < N:
        raise VcaError("vca_kmeans_permutation_noalloc", -1 if d == 128 else -2)
    _check("vca_kmeans_permutation_noalloc", lib().vca_kmeans_permutation_noalloc(
        _dev(v_head, torch.bfloat16), N, d, k_clusters, iters, seed, b, h, H,
        _dev(labels, torch.int32), _dev(perm, torch.int32), _stream(stream)))


def noalloc_status(stream=None) -> int:
    """Synchronise the stream and read-and-clear the status word of the
    allocation-free grouping call on the current device."""
    return lib().vca_get_status(None, None, _stream(stream))


def debug_expcast(acc, a, b, out, stream=None):
    _check("vca_debug_expcast", lib().vca_debug_expcast(
        _dev(acc, torch.float32), _dev(a, torch.float32), _dev(b, torch.float32),
        _dev(out, torch.uint8), acc.numel(), _stream(stream)))


def debug_expcast_rows(s, a, M, valid, codes, Mn, stream=None):
    """The attention softmax's per-row ExpCast step on rows of 128 scores."""
    _check("vca_debug_expcast_rows", lib().vca_debug_expcast_rows(
        _dev(s, torch.float32), _dev(a, torch.float32), _dev(M, torch.float32),
        _dev(valid, torch.int32), _dev(codes, torch.uint8), _dev(Mn, torch.float32),
        s.numel() // 128, _stream(stream)))


def debug_wait_timeout(mode, limit_ns, status, out, stream=None):
    """A CTA whose barriers are never arrived at (the bounded waits' failure path)."""
    _check("vca_debug_wait_timeout", lib().vca_debug_wait_timeout(
        mode, limit_ns, _dev(status, torch.int32), _dev(out, torch.int64), _stream(stream)))


def debug_encode(x, out_e4m3, out_e2m1, stream=None):
    _check("vca_debug_encode", lib().vca_debug_encode(
        _dev(x, torch.float32), _dev(out_e4m3, torch.uint8), _dev(out_e2m1, torch.uint8),
        x.numel(), _stream(stream)))


def debug_mma(mode, a, b, d, stream=None):
    _check("vca_debug_mma", lib().vca_debug_mma(mode, _dev(a), _dev(b), _dev(d, torch.float32),
                                                _stream(stream)))


# ----------------------------------------------------------------------------
def scale_tile_to_rows(tile):
    """A 1024-byte scale tile (tensor-core order) as a [128 rows][8 blocks] array."""
    t = tile.reshape(*tile.shape[:-1], 2, 32, 4, 4)          # [kb/4][m%32][m/32][kb%4]
    n = t.dim()
    return t.permute(*range(n - 4), n - 2, n - 3, n - 4, n - 1).reshape(*tile.shape[:-1], 128, 8)


def state_view(state: torch.Tensor, shape, k_clusters, bits=8) -> dict:
    """Typed views of the arrays of a prepared state blob (for inspection)."""
    B, H, N, d = shape
    L = state_layout(B, H, N, d, k_clusters, bits)
    BH, nb = B * H, (N + 127) // 128
    Npad = nb * 128

    def v(off, n, dtype, shp):
        nbytes = n * torch.tensor([], dtype=dtype).element_size()
        return state[off:off + nbytes].view(dtype).view(*shp)

    out = dict(
        labels=v(L.labels, BH * N, torch.int32, (BH, N)),
        perm=v(L.perm, BH * N, torch.int32, (BH, N)),
        centroids=v(L.centroids, BH * k_clusters * d, torch.int8, (BH, k_clusters, d)),
        grid_scale=v(L.grid + 4 * BH, BH, torch.float32, (BH,)),   # k-means feature grid
        kbar=v(L.kbar, BH * d, torch.int16, (BH, d)),
        mu=v(L.mu, BH * nb * d, torch.int16, (BH, nb, d)),
        status=v(L.status, 1, torch.int32, (1,)),
    )
    if bits == 8:
        out.update(
            mside=v(L.mside, BH * ((nb + 7) // 8) * 4096, torch.int16,
                    (BH, (nb + 7) // 8, 2, 2048)),
            qhat=v(L.qhat, BH * Npad * d, torch.uint8, (BH, Npad, d)),
            sq=v(L.sq, BH * nb, torch.float32, (BH, nb)),
            khat=v(L.khat, BH * Npad * d, torch.uint8, (BH, Npad, d)),
            sk=v(L.sk, BH * nb, torch.float32, (BH, nb)),
            rhatT=v(L.rhatT, BH * d * Npad, torch.uint8, (BH, d, Npad)),
            sv=v(L.sv, BH * d, torch.float32, (BH, d)),
            mutilde=v(L.mutilde, BH * nb * d, torch.float32, (BH, nb, d)),
        )
    else:
        out.update(
            mside=v(L.mside, BH * ((nb + 3) // 4) * 2048, torch.int16,
                    (BH, (nb + 3) // 4, 2048)),
            q4=v(L.q4, BH * Npad * d // 2, torch.uint8, (BH, Npad, d // 2)),
            q4s=v(L.q4s, BH * nb * 1024, torch.uint8, (BH, nb, 1024)),
            k4=v(L.k4, BH * Npad * d // 2, torch.uint8, (BH, Npad, d // 2)),
            kr4s=v(L.kr4s, BH * nb * 2048, torch.uint8, (BH, nb, 2, 1024)),
            r4T=v(L.r4T, BH * d * Npad // 2, torch.uint8, (BH, d, Npad // 2)),
            g4=v(L.g4, BH * 4, torch.float32, (BH, 4)),
        )
    return out


def pipeline_workspace_bytes(B, H, N, d, k_clusters, bits, slots) -> int:
    return lib().vca_pipeline_workspace_bytes(B, H, N, d, k_clusters, bits, slots)


def _host(t: torch.Tensor):
    assert t.device.type == "cpu" and t.is_contiguous() and t.dtype == torch.bfloat16, \
        "expected a contiguous bf16 host tensor"
    return C.c_void_p(t.data_ptr())


class HostPipeline:
    """The serving loop's end-to-end call (vca_pipeline_*): each submit takes
    Q, K, V from host tensors (page-locked for overlap), runs the V-Smooth
    preparation and the attention of `bits`, and writes O to a host tensor;
    steps rotate over `slots` device staging slots so that copies overlap the
    compute of neighbouring steps.  O of step s is valid after wait(s) or
    flush()."""

    def __init__(self, B, H, N, d=128, k_clusters=64, bits=8, slots=4, iters=DEFAULT_ITERS,
                 seed=0, qk_hadamard=False, fp8_exp=False, stream=None, device="cuda"):
        self.shape = (B, H, N, d)
        self.bits, self.iters, self.seed = bits, iters, seed
        self.flags = (PREP_QK_HADAMARD if qk_hadamard else 0) | (PIPELINE_FP8_EXP if fp8_exp else 0)
        nb = pipeline_workspace_bytes(B, H, N, d, k_clusters, bits, slots)
        if nb == 0:
            raise VcaError("vca_pipeline_workspace_bytes", -1)
        self.workspace = torch.empty(nb, dtype=torch.uint8, device=device)
        self._stream = stream if stream is not None else torch.cuda.current_stream(device)
        self._p = C.c_void_p()
        _check("vca_pipeline_create", lib().vca_pipeline_create(
            B, H, N, d, k_clusters, bits, slots, C.c_void_p(self.workspace.data_ptr()), nb,
            C.c_void_p(self._stream.cuda_stream), C.byref(self._p)))
        self._held = {}   # step -> host tensors, kept alive until the step is waited for
        self.state = self.workspace[:state_bytes(B, H, N, d, k_clusters, bits)]

    def submit(self, q, k, v, out, reuse_perm=False, iters=None) -> int:
        for t in (q, k, v, out):
            assert tuple(t.shape) == self.shape, f"expected shape {self.shape}"
        step = C.c_int64()
        _check("vca_pipeline_submit", lib().vca_pipeline_submit(
            self._p, _host(q), _host(k), _host(v), _host(out), int(reuse_perm),
            self.iters if iters is None else iters, self.seed, self.flags, C.byref(step)))
        self._held[step.value] = (q, k, v, out)
        return step.value

    def wait(self, step):
        _check("vca_pipeline_wait", lib().vca_pipeline_wait(self._p, step))
        for s in [s for s in self._held if s <= step]:
            del self._held[s]

    def flush(self):
        _check("vca_pipeline_flush", lib().vca_pipeline_flush(self._p))
        self._held.clear()

    def close(self):
        if self._p:
            rc = lib().vca_pipeline_destroy(self._p)
            self._p = C.c_void_p()
            self._held.clear()
            _check("vca_pipeline_destroy", rc)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class VCAttention:
    """Convenience wrapper: owns a state blob for one problem shape."""

    def __init__(self, B, H, N, d=128, k_clusters=64, bits=8, iters=DEFAULT_ITERS,
                 seed=DEFAULT_SEED, device="cuda", qk_hadamard=False):
        self.shape = (B, H, N, d)
        self.k, self.bits, self.iters, self.seed = k_clusters, bits, iters, seed
        self.flags = PREP_QK_HADAMARD if qk_hadamard else 0
        self.state = alloc_state(B, H, N, d, k_clusters, bits, device)

    def prepare(self, q, k, v, reuse_perm=False, stream=None, iters=None):
        """reuse_perm: PERM_FRESH / PERM_REUSE / PERM_WARM / PERM_PLAIN (or
        False / True);
        iters overrides the Lloyd iteration count of this call (a warm start
        usually runs fewer)."""
        vsmooth_prepare(q, k, v, self.k, self.state, reuse_perm, self.bits,
                        self.iters if iters is None else iters, self.seed, stream, self.flags)

    def attention(self, out, stream=None):
        fn = attention_fp8 if self.bits == 8 else attention_nvfp4
        fn(self.state, self.shape, out, stream)

    def __call__(self, q, k, v, out=None, reuse_perm=False, stream=None):
        if out is None:
            out = torch.empty_like(q)
        self.prepare(q, k, v, reuse_perm, stream)
        self.attention(out, stream)
        return out

    def status(self, stream=None) -> int:
        return get_status(self.state, None, stream)
