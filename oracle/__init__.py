"""VC-Attention CPU oracle: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's ``cpu_baseline``
leg may import this package. It wraps the single-threaded C++ restatement of
the method in ``oracle.cpp`` (see ``oracle.h`` for what each function computes
and which passage of the paper it follows). The oracle shares no code with the
CUDA library.

Arrays cross the boundary as numpy arrays. bf16 travels as ``uint16`` bit
patterns.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None

BV = 128


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` in-tree (g++, -O2, no FMA contraction)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oracle.h"))
    ):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math",
             "-fPIC", "-shared", "-o", tmp, _SRC]
        )
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = C.CDLL(_LIB)
        _declare(_lib)
    return _lib


class HeadCfg(C.Structure):
    _fields_ = [("N", C.c_int), ("d", C.c_int), ("k", C.c_int), ("iters", C.c_int),
                ("bits", C.c_int), ("Bv", C.c_int), ("seed", C.c_uint64),
                ("b", C.c_int), ("h", C.c_int), ("H", C.c_int)]


_P = C.c_void_p


class Prep8Out(C.Structure):
    _fields_ = [(n, _P) for n in ("labels", "perm", "centroids", "grid_scale", "qhat", "sq",
                                  "khat", "sk", "kbar", "rhatT", "sv", "mu", "mutilde")]


class Prep4Out(C.Structure):
    _fields_ = [(n, _P) for n in ("labels", "perm", "centroids", "grid_scale", "q4", "q4s", "gq",
                                  "k4", "k4s", "gk", "kbar", "r4T", "r4s", "gr", "mu")]


def _declare(L):
    L.orc_bf16_to_f32.restype = C.c_float
    L.orc_bf16_to_f32.argtypes = [C.c_uint16]
    L.orc_f32_to_bf16.restype = C.c_uint16
    L.orc_f32_to_bf16.argtypes = [C.c_float]
    L.orc_e4m3_decode.restype = C.c_double
    L.orc_e4m3_decode.argtypes = [C.c_uint8]
    L.orc_e4m3_encode.restype = C.c_uint8
    L.orc_e4m3_encode.argtypes = [C.c_float]
    L.orc_e2m1_decode.restype = C.c_double
    L.orc_e2m1_decode.argtypes = [C.c_uint8]
    L.orc_e2m1_encode.restype = C.c_uint8
    L.orc_e2m1_encode.argtypes = [C.c_float]
    L.orc_e4m3_encode_array.restype = None
    L.orc_e4m3_encode_array.argtypes = [_P, _P, C.c_size_t]
    L.orc_e2m1_encode_array.restype = None
    L.orc_e2m1_encode_array.argtypes = [_P, _P, C.c_size_t]
    L.orc_expcast_code.restype = C.c_int
    L.orc_expcast_code.argtypes = [C.c_double]
    L.orc_expcast_code_f32.restype = C.c_int
    L.orc_expcast_code_f32.argtypes = [C.c_float, C.c_float, C.c_float]
    L.orc_expcast_f32_array.restype = None
    L.orc_expcast_f32_array.argtypes = [_P, _P, _P, _P, C.c_size_t]
    L.orc_kmeans_init_indices.restype = None
    L.orc_kmeans_init_indices.argtypes = [C.c_uint64, C.c_int, C.c_int, C.c_int, C.c_int,
                                          C.c_int, _P]
    L.orc_kmeans.restype = None
    L.orc_kmeans.argtypes = [_P, C.POINTER(HeadCfg), _P, _P, _P, _P]
    L.orc_kmeans_warm.restype = None
    L.orc_kmeans_warm.argtypes = [_P, C.POINTER(HeadCfg), _P, C.c_float, _P, _P, _P, _P]
    L.orc_stable_argsort.restype = None
    L.orc_stable_argsort.argtypes = [_P, C.c_int, C.c_int, _P]
    L.orc_block_demean.restype = None
    L.orc_block_demean.argtypes = [_P, C.c_int, C.c_int, C.c_int, _P, _P]
    L.orc_prepare8.restype = None
    L.orc_prepare8.argtypes = [_P, _P, _P, C.POINTER(HeadCfg), _P, C.POINTER(Prep8Out)]
    L.orc_prepare4.restype = None
    L.orc_prepare4.argtypes = [_P, _P, _P, C.POINTER(HeadCfg), _P, C.POINTER(Prep4Out)]
    L.orc_prepare8_plain.restype = None
    L.orc_prepare8_plain.argtypes = [_P, _P, _P, C.POINTER(HeadCfg), _P, C.POINTER(Prep8Out)]
    L.orc_prepare4_plain.restype = None
    L.orc_prepare4_plain.argtypes = [_P, _P, _P, C.POINTER(HeadCfg), _P, C.POINTER(Prep4Out)]
    L.orc_attention_exact.restype = None
    L.orc_attention_exact.argtypes = [_P, _P, _P, C.c_int, C.c_int, _P, C.c_int, _P]
    L.orc_attention_recurrence.restype = None
    L.orc_attention_recurrence.argtypes = [_P, _P, _P, _P, C.c_int, C.c_int, C.c_int, C.c_int,
                                           _P, C.c_int, _P]
    L.orc_attention8.restype = None
    L.orc_attention8.argtypes = [C.POINTER(Prep8Out), C.c_int, C.c_int, _P, C.c_int, _P, _P]
    L.orc_attention8_exp.restype = None
    L.orc_attention8_exp.argtypes = [C.POINTER(Prep8Out), C.c_int, C.c_int, _P, C.c_int, _P, _P]
    L.orc_prepare8_ex.restype = None
    L.orc_prepare8_ex.argtypes = [_P, _P, _P, C.POINTER(HeadCfg), _P, C.c_uint,
                                  C.POINTER(Prep8Out)]
    L.orc_prepare4_ex.restype = None
    L.orc_prepare4_ex.argtypes = [_P, _P, _P, C.POINTER(HeadCfg), _P, C.c_uint,
                                  C.POINTER(Prep4Out)]
    L.orc_prepare8_hadamard.restype = None
    L.orc_prepare8_hadamard.argtypes = [_P, _P, _P, C.POINTER(HeadCfg), _P, C.POINTER(Prep8Out)]
    L.orc_prepare4_hadamard.restype = None
    L.orc_prepare4_hadamard.argtypes = [_P, _P, _P, C.POINTER(HeadCfg), _P, C.POINTER(Prep4Out)]
    L.orc_hadamard128.restype = None
    L.orc_hadamard128.argtypes = [_P, _P]
    L.orc_prepare8_naive.restype = None
    L.orc_prepare8_naive.argtypes = [_P, _P, _P, C.POINTER(HeadCfg), C.POINTER(Prep8Out)]
    L.orc_attention4.restype = None
    L.orc_attention4.argtypes = [C.POINTER(Prep4Out), C.c_int, C.c_int, _P, C.c_int, _P, _P]


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------- formats
def bf16_to_f32(bits) -> np.ndarray:
    L = lib()
    b = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([L.orc_bf16_to_f32(int(x)) for x in b], dtype=np.float32)


def f32_to_bf16(x) -> np.ndarray:
    L = lib()
    return np.array([L.orc_f32_to_bf16(float(v)) for v in np.asarray(x, np.float32).ravel()],
                    dtype=np.uint16)


def e4m3_encode(x) -> np.ndarray:
    L = lib()
    return np.array([L.orc_e4m3_encode(float(v)) for v in np.asarray(x, np.float32).ravel()],
                    dtype=np.uint8)


def e4m3_encode_array(x) -> np.ndarray:
    x = _c(x, np.float32).ravel()
    out = np.zeros(x.size, np.uint8)
    lib().orc_e4m3_encode_array(_ptr(x), _ptr(out), x.size)
    return out


def e2m1_encode_array(x) -> np.ndarray:
    x = _c(x, np.float32).ravel()
    out = np.zeros(x.size, np.uint8)
    lib().orc_e2m1_encode_array(_ptr(x), _ptr(out), x.size)
    return out


def e4m3_decode(c) -> np.ndarray:
    L = lib()
    return np.array([L.orc_e4m3_decode(int(v)) for v in np.asarray(c, np.uint8).ravel()])


def e2m1_encode(x) -> np.ndarray:
    L = lib()
    return np.array([L.orc_e2m1_encode(float(v)) for v in np.asarray(x, np.float32).ravel()],
                    dtype=np.uint8)


def e2m1_decode(c) -> np.ndarray:
    L = lib()
    return np.array([L.orc_e2m1_decode(int(v)) for v in np.asarray(c, np.uint8).ravel()])


# ----------------------------------------------------------------- ExpCast
def expcast_code(u: float) -> int:
    return lib().orc_expcast_code(float(u))


def expcast_codes(u) -> np.ndarray:
    L = lib()
    return np.array([L.orc_expcast_code(float(v)) for v in np.asarray(u, np.float64).ravel()],
                    dtype=np.int32)


def expcast_f32(acc, a, b) -> np.ndarray:
    acc, a, b = (_c(x, np.float32).ravel() for x in (acc, a, b))
    out = np.zeros(acc.size, np.uint8)
    lib().orc_expcast_f32_array(_ptr(acc), _ptr(a), _ptr(b), _ptr(out), acc.size)
    return out


# ----------------------------------------------------------------- V-Smooth
def _cfg(N, d, k, iters, bits, seed, b, h, H, Bv=BV):
    return HeadCfg(N, d, k, iters, bits, Bv, seed, b, h, H)


def kmeans_init_indices(seed, b, h, H, N, k) -> np.ndarray:
    out = np.zeros(k, np.int32)
    lib().orc_kmeans_init_indices(seed, b, h, H, N, k, _ptr(out))
    return out


def kmeans(v_head: np.ndarray, k: int, iters: int, seed: int, b=0, h=0, H=1):
    """v_head: uint16 bf16 [N, d]. Returns (x int8 [N,d], grid_scale, labels, centroids)."""
    v = _c(v_head, np.uint16)
    N, d = v.shape
    cfg = _cfg(N, d, k, iters, 8, seed, b, h, H)
    x = np.zeros((N, d), np.int8)
    gs = np.zeros(1, np.float32)
    labels = np.zeros(N, np.int32)
    cent = np.zeros((k, d), np.int8)
    lib().orc_kmeans(_ptr(v), C.byref(cfg), _ptr(x), _ptr(gs), _ptr(labels), _ptr(cent))
    return x, float(gs[0]), labels, cent


def kmeans_warm(v_head: np.ndarray, prev_centroids: np.ndarray, prev_grid_scale: float,
                iters: int):
    """Warm-started k-means of one head from the previous step's centroids and
    grid scale.  Returns (x int8 [N,d], grid_scale, labels, centroids); with
    iters = 0 the centroids are the previous ones moved to the new grid and
    the labels are -1."""
    v = _c(v_head, np.uint16)
    N, d = v.shape
    prev = _c(prev_centroids, np.int8)
    k = prev.shape[0]
    cfg = _cfg(N, d, k, iters, 8, 0, 0, 0, 1)
    x = np.zeros((N, d), np.int8)
    gs = np.zeros(1, np.float32)
    labels = np.full(N, -1, np.int32)
    cent = np.zeros((k, d), np.int8)
    lib().orc_kmeans_warm(_ptr(v), C.byref(cfg), _ptr(prev), float(prev_grid_scale), _ptr(x),
                          _ptr(gs), _ptr(labels), _ptr(cent))
    return x, float(gs[0]), labels, cent


def stable_argsort(labels: np.ndarray, k: int) -> np.ndarray:
    z = _c(labels, np.int32)
    out = np.zeros(z.size, np.int32)
    lib().orc_stable_argsort(_ptr(z), z.size, k, _ptr(out))
    return out


def block_demean(vperm_bf16: np.ndarray, Bv: int):
    v = _c(vperm_bf16, np.uint16)
    N, d = v.shape
    nb = (N + Bv - 1) // Bv
    mu = np.zeros((nb, d), np.uint16)
    r = np.zeros((nb * Bv, d), np.float32)
    lib().orc_block_demean(_ptr(v), N, d, Bv, _ptr(mu), _ptr(r))
    return mu, r


def _opts(plain, naive, hadamard) -> int:
    """Option bits of orc_prepare8_ex / orc_prepare4_ex."""
    return (1 if plain else 0) | (2 if naive else 0) | (4 if hadamard else 0)


def hadamard128(x: np.ndarray) -> np.ndarray:
    """The QK Hadamard rotation of each 128-channel row of x (fp32)."""
    x = _c(x, np.float32).reshape(-1, 128)
    y = np.empty_like(x)
    for i in range(x.shape[0]):
        lib().orc_hadamard128(_ptr(x[i]), _ptr(y[i]))
    return y


def prepare8(q, k, v, k_clusters, iters, seed, b=0, h=0, H=1, perm=None, plain=False,
             naive=False, hadamard=False) -> dict:
    """One head, inputs uint16 bf16 [N, d]. Returns a dict of numpy arrays.
    plain: a step after the grouping window (needs perm): no block demeaning.
    naive: the comparison preparation that smooths nothing (sequence order, no
    key centring, no demeaning); labels stay -1."""
    if plain and perm is None:
        raise ValueError("the plain preparation needs the permutation")
    q, k, v = (_c(x, np.uint16) for x in (q, k, v))
    N, d = q.shape
    nb = (N + BV - 1) // BV
    Npad = nb * BV
    o = dict(labels=np.full(N, -1, np.int32), perm=np.zeros(N, np.int32),
             centroids=np.zeros((k_clusters, d), np.int8), grid_scale=np.zeros(1, np.float32),
             qhat=np.zeros((Npad, d), np.uint8), sq=np.zeros(nb, np.float32),
             khat=np.zeros((Npad, d), np.uint8), sk=np.zeros(nb, np.float32),
             kbar=np.zeros(d, np.uint16), rhatT=np.zeros((d, Npad), np.uint8),
             sv=np.zeros(d, np.float32), mu=np.zeros((nb, d), np.uint16),
             mutilde=np.zeros((nb, d), np.float32))
    st = Prep8Out(*[_ptr(o[n]) for n, _ in Prep8Out._fields_])
    cfg = _cfg(N, d, k_clusters, iters, 8, seed, b, h, H)
    keep = _c(perm, np.int32) if perm is not None else None
    lib().orc_prepare8_ex(_ptr(q), _ptr(k), _ptr(v), C.byref(cfg),
                          _ptr(keep) if keep is not None else None,
                          _opts(plain, naive, hadamard), C.byref(st))
    o["N"], o["d"], o["_struct"] = N, d, st
    return o


def prepare4(q, k, v, k_clusters, iters, seed, b=0, h=0, H=1, perm=None, plain=False,
             naive=False, hadamard=False) -> dict:
    if plain and perm is None:
        raise ValueError("the plain preparation needs the permutation")
    q, k, v = (_c(x, np.uint16) for x in (q, k, v))
    N, d = q.shape
    nb = (N + BV - 1) // BV
    Npad = nb * BV
    o = dict(labels=np.full(N, -1, np.int32), perm=np.zeros(N, np.int32),
             centroids=np.zeros((k_clusters, d), np.int8), grid_scale=np.zeros(1, np.float32),
             q4=np.zeros((Npad, d), np.uint8), q4s=np.zeros((Npad, d // 16), np.uint8),
             gq=np.zeros(1, np.float32),
             k4=np.zeros((Npad, d), np.uint8), k4s=np.zeros((Npad, d // 16), np.uint8),
             gk=np.zeros(1, np.float32), kbar=np.zeros(d, np.uint16),
             r4T=np.zeros((d, Npad), np.uint8), r4s=np.zeros((d, Npad // 16), np.uint8),
             gr=np.zeros(1, np.float32), mu=np.zeros((nb, d), np.uint16))
    st = Prep4Out(*[_ptr(o[n]) for n, _ in Prep4Out._fields_])
    cfg = _cfg(N, d, k_clusters, iters, 4, seed, b, h, H)
    keep = _c(perm, np.int32) if perm is not None else None
    lib().orc_prepare4_ex(_ptr(q), _ptr(k), _ptr(v), C.byref(cfg),
                          _ptr(keep) if keep is not None else None,
                          _opts(plain, naive, hadamard), C.byref(st))
    o["N"], o["d"], o["_struct"] = N, d, st
    return o


# ----------------------------------------------------------------- attention
def _rows(rows, N):
    return _c(np.arange(N) if rows is None else rows, np.int32)


def attention_exact(q, k, v, rows=None) -> np.ndarray:
    q, k, v = (_c(x, np.uint16) for x in (q, k, v))
    N, d = q.shape
    r = _rows(rows, N)
    out = np.zeros((r.size, d), np.float64)
    lib().orc_attention_exact(_ptr(q), _ptr(k), _ptr(v), N, d, _ptr(r), r.size, _ptr(out))
    return out


def attention_recurrence(q, kp, r, mu, Bv, pmode, rows=None) -> np.ndarray:
    q, kp, r, mu = (_c(x, np.float64) for x in (q, kp, r, mu))
    N, d = kp.shape
    rr = _rows(rows, q.shape[0])
    out = np.zeros((rr.size, d), np.float64)
    lib().orc_attention_recurrence(_ptr(q), _ptr(kp), _ptr(r), _ptr(mu), N, d, Bv, pmode,
                                   _ptr(rr), rr.size, _ptr(out))
    return out


def attention8(prep: dict, rows=None, expcast=True):
    """Returns (bf16 bits [nrows, d], fp64 values before rounding).
    expcast=False: the conventional exponential-then-E4M3-cast bytes."""
    N, d = prep["N"], prep["d"]
    r = _rows(rows, N)
    out = np.zeros((r.size, d), np.uint16)
    out64 = np.zeros((r.size, d), np.float64)
    fn = lib().orc_attention8 if expcast else lib().orc_attention8_exp
    fn(C.byref(prep["_struct"]), N, d, _ptr(r), r.size, _ptr(out), _ptr(out64))
    return out, out64


def attention4(prep: dict, rows=None):
    N, d = prep["N"], prep["d"]
    r = _rows(rows, N)
    out = np.zeros((r.size, d), np.uint16)
    out64 = np.zeros((r.size, d), np.float64)
    lib().orc_attention4(C.byref(prep["_struct"]), N, d, _ptr(r), r.size, _ptr(out), _ptr(out64))
    return out, out64
