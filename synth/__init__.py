"""Seeded synthetic Q, K, V for the VC-Attention workloads (see ``synth.c``).

The module holds no arithmetic of the method: it only builds the bf16 inputs
that both the CUDA library and the CPU oracle consume. Shapes follow the
paper's video-DiT settings (Appx A: Wan2.2 720p is 21x45x80 = 75600 tokens,
head dimension 128, 40 heads); the captured tensors themselves are not
available, so these distributions stand in for them.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "_build", "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = C.CDLL(_LIB)
        P = C.c_void_p
        _lib.synth_qk.argtypes = [P, C.c_int, C.c_int, C.c_int, C.c_int, C.c_uint64, C.c_int]
        _lib.synth_v.argtypes = [P, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_uint64]
        _lib.synth_v_labels.argtypes = [P, P, C.c_int, C.c_int, C.c_int, C.c_int, C.c_uint64,
                                        C.c_int, C.c_int]
    return _lib


@dataclass(frozen=True)
class Workload:
    """One benchmark / parity configuration."""
    name: str
    B: int
    H: int
    N: int
    d: int
    clusters: int     # Gaussian clusters in V
    k: int            # k-means clusters
    bits: int         # 8 or 4
    seed: int

    @property
    def flops(self) -> float:
        """Attention FLOPs counted as 4 B H N^2 d (two N x N x d products)."""
        return 4.0 * self.B * self.H * self.N * self.N * self.d


# The five configurations of the workload list; the seeds are 0xC0FFEE + id.
CONFIGS = {
    "pr1": Workload("pr1_B1_H1_N1024", 1, 1, 1024, 128, 16, 16, 8, 0xC0FFEE + 1),
    "h8": Workload("h8_B1_H8_N8192", 1, 8, 8192, 128, 32, 32, 8, 0xC0FFEE + 2),
    "wan720p": Workload("wan720p_B1_H40_N75600", 1, 40, 75600, 128, 64, 64, 8, 0xC0FFEE + 3),
    "sweep16k": Workload("sweep_B1_H24_N16384", 1, 24, 16384, 128, 64, 64, 8, 0xC0FFEE + 4),
    "sweep32k": Workload("sweep_B1_H24_N32768", 1, 24, 32768, 128, 64, 64, 8, 0xC0FFEE + 4),
    "sweep64k": Workload("sweep_B1_H24_N65536", 1, 24, 65536, 128, 64, 64, 8, 0xC0FFEE + 4),
    "sweep128k": Workload("sweep_B1_H24_N131072", 1, 24, 131072, 128, 64, 64, 8, 0xC0FFEE + 4),
    "wan720p_fp4": Workload("wan720p_nvfp4_B1_H40_N75600", 1, 40, 75600, 128, 64, 64, 4,
                            0xC0FFEE + 5),
    "sweep16k_fp4": Workload("sweep_nvfp4_B1_H24_N16384", 1, 24, 16384, 128, 64, 64, 4,
                             0xC0FFEE + 5),
}


def make_qkv(B, H, N, d, clusters, seed, out=None):
    """Return (q, k, v) as uint16 bf16 bit arrays of shape [B, H, N, d].

    ``out`` may be a tuple of three preallocated uint16 arrays (e.g. views of
    pinned host tensors) to fill in place.
    """
    L = lib()
    if out is None:
        out = tuple(np.empty((B, H, N, d), np.uint16) for _ in range(3))
    q, k, v = out
    for a in out:
        assert a.dtype == np.uint16 and a.flags["C_CONTIGUOUS"] and a.size == B * H * N * d
    L.synth_qk(q.ctypes.data_as(C.c_void_p), B, H, N, d, seed, 0)
    L.synth_qk(k.ctypes.data_as(C.c_void_p), B, H, N, d, seed, 1)
    L.synth_v(v.ctypes.data_as(C.c_void_p), B, H, N, d, clusters, seed)
    return q, k, v


def make(w: Workload, out=None):
    return make_qkv(w.B, w.H, w.N, w.d, w.clusters, w.seed, out=out)


def v_labels(B, H, N, clusters, seed, b, h):
    """Ground-truth cluster label and outlier flag of each token of one head."""
    L = lib()
    lab = np.zeros(N, np.int32)
    out = np.zeros(N, np.uint8)
    L.synth_v_labels(lab.ctypes.data_as(C.c_void_p), out.ctypes.data_as(C.c_void_p), B, H, N,
                     clusters, seed, b, h)
    return lab, out.astype(bool)
