"""Timing of the CPU oracle for the benchmark's ``cpu_baseline`` leg and its
reference arm: TEST INFRASTRUCTURE ONLY (the oracle is never on the product
path).

``head_sample`` runs one head of a workload through the oracle as it stands:
the full preparation (a fresh grouping with ``iters`` Lloyd iterations) and
``rows`` attention rows.  It is a module-level function so that a ``spawn``
process pool can run one head per host core.
"""
from __future__ import annotations

import time

import numpy as np


def head_sample(task):
    """task = (N, d, clusters, seed, k, iters, bits, rows, seed_rows).
    Returns (seconds of the preparation, seconds of the rows)."""
    import oracle
    import synth
    N, d, clusters, seed, k, iters, bits, rows, seed_rows = task
    q, kk, v = synth.make_qkv(1, 1, N, d, clusters, seed)
    prepare, attention = ((oracle.prepare8, oracle.attention8) if bits == 8
                          else (oracle.prepare4, oracle.attention4))
    t0 = time.perf_counter()
    p = prepare(q[0, 0], kk[0, 0], v[0, 0], k, iters, 0, b=0, h=0, H=1)
    t_prep = time.perf_counter() - t0
    r = np.random.default_rng(seed_rows).choice(N, rows, replace=False)
    t0 = time.perf_counter()
    attention(p, r)
    return t_prep, time.perf_counter() - t0
