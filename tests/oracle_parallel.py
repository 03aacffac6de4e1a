"""The fp64 oracle over every segment of a workload, on all host cores.

Test infrastructure only. The oracle's C code is single-threaded and keeps no
global state, and ctypes releases the GIL while a call runs, so a pool of
threads decodes whole segments side by side. Segments are independent in the
method (each token attends only to its own segment's KV rows), so the output
of a segment equals what one oracle call over the whole batch gives for its
tokens.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle


def decode_segments(h: dict, sm_scale: float, heads: int = 16, dqk: int = 576, dv: int = 512,
                    workers: int | None = None) -> np.ndarray:
    """h: raw host codes as synth.to_host_codes() returns them. Returns out [total_q, heads, dv] (fp64)."""
    qo = np.asarray(h["qo_indptr"], np.int64)
    kvp = np.asarray(h["kv_indptr"], np.int64)
    batch = qo.size - 1
    out = np.zeros((int(qo[-1]), heads, dv), np.float64)

    def one(b: int) -> None:
        q0, q1, k0, k1 = int(qo[b]), int(qo[b + 1]), int(kvp[b]), int(kvp[b + 1])
        if q1 == q0:
            return
        ks = h["kv_scale"][k0:k1] if h["kv_dtype"] == oracle.MXFP4 else h["kv_scale"]
        out[q0:q1] = oracle.mla_decode(h["q"][q0:q1], h["q_dtype"], h["q_scale"], h["kv"][k0:k1], h["kv_dtype"], ks,
                                       np.array([0, q1 - q0], np.int32), np.array([0, k1 - k0], np.int32),
                                       heads=heads, dqk=dqk, dv=dv, sm_scale=sm_scale)

    order = sorted(range(batch), key=lambda b: -(int(kvp[b + 1] - kvp[b]) * int(qo[b + 1] - qo[b])))
    with ThreadPoolExecutor(max_workers=workers or max(1, os.cpu_count() or 1)) as ex:
        list(ex.map(one, order))
    return out


def per_segment_rel_l2(got: np.ndarray, ref: np.ndarray, qo_indptr) -> np.ndarray:
    """||got_b - ref_b||_2 / ||ref_b||_2 for every segment b with tokens (nan for segments without)."""
    qo = np.asarray(qo_indptr, np.int64)
    rel = np.full(qo.size - 1, np.nan)
    for b in range(qo.size - 1):
        g, r = got[qo[b]:qo[b + 1]], ref[qo[b]:qo[b + 1]]
        if g.size:
            n = np.linalg.norm(r)
            rel[b] = np.linalg.norm(g - r) / n if n > 0 else np.linalg.norm(g)
    return rel
