"""TEST INFRASTRUCTURE ONLY -- the fp64 CPU oracle for MLA decode attention.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package. The product path (the CUDA library and its binding)
never touches it.

The arithmetic lives in ``mla_oracle.c`` (plain C, fp64, single-threaded). This
module compiles it with gcc on first use and exposes numpy-friendly wrappers.
What it computes is the problem statement and naive reference of
kernelbot-amd-mixed-mla-675627 ("MLA decode kernel -- submission template"):
segmented ``softmax(q . k^T * sm_scale) . v`` with K = all 576 KV dims and
V = the first 512, over the dequantised KV cache.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

BF16, FP8_E4M3, MXFP4 = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/liboracle.so (gcc, -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
             "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.orc_decode_array.argtypes = [ctypes.c_int, i64, P, P, P]
            lib.orc_decode_array.restype = ctypes.c_int
            lib.orc_attention_f64.argtypes = [P, P, P, P, ctypes.c_int, i64, i64, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, dbl, P, P]
            lib.orc_attention_f64.restype = ctypes.c_int
            lib.orc_mla_decode.argtypes = [P, ctypes.c_int, P, P, ctypes.c_int, P, P, P, ctypes.c_int,
                                           i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, dbl,
                                           i64, P, P, P, P]
            lib.orc_mla_decode.restype = ctypes.c_int
            lib.orc_lse_combine.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P, P]
            lib.orc_lse_combine.restype = None
            del i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def decode_array(kind: str, codes, params=None) -> np.ndarray:
    """Decode raw codes to float64. kind: 'bf16' (uint16 bits), 'e4m3fn', 'e2m1'
    (one nibble per byte), 'e8m0', or 'minifloat' with params=(ebits, mbits, bias)
    and uint32 codes."""
    kinds = {"bf16": (0, np.uint16), "e4m3fn": (1, np.uint8), "e2m1": (2, np.uint8),
             "e8m0": (3, np.uint8), "minifloat": (4, np.uint32)}
    k, dt = kinds[kind]
    src = _c(codes, dt).reshape(-1)
    dst = np.empty(src.size, dtype=np.float64)
    prm = None if params is None else _c(params, np.int32)
    rc = _load().orc_decode_array(k, src.size, _ptr(src), _ptr(dst), _ptr(prm))
    if rc != 0:
        raise ValueError(f"orc_decode_array rc={rc}")
    return dst.reshape(np.shape(codes))


def attention_f64(q, kv, qo_indptr, kv_indptr, sm_scale, dv, want_lse=False):
    """Segmented attention over decoded float64 arrays.
    q: [total_q, H, D], kv: [total_kv, D]; returns out [total_q, H, dv] (and lse [total_q, H])."""
    q = _c(q, np.float64)
    kv = _c(kv, np.float64)
    qo = _c(qo_indptr, np.int32)
    kvp = _c(kv_indptr, np.int32)
    total_q, H, D = q.shape
    total_kv = kv.shape[0]
    assert kv.ndim == 2 and (kv.shape[1] == D or total_kv == 0)
    out = np.empty((total_q, H, dv), dtype=np.float64)
    lse = np.empty((total_q, H), dtype=np.float64)
    rc = _load().orc_attention_f64(_ptr(q), _ptr(kv), _ptr(qo), _ptr(kvp), qo.size - 1, total_q,
                                   total_kv, H, D, dv, float(sm_scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"orc_attention_f64 rc={rc}")
    return (out, lse) if want_lse else out


def mla_decode(q, q_dtype, q_scale, kv, kv_dtype, kv_scale, qo_indptr, kv_indptr, *, heads, dqk,
               dv, sm_scale, rows=None, want_lse=False):
    """The full decode from raw encodings (numpy arrays of codes).

    q: uint16 bf16 bits [total_q, heads, dqk] or uint8 e4m3 codes (q_dtype=FP8_E4M3 with
    q_scale a float); kv: uint16 [total_kv, dqk] (BF16), uint8 [total_kv, dqk] (FP8_E4M3, kv_scale
    float) or uint8 [total_kv, dqk/2] (MXFP4, kv_scale uint8 [total_kv, dqk/32]).
    rows: optional (tokens, heads) index arrays -> out [n, dv]; else out [total_q, heads, dv]."""
    lib = _load()
    qo = _c(qo_indptr, np.int32)
    kvp = _c(kv_indptr, np.int32)
    batch = qo.size - 1
    qa = _c(q, np.uint16 if q_dtype == BF16 else np.uint8)
    total_q = qa.shape[0] if qa.ndim else 0
    kv_dt = np.uint16 if kv_dtype == BF16 else np.uint8
    kva = _c(kv, kv_dt)
    total_kv = kva.shape[0]
    qs = None if q_dtype == BF16 else _c([q_scale], np.float32)
    if kv_dtype == BF16:
        ks = None
    elif kv_dtype == FP8_E4M3:
        ks = _c([kv_scale], np.float32)
    else:
        ks = _c(kv_scale, np.uint8)
    if rows is None:
        n_rows, rt, rh = -1, None, None
        out = np.empty((total_q, heads, dv), dtype=np.float64)
        lse = np.empty((total_q, heads), dtype=np.float64)
    else:
        rt = _c(rows[0], np.int32)
        rh = _c(rows[1], np.int32)
        n_rows = rt.size
        out = np.empty((n_rows, dv), dtype=np.float64)
        lse = np.empty((n_rows,), dtype=np.float64)
    rc = lib.orc_mla_decode(_ptr(qa), q_dtype, _ptr(qs), _ptr(kva), kv_dtype, _ptr(ks), _ptr(qo),
                            _ptr(kvp), batch, total_q, total_kv, heads, dqk, dv, float(sm_scale),
                            n_rows, _ptr(rt), _ptr(rh), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"orc_mla_decode rc={rc}")
    return (out, lse) if want_lse else out


def lse_combine(o, lse):
    """Merge per-split (normalised output, natural-log LSE) pairs of one query row."""
    o = _c(o, np.float64)
    lse = _c(lse, np.float64)
    nsplit, dv = o.shape
    out = np.empty(dv, dtype=np.float64)
    lse_out = np.empty(1, dtype=np.float64)
    _load().orc_lse_combine(nsplit, dv, _ptr(o), _ptr(lse), _ptr(out), _ptr(lse_out))
    return out, float(lse_out[0])


def paged_rows(kv_pages, page_indptr, page_indices, last_page_len, page_size):
    """The KV rows a page table names, laid out contiguously, with their row offsets.

    The page-table form is that of kernelbot-amd-mixed-mla-753817, which hands
    ``kv_indices``, ``kv_last_page_len`` and ``page_size`` to the vendor a8w8
    decode: segment b owns table entries [page_indptr[b], page_indptr[b+1]);
    its row i is row i % page_size of page page_indices[page_indptr[b] + i // page_size].
    A segment of n > 0 pages has (n - 1) * page_size + last_page_len[b] rows; with
    page_size 1 it has n rows (the pages pass the segment lengths as
    ``kv_last_page_len`` there, which only this reading accepts).

    kv_pages: [num_pages, page_size, ...]; returns (rows [total, ...], kv_indptr [batch + 1]).
    Pure index work, written as plain loops."""
    pages = np.asarray(kv_pages)
    pip = [int(x) for x in np.asarray(page_indptr).reshape(-1)]
    idx = [int(x) for x in np.asarray(page_indices).reshape(-1)]
    batch = len(pip) - 1
    assert pip[0] == 0 and all(pip[b + 1] >= pip[b] for b in range(batch))
    rows, kv_indptr = [], [0]
    for b in range(batch):
        n = pip[b + 1] - pip[b]
        if n == 0:
            length = 0
        elif page_size == 1:
            length = n
        else:
            last = int(np.asarray(last_page_len).reshape(-1)[b])
            assert 1 <= last <= page_size
            length = (n - 1) * page_size + last
        for i in range(length):
            page = idx[pip[b] + i // page_size]
            assert 0 <= page < pages.shape[0]
            rows.append(pages[page, i % page_size])
        kv_indptr.append(kv_indptr[-1] + length)
    shape = (0,) + pages.shape[2:]
    out = np.stack(rows) if rows else np.zeros(shape, dtype=pages.dtype)
    return out, np.asarray(kv_indptr, dtype=np.int32)
