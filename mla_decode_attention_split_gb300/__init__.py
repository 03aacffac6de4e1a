"""GB300 (sm_103a) MLA decode: Python binding of the C-ABI library.

Every function here only marshals arguments to ``libmla_decode.so`` (declared
in ``include/mla_decode.h``); all computation runs in the library's CUDA
kernels. PyTorch is used for device memory and streams only. There is no CPU
fallback: if the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

# Sizes and storage-format codes of mla_decode.h (MLA_NUM_HEADS, MLA_D_QK,
# MLA_D_V, MLA_MX_BLOCK; mla_dtype_t).
HEADS, D_QK, D_V, MX_BLOCK = 16, 576, 512, 32
BF16, FP8_E4M3, MXFP4 = 0, 1, 2

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmla_decode.so")

MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_WORKSPACE = 0, 1, 2, 3
MLA_ERR_CUDA, MLA_ERR_TIMEOUT, MLA_ERR_DEVICE_CHECK = 4, 5, 6
DEVFLAG_TIMEOUT, DEVFLAG_BAD_INDPTR = 0x1, 0x2

EXPORTED = ("mla_plan", "mla_decode_workspace_size", "mla_decode", "mla_decode_from_host", "mla_dequant_rows",
            "mla_get_device_error", "mla_reset_device_error", "mla_event_elapsed_ms", "mla_decode_static_workspace",
            "mla_decode_paged_workspace_size", "mla_decode_paged", "mla_decode_pairs_workspace_size",
            "mla_decode_group_workspace_size",
            "mla_validate_inputs", "mla_static_workspace_device_error", "mla_status_string")
DEVFLAG_BAD_PAGE = 0x4
MLA_ERR_TOO_LARGE = 7
STATIC_WORKSPACE_BYTES = 16 * 1024 * 1024


class MlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


class DecodeOpts(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("total_q", ctypes.c_int32), ("total_kv", ctypes.c_int32),
                ("sm_scale", ctypes.c_float), ("q_dtype", ctypes.c_int), ("q_scale", ctypes.c_void_p),
                ("num_splits", ctypes.c_int32), ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("profile_events", ctypes.c_void_p * 3), ("quantize_q", ctypes.c_int32),
                ("token_group", ctypes.c_int32)]


class DeviceBuffers(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("kv", ctypes.c_void_p), ("kv_scale", ctypes.c_void_p),
                ("q_scale", ctypes.c_void_p), ("qo_indptr", ctypes.c_void_p), ("kv_indptr", ctypes.c_void_p),
                ("out", ctypes.c_void_p)]


class PagedKV(ctypes.Structure):
    _fields_ = [("page_indptr", ctypes.c_void_p), ("page_indices", ctypes.c_void_p),
                ("last_page_len", ctypes.c_void_p), ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return LIB_PATH


def lib():
    """The loaded CUDA library (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -m mla_decode_attention_split_gb300.build` (no CPU fallback exists)")
            L = ctypes.CDLL(LIB_PATH)
            P, i32, st = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int
            L.mla_plan.argtypes = [i32, i32, i32, st, i32, ctypes.POINTER(i32)]
            L.mla_decode_workspace_size.argtypes = [i32, i32, i32, st, i32, ctypes.POINTER(ctypes.c_size_t)]
            L.mla_decode.argtypes = [P, P, P, P, P, P, st, ctypes.POINTER(DecodeOpts), P]
            L.mla_decode_from_host.argtypes = [P, P, P, P, P, P, P, st, ctypes.POINTER(DecodeOpts),
                                               ctypes.POINTER(DeviceBuffers), P]
            L.mla_dequant_rows.argtypes = [P, P, st, i32, i32, i32, P, P]
            L.mla_get_device_error.argtypes = [P, P, ctypes.POINTER(ctypes.c_uint32)]
            L.mla_reset_device_error.argtypes = [P, P]
            L.mla_event_elapsed_ms.argtypes = [P, P, ctypes.POINTER(ctypes.c_float)]
            L.mla_decode_static_workspace.argtypes = [P, P, P, P, P, P, st, ctypes.POINTER(DecodeOpts), P]
            L.mla_decode_paged_workspace_size.argtypes = [i32, i32, i32, st, i32, ctypes.POINTER(ctypes.c_size_t)]
            L.mla_decode_pairs_workspace_size.argtypes = [i32, i32, i32, st, i32, ctypes.POINTER(ctypes.c_size_t)]
            L.mla_decode_group_workspace_size.argtypes = [i32, i32, i32, st, i32, i32,
                                                          ctypes.POINTER(ctypes.c_size_t)]
            L.mla_decode_paged.argtypes = [P, P, P, P, ctypes.POINTER(PagedKV), P, st, ctypes.POINTER(DecodeOpts), P]
            L.mla_validate_inputs.argtypes = [P, P, i32, i32, i32, st, P, P, ctypes.POINTER(ctypes.c_int64)]
            L.mla_static_workspace_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
            L.mla_status_string.argtypes = [st]
            L.mla_status_string.restype = ctypes.c_char_p
            for name in EXPORTED[:-1]:
                getattr(L, name).restype = st
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().mla_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != MLA_OK:
        raise MlaError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(getattr(stream, "cuda_stream", stream) or 0)


def plan(batch: int, total_q: int, total_kv: int, kv_dtype: int, sm_count: int = 0) -> int:
    """Number of KV partitions (stage-1 CTAs) the library would use."""
    out = ctypes.c_int32(0)
    _check(lib().mla_plan(batch, total_q, total_kv, kv_dtype, sm_count, ctypes.byref(out)), "mla_plan")
    return out.value


def workspace_size(batch: int, total_q: int, total_kv: int, kv_dtype: int, num_splits: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().mla_decode_workspace_size(batch, total_q, total_kv, kv_dtype, num_splits, ctypes.byref(out)),
           "mla_decode_workspace_size")
    return out.value


def alloc_workspace(batch: int, total_q: int, total_kv: int, kv_dtype: int, num_splits: int = 0, device="cuda"):
    """A zeroed device workspace (torch uint8 tensor, 256-byte aligned by the caching allocator)."""
    import torch
    n = workspace_size(batch, total_q, total_kv, kv_dtype, num_splits)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def make_opts(batch, total_q, total_kv, *, q_dtype=BF16, q_scale=None, sm_scale=0.0, num_splits=0,
              workspace=None, events=None, quantize_q=False, token_pairs=False, token_group=0) -> DecodeOpts:
    """token_group: query tokens per KV pass (0/1, 2, 4); token_pairs=True is token_group=2."""
    o = DecodeOpts(batch=batch, total_q=total_q, total_kv=total_kv, sm_scale=float(sm_scale), q_dtype=q_dtype,
                   q_scale=None if q_scale is None else q_scale.data_ptr(), num_splits=num_splits,
                   workspace=None if workspace is None else workspace.data_ptr(),
                   workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size(),
                   quantize_q=1 if quantize_q else 0,
                   token_group=int(token_group) if token_group else (2 if token_pairs else 0))
    if events is not None:  # three torch.cuda.Event(enable_timing=True)
        for i, ev in enumerate(events):
            if ev is not None and not ev.cuda_event:
                ev.record()  # torch creates the CUDA event on its first record
            o.profile_events[i] = None if ev is None else ev.cuda_event
    return o


def decode(q, kv, kv_scale, qo_indptr, kv_indptr, out, kv_dtype: int, *, workspace, q_dtype: int = BF16,
           q_scale=None, sm_scale: float = 0.0, num_splits: int = 0, stream=None, events=None,
           quantize_q: bool = False, token_pairs: bool = False, token_group: int = 0) -> None:
    """mla_decode() on torch CUDA tensors (layouts as in mla_decode.h). Asynchronous.
    events: optional three CUDA events recorded before and after the launch (1 and 2 back to back).
    quantize_q: quantise bf16 q to e4m3 per tensor inside the call (the a8w8 mode; fp8 KV only).
    token_group: a segment's query tokens share each pass over its KV rows in groups of 2 (fp8 or
    bf16 KV) or 4 (fp8 KV, fp8 q or quantize_q); the workspace comes from group_workspace_size.
    token_pairs=True is token_group=2."""
    opts = make_opts(qo_indptr.numel() - 1, q.shape[0], kv.shape[0], q_dtype=q_dtype, q_scale=q_scale,
                     sm_scale=sm_scale, num_splits=num_splits, workspace=workspace, events=events,
                     quantize_q=quantize_q, token_pairs=token_pairs, token_group=token_group)
    _check(lib().mla_decode(_ptr(q), _ptr(kv), _ptr(kv_scale), _ptr(qo_indptr), _ptr(kv_indptr), _ptr(out),
                            kv_dtype, ctypes.byref(opts), _stream_handle(stream)), "mla_decode")


def pairs_workspace_size(batch: int, total_q: int, total_kv: int, kv_dtype: int, num_splits: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().mla_decode_pairs_workspace_size(batch, total_q, total_kv, kv_dtype, num_splits, ctypes.byref(out)),
           "mla_decode_pairs_workspace_size")
    return out.value


def group_workspace_size(batch: int, total_q: int, total_kv: int, kv_dtype: int, token_group: int,
                         num_splits: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().mla_decode_group_workspace_size(batch, total_q, total_kv, kv_dtype, num_splits, token_group,
                                                 ctypes.byref(out)), "mla_decode_group_workspace_size")
    return out.value


def alloc_group_workspace(batch: int, total_q: int, total_kv: int, kv_dtype: int, token_group: int,
                          num_splits: int = 0, device="cuda"):
    """A zeroed device workspace for decode(..., token_group=token_group)."""
    import torch
    n = group_workspace_size(batch, total_q, total_kv, kv_dtype, token_group, num_splits)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def alloc_pairs_workspace(batch: int, total_q: int, total_kv: int, kv_dtype: int, num_splits: int = 0,
                          device="cuda"):
    """A zeroed device workspace for decode(..., token_pairs=True)."""
    import torch
    n = pairs_workspace_size(batch, total_q, total_kv, kv_dtype, num_splits)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def paged_workspace_size(batch: int, total_q: int, total_kv: int, kv_dtype: int, num_splits: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().mla_decode_paged_workspace_size(batch, total_q, total_kv, kv_dtype, num_splits, ctypes.byref(out)),
           "mla_decode_paged_workspace_size")
    return out.value


def alloc_paged_workspace(batch: int, total_q: int, total_kv: int, kv_dtype: int, num_splits: int = 0,
                          device="cuda"):
    """A zeroed device workspace for decode_paged (torch uint8 tensor)."""
    import torch
    n = paged_workspace_size(batch, total_q, total_kv, kv_dtype, num_splits)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def decode_paged(q, kv_pages, kv_scale, qo_indptr, page_indptr, page_indices, last_page_len, page_size: int,
                 out, kv_dtype: int, *, total_kv: int, workspace, q_dtype: int = BF16, q_scale=None,
                 sm_scale: float = 0.0, num_splits: int = 0, stream=None, events=None,
                 quantize_q: bool = False) -> None:
    """mla_decode_paged() on torch CUDA tensors: kv_pages is [num_pages][page_size][576] e4m3 codes (uint8),
    the page table is int32 (last_page_len may be None when page_size == 1); total_kv is the logical row count
    (sum of the segment lengths). Asynchronous."""
    opts = make_opts(qo_indptr.numel() - 1, q.shape[0], total_kv, q_dtype=q_dtype, q_scale=q_scale,
                     sm_scale=sm_scale, num_splits=num_splits, workspace=workspace, events=events,
                     quantize_q=quantize_q)
    pg = PagedKV(page_indptr=page_indptr.data_ptr(), page_indices=page_indices.data_ptr(),
                 last_page_len=None if last_page_len is None else last_page_len.data_ptr(),
                 page_size=int(page_size), num_pages=int(kv_pages.shape[0]))
    _check(lib().mla_decode_paged(_ptr(q), _ptr(kv_pages), _ptr(kv_scale), _ptr(qo_indptr), ctypes.byref(pg),
                                  _ptr(out), kv_dtype, ctypes.byref(opts), _stream_handle(stream)),
           "mla_decode_paged")


def decode_from_host(h, dev, kv_dtype: int, *, q_dtype: int, workspace, sm_scale: float = 0.0,
                     num_splits: int = 0, stream=None) -> None:
    """mla_decode_from_host(): h and dev are dicts of (pinned host / device) torch tensors with keys
    q, kv, kv_scale, q_scale, qo_indptr, kv_indptr, out. Asynchronous; synchronise before reading h['out']."""
    opts = make_opts(h["qo_indptr"].numel() - 1, h["q"].shape[0], h["kv"].shape[0], q_dtype=q_dtype,
                     sm_scale=sm_scale, num_splits=num_splits, workspace=workspace)
    bufs = DeviceBuffers(**{k: (None if dev.get(k) is None else dev[k].data_ptr()) for k, _ in DeviceBuffers._fields_})
    _check(lib().mla_decode_from_host(_ptr(h["q"]), _ptr(h["kv"]), _ptr(h.get("kv_scale")), _ptr(h.get("q_scale")),
                                      _ptr(h["qo_indptr"]), _ptr(h["kv_indptr"]), _ptr(h["out"]), kv_dtype,
                                      ctypes.byref(opts), ctypes.byref(bufs), _stream_handle(stream)),
           "mla_decode_from_host")


def dequant_rows(kv, kv_scale, kv_dtype: int, row0: int, nrows: int, out, stream=None) -> None:
    """mla_dequant_rows(): rows [row0, row0+nrows) through the decode kernels' operand path -> out f32."""
    _check(lib().mla_dequant_rows(_ptr(kv), _ptr(kv_scale), kv_dtype, kv.shape[0], row0, nrows, _ptr(out),
                                  _stream_handle(stream)), "mla_dequant_rows")


def device_error(workspace, stream=None) -> tuple[int, int]:
    """(status, flags) from the workspace header. Synchronises the stream."""
    flags = ctypes.c_uint32(0)
    st = lib().mla_get_device_error(_ptr(workspace), _stream_handle(stream), ctypes.byref(flags))
    return st, flags.value


def validate_inputs(qo_indptr, kv_indptr, total_q: int, total_kv: int, kv_dtype: int, kv_scale=None,
                    stream=None) -> tuple[int, int]:
    """mla_validate_inputs(): (status, first bad index or -1). Synchronises the stream."""
    bad = ctypes.c_int64(-1)
    st = lib().mla_validate_inputs(_ptr(qo_indptr), _ptr(kv_indptr), qo_indptr.numel() - 1, total_q, total_kv,
                                   kv_dtype, _ptr(kv_scale), _stream_handle(stream), ctypes.byref(bad))
    return st, bad.value


def static_workspace_device_error(stream=None) -> tuple[int, int]:
    """(status, flags) of the last mla_decode_static_workspace() call on the current device."""
    flags = ctypes.c_uint32(0)
    st = lib().mla_static_workspace_device_error(_stream_handle(stream), ctypes.byref(flags))
    return st, flags.value


def reset_device_error(workspace, stream=None) -> None:
    _check(lib().mla_reset_device_error(_ptr(workspace), _stream_handle(stream)), "mla_reset_device_error")


def elapsed_ms(ev_start, ev_end) -> float:
    """Milliseconds between two torch CUDA events that the library recorded
    (profile events); torch's own Event.elapsed_time only accepts events it
    recorded itself."""
    ms = ctypes.c_float(0.0)
    _check(lib().mla_event_elapsed_ms(ctypes.c_void_p(ev_start.cuda_event), ctypes.c_void_p(ev_end.cuda_event),
                                      ctypes.byref(ms)), "mla_event_elapsed_ms")
    return ms.value
