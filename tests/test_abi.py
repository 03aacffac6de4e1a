"""The C-ABI library builds (cross-compiled for sm_103a), loads without a GPU,
and exports every entry point that include/mla_decode.h declares; host-only
logic (planner, workspace sizing, argument checks) is exercised on CPU."""
import ctypes
import os
import re

import pytest

import mla_decode_attention_split_gb300 as m
from mla_decode_attention_split_gb300 import build as b

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mla_decode.h")


@pytest.fixture(scope="module")
def lib():
    b.build()
    return m.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("mla_decode", "mla_decode_workspace_size", "mla_plan", "mla_status_string"):
        assert required in names
    assert set(names) == set(m.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_library_is_built_for_sm103a_only(lib):
    log = open(os.path.join(b.BUILD_DIR, "ptxas.log")).read()
    assert "sm_103a" in log and "sm_100" not in log.replace("sm_103a", "")


def test_status_strings(lib):
    for s in range(8):
        assert m.status_string(s).startswith("MLA_")
    assert "unknown" in m.status_string(99)


def test_planner_host_logic(lib):
    # more segments than SMs: one CTA per SM (straddling beats idle SMs)
    assert m.plan(256, 256, 256 * 8192, m.FP8_E4M3, sm_count=152) == 152
    assert m.plan(128, 128, 128 * 8192, m.MXFP4, sm_count=152) == 152
    # fewer segments: a multiple of the segment count, so each CTA holds one
    # piece of one segment (measured 44 us at 128 splits against 53 at 152 for
    # 32 x 8192 rows; 20 against 29 for 64 x 1024)
    assert m.plan(32, 32, 32 * 8192, m.FP8_E4M3, sm_count=152) == 128
    assert m.plan(64, 64, 64 * 1024, m.FP8_E4M3, sm_count=152) == 128
    # short segments: splitting them further costs merges; one CTA per segment
    assert m.plan(64, 64, 64 * 8, m.FP8_E4M3, sm_count=152) == 64
    assert m.plan(4, 4, 4 * 64, m.FP8_E4M3, sm_count=152) == 4
    # 4 x 1024 rows: 8 splits per segment, each one full tile
    assert m.plan(4, 4, 4096, m.BF16, sm_count=152) == 32
    assert m.plan(1, 1, 1, m.FP8_E4M3, sm_count=152) == 1
    assert m.plan(1, 1, 0, m.FP8_E4M3, sm_count=152) == 1
    # q_len > 1: one unit of work per query token
    assert m.plan(2, 8, 256, m.BF16, sm_count=152) == 8
    assert m.plan(32, 64, 32 * 8192, m.FP8_E4M3, sm_count=152) == 128
    # never more CTAs than SMs
    for b, kv in ((1, 10 ** 6), (7, 7 * 3000), (300, 300 * 50)):
        assert 1 <= m.plan(b, b, kv, m.FP8_E4M3, sm_count=152) <= 152
    with pytest.raises(m.MlaError):
        m.plan(-1, 1, 1, m.BF16, sm_count=152)


def test_workspace_size(lib):
    n = m.workspace_size(4, 4, 4096, m.BF16, num_splits=32)
    slots = 32 + 4
    # header, 4 token counters padded to 256 B, partial outputs, partial LSEs
    assert n == 256 + 256 + slots * 16 * 512 * 4 + slots * 16 * 4
    n = m.workspace_size(4, 65, 4096, m.BF16, num_splits=32)
    slots = 32 + 65
    assert n == 256 + 512 + slots * 16 * 512 * 4 + slots * 16 * 4
    with pytest.raises(m.MlaError):
        m.workspace_size(4, 4, 4096, m.BF16, num_splits=-2)


def test_argument_checks_fail_before_any_device_work(lib):
    L = lib
    st = L.mla_decode(None, None, None, None, None, None, m.BF16, None, None)
    assert st == m.MLA_ERR_INVALID_ARG
    opts = m.DecodeOpts(batch=0, total_q=1, total_kv=1, sm_scale=0.0, q_dtype=m.BF16, q_scale=None, num_splits=1,
                        workspace=None, workspace_bytes=0)
    assert L.mla_decode(None, None, None, None, None, None, m.BF16, ctypes.byref(opts), None) == m.MLA_ERR_INVALID_ARG
    # misaligned q pointer
    opts.batch = 1
    buf = (ctypes.c_uint8 * 64)()
    base = ctypes.addressof(buf)
    aligned = (base + 15) & ~15
    st = L.mla_decode(ctypes.c_void_p(aligned + 2), ctypes.c_void_p(aligned), None, ctypes.c_void_p(aligned),
                      ctypes.c_void_p(aligned), ctypes.c_void_p(aligned), m.BF16, ctypes.byref(opts), None)
    assert st == m.MLA_ERR_INVALID_ARG
    # fp8 KV without its scale
    st = L.mla_decode(ctypes.c_void_p(aligned), ctypes.c_void_p(aligned), None, ctypes.c_void_p(aligned),
                      ctypes.c_void_p(aligned), ctypes.c_void_p(aligned), m.FP8_E4M3, ctypes.byref(opts), None)
    assert st == m.MLA_ERR_INVALID_ARG
    # fp8 q without q_scale
    opts.q_dtype = m.FP8_E4M3
    st = L.mla_decode(ctypes.c_void_p(aligned), ctypes.c_void_p(aligned), None, ctypes.c_void_p(aligned),
                      ctypes.c_void_p(aligned), ctypes.c_void_p(aligned), m.BF16, ctypes.byref(opts), None)
    assert st == m.MLA_ERR_INVALID_ARG
    # in-call q quantisation: bf16 q and fp8 KV only
    opts.q_dtype, opts.quantize_q = m.FP8_E4M3, 1
    st = L.mla_decode(ctypes.c_void_p(aligned), ctypes.c_void_p(aligned), ctypes.c_void_p(aligned),
                      ctypes.c_void_p(aligned), ctypes.c_void_p(aligned), ctypes.c_void_p(aligned), m.FP8_E4M3,
                      ctypes.byref(opts), None)
    assert st in (m.MLA_ERR_UNSUPPORTED, m.MLA_ERR_INVALID_ARG)
    opts.q_dtype = m.BF16
    st = L.mla_decode(ctypes.c_void_p(aligned), ctypes.c_void_p(aligned), None, ctypes.c_void_p(aligned),
                      ctypes.c_void_p(aligned), ctypes.c_void_p(aligned), m.BF16, ctypes.byref(opts), None)
    assert st == m.MLA_ERR_UNSUPPORTED
    opts.quantize_q = 0
    # mxfp4 block scales must be 16-byte aligned (they come in by bulk copies)
    st = L.mla_decode(ctypes.c_void_p(aligned), ctypes.c_void_p(aligned), ctypes.c_void_p(aligned + 2),
                      ctypes.c_void_p(aligned), ctypes.c_void_p(aligned), ctypes.c_void_p(aligned), m.MXFP4,
                      ctypes.byref(opts), None)
    assert st == m.MLA_ERR_INVALID_ARG
    # missing workspace
    opts.q_dtype = m.BF16
    st = L.mla_decode(ctypes.c_void_p(aligned), ctypes.c_void_p(aligned), None, ctypes.c_void_p(aligned),
                      ctypes.c_void_p(aligned), ctypes.c_void_p(aligned), m.BF16, ctypes.byref(opts), None)
    assert st == m.MLA_ERR_WORKSPACE
    # dequant entry: row range beyond the cache
    st = L.mla_dequant_rows(ctypes.c_void_p(aligned), None, m.FP8_E4M3, 10, 5, 6, ctypes.c_void_p(aligned), None)
    assert st == m.MLA_ERR_INVALID_ARG
    # mxfp4 rows need their block scales
    st = L.mla_dequant_rows(ctypes.c_void_p(aligned), None, m.MXFP4, 10, 0, 6, ctypes.c_void_p(aligned), None)
    assert st == m.MLA_ERR_INVALID_ARG
    assert L.mla_get_device_error(None, None, None) == m.MLA_ERR_INVALID_ARG


def test_paged_workspace_size_and_argument_checks(lib):
    L = lib
    base = m.workspace_size(4, 4, 4096, m.FP8_E4M3, num_splits=32)
    # room for the logical row offsets: batch + 1 int32, padded to 256 bytes
    assert m.paged_workspace_size(4, 4, 4096, m.FP8_E4M3, num_splits=32) == base + 256
    assert m.paged_workspace_size(64, 64, 4096, m.FP8_E4M3, num_splits=32) == \
        m.workspace_size(64, 64, 4096, m.FP8_E4M3, num_splits=32) + 512
    buf = (ctypes.c_uint8 * 64)()
    a = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    opts = m.DecodeOpts(batch=1, total_q=1, total_kv=10, sm_scale=0.0, q_dtype=m.BF16, q_scale=None, num_splits=1,
                        workspace=None, workspace_bytes=0)
    pg = m.PagedKV(page_indptr=a.value, page_indices=a.value, last_page_len=a.value, page_size=4, num_pages=3)
    args = lambda dt: (a, a, a, a, ctypes.byref(pg), a, dt, ctypes.byref(opts), None)  # noqa: E731
    assert L.mla_decode_paged(a, a, a, a, None, a, m.FP8_E4M3, ctypes.byref(opts), None) == m.MLA_ERR_INVALID_ARG
    pg.page_size = 0
    assert L.mla_decode_paged(*args(m.FP8_E4M3)) == m.MLA_ERR_INVALID_ARG
    pg.page_size, pg.last_page_len = 4, None  # last-page lengths are needed when page_size > 1
    assert L.mla_decode_paged(*args(m.FP8_E4M3)) == m.MLA_ERR_INVALID_ARG
    pg.page_size = 1  # ... but not with one row per page
    assert L.mla_decode_paged(*args(m.FP8_E4M3)) == m.MLA_ERR_WORKSPACE
    pg.num_pages = 0
    assert L.mla_decode_paged(*args(m.FP8_E4M3)) == m.MLA_ERR_INVALID_ARG
    pg.num_pages = 3
    for dt in (m.BF16, m.MXFP4):  # the paged path is the fp8 tensor-core kernel
        assert L.mla_decode_paged(*args(dt)) == m.MLA_ERR_UNSUPPORTED
    # token groups are not combined with a page table
    for g in (2, 4):
        opts.token_group = g
        assert L.mla_decode_paged(*args(m.FP8_E4M3)) == m.MLA_ERR_UNSUPPORTED
    opts.token_group = 0
    # a workspace sized for the contiguous call is too small for the paged one
    n = m.workspace_size(1, 1, 10, m.FP8_E4M3, num_splits=1)
    opts.workspace, opts.workspace_bytes = 256, n
    assert L.mla_decode_paged(*args(m.FP8_E4M3)) == m.MLA_ERR_WORKSPACE


def test_pairs_workspace_size(lib):
    # token pairs: 2 num_splits + total_q partial slots
    n = m.pairs_workspace_size(4, 8, 4096, m.FP8_E4M3, num_splits=32)
    slots = 2 * 32 + 8
    assert n == 256 + 256 + slots * 16 * 512 * 4 + slots * 16 * 4
    assert n == m.workspace_size(4, 8, 4096, m.FP8_E4M3, num_splits=64)
    with pytest.raises(m.MlaError):
        m.pairs_workspace_size(4, 8, 4096, m.FP8_E4M3, num_splits=-1)


def test_group_workspace_size(lib):
    # groups of G tokens: G num_splits + total_q partial slots
    for g in (0, 1, 2, 4):
        n = m.group_workspace_size(4, 8, 4096, m.FP8_E4M3, g, num_splits=32)
        assert n == m.workspace_size(4, 8, 4096, m.FP8_E4M3, num_splits=32 * max(g, 1))
    assert m.group_workspace_size(4, 8, 4096, m.FP8_E4M3, 2, num_splits=32) == \
        m.pairs_workspace_size(4, 8, 4096, m.FP8_E4M3, num_splits=32)
    for g in (-1, 3, 5, 8):
        with pytest.raises(m.MlaError):
            m.group_workspace_size(4, 8, 4096, m.FP8_E4M3, g, num_splits=32)


def test_token_group_argument_checks(lib):
    """token_group: 0/1/2/4 only; 4 needs an fp8 cache and fp8 q (given or quantised in the call);
    no grouping with an mxfp4 cache. All of it is checked before any device work."""
    L = lib
    buf = (ctypes.c_uint8 * 64)()
    a = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    opts = m.DecodeOpts(batch=1, total_q=4, total_kv=8, sm_scale=0.0, q_dtype=m.FP8_E4M3, q_scale=a.value,
                        num_splits=1, workspace=None, workspace_bytes=0)

    def call(kv_dtype, group, q_dtype=m.FP8_E4M3, quantize=0):
        opts.token_group, opts.q_dtype, opts.quantize_q = group, q_dtype, quantize
        return L.mla_decode(a, a, a, a, a, a, kv_dtype, ctypes.byref(opts), None)

    for g in (-1, 3, 5, 8):
        assert call(m.FP8_E4M3, g) == m.MLA_ERR_INVALID_ARG
    for g in (0, 1, 2, 4):  # accepted: the call gets as far as the (missing) workspace
        assert call(m.FP8_E4M3, g) == m.MLA_ERR_WORKSPACE
    assert call(m.FP8_E4M3, 4, q_dtype=m.BF16, quantize=1) == m.MLA_ERR_WORKSPACE
    assert call(m.FP8_E4M3, 4, q_dtype=m.BF16) == m.MLA_ERR_UNSUPPORTED  # bf16 q needs hi + lo rows
    assert call(m.BF16, 4, q_dtype=m.BF16) == m.MLA_ERR_UNSUPPORTED
    assert call(m.BF16, 2, q_dtype=m.BF16) == m.MLA_ERR_WORKSPACE
    for g in (2, 4):
        assert call(m.MXFP4, g, q_dtype=m.BF16) == m.MLA_ERR_UNSUPPORTED
    # the allocation-free entry checks the group before sizing its scratch
    opts.token_group = 3
    assert L.mla_decode_static_workspace(a, a, a, a, a, a, m.FP8_E4M3, ctypes.byref(opts), None) in (
        m.MLA_ERR_INVALID_ARG, m.MLA_ERR_CUDA)


def test_validate_inputs_argument_errors(lib):
    bad = ctypes.c_int64(0)
    # NULL arrays and negative sizes are rejected before any device access
    assert lib.mla_validate_inputs(None, None, 1, 1, 1, m.FP8_E4M3, None, None, ctypes.byref(bad)) == \
        m.MLA_ERR_INVALID_ARG
    assert bad.value == -1
    p = ctypes.c_void_p(16)
    assert lib.mla_validate_inputs(p, p, 0, 1, 1, m.FP8_E4M3, None, None, None) == m.MLA_ERR_INVALID_ARG
    assert lib.mla_validate_inputs(p, p, 1, -1, 1, m.FP8_E4M3, None, None, None) == m.MLA_ERR_INVALID_ARG
    assert lib.mla_validate_inputs(p, p, 1, 1, 1, 7, None, None, None) == m.MLA_ERR_INVALID_ARG
