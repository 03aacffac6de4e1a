"""GPU parity of the paged-KV decode (fp8 e4m3 cache, tcgen05 kernel).

Each case is checked two ways: against the fp64 oracle run on the rows that
the oracle's own page-table gather names (same tolerance as the contiguous
parity tests), and bit for bit against the contiguous decode of those same
rows with the same partition count (the two paths differ only in how rows
reach shared memory).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import mla_decode_attention_split_gb300 as m
from mla_decode_attention_split_gb300 import synth

from test_parity_gpu import check, oracle_ref, run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from mla_decode_attention_split_gb300 import build
    build.build()
    oracle.build()
    m.lib()


def run_paged(pin, num_splits=0, quantize_q=False, expect=m.MLA_OK, table=None):
    t = dict(page_indptr=pin.page_indptr, page_indices=pin.page_indices, last_page_len=pin.last_page_len)
    if table:
        t.update(table)
    out = torch.full((pin.total_q, synth.HEADS, synth.D_V), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = m.alloc_paged_workspace(pin.batch, pin.total_q, pin.total_kv, synth.FP8_E4M3, num_splits=num_splits)
    m.decode_paged(pin.q, pin.kv_pages, pin.kv_scale, pin.qo_indptr, t["page_indptr"], t["page_indices"],
                   t["last_page_len"], pin.page_size, out, synth.FP8_E4M3, total_kv=pin.total_kv, workspace=ws,
                   q_dtype=pin.q_dtype, q_scale=pin.q_scale, num_splits=num_splits, quantize_q=quantize_q)
    torch.cuda.synchronize()
    st, flags = m.device_error(ws)
    assert st == expect, (m.status_string(st), flags)
    return out, flags


def gathered(pin):
    """The contiguous Inputs holding the rows the page table names (oracle gather)."""
    rows, kvp = oracle.paged_rows(pin.kv_pages.cpu().numpy(), pin.page_indptr.cpu().numpy(),
                                  pin.page_indices.cpu().numpy(), pin.last_page_len.cpu().numpy(), pin.page_size)
    return synth.Inputs(q=pin.q, q_scale=pin.q_scale, kv=torch.from_numpy(np.ascontiguousarray(rows)).cuda(),
                        kv_scale=pin.kv_scale, qo_indptr=pin.qo_indptr, kv_indptr=torch.from_numpy(kvp).cuda(),
                        q_dtype=pin.q_dtype, kv_dtype=synth.FP8_E4M3)


LENS = [1, 63, 64, 65, 700, 0, 1301, 129, 2]


@pytest.mark.parametrize("page_size", [1, 7, 16, 64, 128, 300])
@pytest.mark.parametrize("q_dtype", [synth.BF16, synth.FP8_E4M3])
def test_paged_equals_contiguous_and_oracle(page_size, q_dtype):
    w = synth.Workload("paged", len(LENS), 1, 0, q_dtype, synth.FP8_E4M3, seed=40 + page_size)
    pin = synth.make_paged_inputs(w, "cuda", kv_lens=LENS, page_size=page_size, spare_pages=3)
    inp = gathered(pin)
    ref = oracle_ref(inp)
    for ns in (1, 7, 40, 0):
        got, _ = run_paged(pin, num_splits=ns)
        assert torch.equal(got, run_decode(inp, num_splits=ns)), f"num_splits {ns}"
        check(got.float().cpu().numpy(), ref)
    assert np.array_equal(got[5].float().cpu().numpy(), np.zeros((synth.HEADS, synth.D_V)))  # empty segment


def test_paged_multi_token_segments():
    lens, qlens = [5, 0, 300, 64, 77], [2, 1, 3, 0, 1]
    w = synth.Workload("pagedmt", len(lens), 1, 0, synth.BF16, synth.FP8_E4M3, seed=44)
    pin = synth.make_paged_inputs(w, "cuda", kv_lens=lens, q_lens=qlens, page_size=16, spare_pages=2)
    inp = gathered(pin)
    for ns in (1, 4, 16):
        got, _ = run_paged(pin, num_splits=ns)
        assert torch.equal(got, run_decode(inp, num_splits=ns))
        check(got.float().cpu().numpy(), oracle_ref(inp))


def test_page_size_one_with_the_pages_arguments():
    # the argument form of kernelbot-amd-mixed-mla-753817's paged call: one row
    # per page, kv_indices = arange(total_kv), kv_last_page_len = the lengths
    lens = [700, 1, 1301, 64]
    w = synth.Workload("identity", len(lens), 1, 0, synth.BF16, synth.FP8_E4M3, seed=45)
    inp = synth.make_inputs(w, "cuda", kv_lens=lens)
    pin = synth.PagedInputs(q=inp.q, q_scale=None, kv_pages=inp.kv.view(-1, 1, synth.D_QK), kv_scale=inp.kv_scale,
                            qo_indptr=inp.qo_indptr, page_indptr=inp.kv_indptr,
                            page_indices=torch.arange(inp.total_kv, dtype=torch.int32, device="cuda"),
                            last_page_len=torch.tensor(lens, dtype=torch.int32, device="cuda"), page_size=1,
                            total_kv=inp.total_kv, q_dtype=synth.BF16)
    for ns in (3, 0):
        got, _ = run_paged(pin, num_splits=ns)
        assert torch.equal(got, run_decode(inp, num_splits=ns))


def test_paged_in_call_q_quantisation_equals_contiguous():
    w = synth.Workload("pagedq", len(LENS), 1, 0, synth.BF16, synth.FP8_E4M3, seed=46)
    pin = synth.make_paged_inputs(w, "cuda", kv_lens=LENS, page_size=16, spare_pages=1)
    inp = gathered(pin)
    got, _ = run_paged(pin, num_splits=9, quantize_q=True)
    out = torch.empty_like(got)
    ws = m.alloc_workspace(inp.batch, inp.total_q, inp.total_kv, synth.FP8_E4M3, num_splits=9)
    m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, synth.FP8_E4M3, workspace=ws,
             num_splits=9, quantize_q=True)
    torch.cuda.synchronize()
    assert torch.equal(got, out)


def test_paged_large_sampled():
    # 32 segments of 8192 rows in pages of one row (the pages' page size),
    # scattered over a pool with spare pages; sampled (token, head) rows
    lens = [8192] * 32
    w = synth.Workload("pagedlarge", len(lens), 1, 0, synth.BF16, synth.FP8_E4M3, seed=47)
    pin = synth.make_paged_inputs(w, "cuda", kv_lens=lens, page_size=1, spare_pages=1000)
    got, _ = run_paged(pin)
    inp = gathered(pin)
    rng = np.random.default_rng(0)
    toks = rng.integers(0, inp.total_q, 24)
    heads = rng.integers(0, synth.HEADS, 24)
    ref = oracle_ref(inp, rows=(toks, heads))
    g = got.float().cpu().numpy()[toks, heads]
    check(g, ref)


def test_bad_page_id_is_flagged_not_read():
    lens = [300, 77]
    w = synth.Workload("badpage", len(lens), 1, 0, synth.BF16, synth.FP8_E4M3, seed=48)
    pin = synth.make_paged_inputs(w, "cuda", kv_lens=lens, page_size=16)
    bad = pin.page_indices.clone()
    bad[3] = pin.num_pages  # one past the pool: the kernels check ids before any access
    _, flags = run_paged(pin, num_splits=4, expect=m.MLA_ERR_DEVICE_CHECK, table=dict(page_indices=bad))
    assert flags & m.DEVFLAG_BAD_PAGE and not flags & m.DEVFLAG_TIMEOUT


@pytest.mark.parametrize("what", ["last_zero", "last_too_big", "sum_mismatch", "indptr_not_monotone"])
def test_bad_page_table_is_rejected_before_any_row_is_read(what):
    lens = [300, 77, 5]
    w = synth.Workload("badtable", len(lens), 1, 0, synth.BF16, synth.FP8_E4M3, seed=49)
    pin = synth.make_paged_inputs(w, "cuda", kv_lens=lens, page_size=16)
    t = {}
    if what == "last_zero":
        last = pin.last_page_len.clone()
        last[1] = 0
        t["last_page_len"] = last
    elif what == "last_too_big":
        last = pin.last_page_len.clone()
        last[0] = 17
        t["last_page_len"] = last
    elif what == "indptr_not_monotone":
        pip = pin.page_indptr.clone()
        pip[1] = pip[2] + 1
        t["page_indptr"] = pip
    else:
        pin = dataclasses.replace(pin, total_kv=pin.total_kv + 1)
    _, flags = run_paged(pin, num_splits=4, expect=m.MLA_ERR_DEVICE_CHECK, table=t)
    assert flags & m.DEVFLAG_BAD_INDPTR and not flags & m.DEVFLAG_TIMEOUT
