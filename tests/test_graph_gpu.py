"""Decode calls captured into a CUDA graph and replayed.

A serving engine captures its decode step once and replays it. Every entry
point used here makes no allocation and no synchronisation inside the call,
so it can be captured; the replays must give the same bits as eager calls
(with the same inputs and partition count). Covered: the contiguous fp8 path
(programmatic dependent launch), in-call q quantisation (two kernels), token
pairs, the paged path (two kernels), mxfp4 and bf16 KV, and the
allocation-free variant.
"""
import ctypes

import pytest
import torch

import mla_decode_attention_split_gb300 as m
from mla_decode_attention_split_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from mla_decode_attention_split_gb300 import build
    build.build()
    m.lib()


def _captured(call, out):
    """out after an eager call, and after two replays of the captured call (output cleared between)."""
    call()
    torch.cuda.synchronize()
    eager = out.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm the launch path on the capture stream's kind
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    replays = []
    for _ in range(2):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        replays.append(out.clone())
    return eager, replays


@pytest.mark.parametrize("kv_dtype,q_dtype,quantize",
                         [(synth.FP8_E4M3, synth.BF16, False), (synth.FP8_E4M3, synth.BF16, True),
                          (synth.FP8_E4M3, synth.FP8_E4M3, False), (synth.MXFP4, synth.BF16, False),
                          (synth.BF16, synth.BF16, False)])
def test_decode_replays_bitwise(kv_dtype, q_dtype, quantize):
    w = synth.Workload("graph", 4, 1, 0, q_dtype, kv_dtype, seed=51)
    inp = synth.make_inputs(w, "cuda", kv_lens=[700, 64, 1301, 3])
    out = torch.empty((inp.total_q, 16, 512), dtype=torch.bfloat16, device="cuda")
    ws = m.alloc_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, num_splits=11)

    def call():
        m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, inp.kv_dtype, workspace=ws,
                 q_dtype=inp.q_dtype, q_scale=inp.q_scale, num_splits=11, quantize_q=quantize)

    eager, replays = _captured(call, out)
    assert m.device_error(ws)[0] == m.MLA_OK
    for r in replays:
        assert torch.equal(r, eager)


@pytest.mark.parametrize("q_dtype", [synth.BF16, synth.FP8_E4M3])
def test_token_pairs_decode_replays_bitwise(q_dtype):
    w = synth.Workload("graphpairs", 4, 1, 0, q_dtype, synth.FP8_E4M3, seed=54)
    inp = synth.make_inputs(w, "cuda", kv_lens=[700, 64, 1301, 3], q_lens=[2, 3, 1, 2])
    out = torch.empty((inp.total_q, 16, 512), dtype=torch.bfloat16, device="cuda")
    ws = m.alloc_pairs_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, num_splits=11)

    def call():
        m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, inp.kv_dtype, workspace=ws,
                 q_dtype=inp.q_dtype, q_scale=inp.q_scale, num_splits=11, token_pairs=True)

    eager, replays = _captured(call, out)
    assert m.device_error(ws)[0] == m.MLA_OK
    for r in replays:
        assert torch.equal(r, eager)


def test_token_groups_of_four_replay_bitwise():
    w = synth.Workload("graphquad", 4, 1, 0, synth.FP8_E4M3, synth.FP8_E4M3, seed=55)
    inp = synth.make_inputs(w, "cuda", kv_lens=[700, 64, 1301, 3], q_lens=[4, 3, 5, 1])
    out = torch.empty((inp.total_q, 16, 512), dtype=torch.bfloat16, device="cuda")
    ws = m.alloc_group_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, 4, num_splits=11)

    def call():
        m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, inp.kv_dtype, workspace=ws,
                 q_dtype=inp.q_dtype, q_scale=inp.q_scale, num_splits=11, token_group=4)

    eager, replays = _captured(call, out)
    assert m.device_error(ws)[0] == m.MLA_OK
    for r in replays:
        assert torch.equal(r, eager)


def test_paged_decode_replays_bitwise():
    lens = [700, 0, 1301, 65]
    w = synth.Workload("graphpaged", len(lens), 1, 0, synth.BF16, synth.FP8_E4M3, seed=52)
    pin = synth.make_paged_inputs(w, "cuda", kv_lens=lens, page_size=16, spare_pages=2)
    out = torch.empty((pin.total_q, 16, 512), dtype=torch.bfloat16, device="cuda")
    ws = m.alloc_paged_workspace(pin.batch, pin.total_q, pin.total_kv, synth.FP8_E4M3, num_splits=9)

    def call():
        m.decode_paged(pin.q, pin.kv_pages, pin.kv_scale, pin.qo_indptr, pin.page_indptr, pin.page_indices,
                       pin.last_page_len, pin.page_size, out, synth.FP8_E4M3, total_kv=pin.total_kv, workspace=ws,
                       num_splits=9)

    eager, replays = _captured(call, out)
    assert m.device_error(ws)[0] == m.MLA_OK
    for r in replays:
        assert torch.equal(r, eager)


def test_static_workspace_decode_replays_bitwise():
    w = synth.Workload("graphstatic", 3, 1, 0, synth.BF16, synth.FP8_E4M3, seed=53)
    inp = synth.make_inputs(w, "cuda", kv_lens=[500, 1200, 77])
    out = torch.empty((inp.total_q, 16, 512), dtype=torch.bfloat16, device="cuda")
    opts = m.make_opts(inp.batch, inp.total_q, inp.total_kv, num_splits=7)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731

    def call():
        st = m.lib().mla_decode_static_workspace(p(inp.q), p(inp.kv), p(inp.kv_scale), p(inp.qo_indptr),
                                                 p(inp.kv_indptr), p(out), inp.kv_dtype, ctypes.byref(opts),
                                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == m.MLA_OK

    eager, replays = _captured(call, out)
    for r in replays:
        assert torch.equal(r, eager)
