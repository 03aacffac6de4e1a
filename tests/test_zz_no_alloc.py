"""The allocation-free decode entry point (mla_decode_static_workspace).

Some callers cannot call cudaMalloc when they decode: code running while a
CUDA stream is being captured into a graph, or engines that reserve all device
memory at start-up and forbid allocations afterwards. They cannot hand
mla_decode() a workspace, so the library offers this variant whose scratch is
a fixed array inside the library. These checks call it through the C ABI
twice in a row, with different inputs, and compare each result with
mla_decode() on a caller-provided workspace: within the parity tests'
tolerance and, since both run the same kernel over the same partition, bit
for bit. This file sorts last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

import mla_decode_attention_split_gb300 as m
from mla_decode_attention_split_gb300 import synth

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 2e-2, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from mla_decode_attention_split_gb300 import build
    build.build()
    m.lib()


def _ref(inp, num_splits):
    out = torch.empty((inp.total_q, 16, 512), dtype=torch.bfloat16, device="cuda")
    ws = m.alloc_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, num_splits=num_splits)
    m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, inp.kv_dtype, workspace=ws,
             q_dtype=inp.q_dtype, q_scale=inp.q_scale, num_splits=num_splits)
    return out


def _static(inp, num_splits):
    out = torch.full((inp.total_q, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    opts = m.make_opts(inp.batch, inp.total_q, inp.total_kv, q_dtype=inp.q_dtype, q_scale=inp.q_scale,
                       num_splits=num_splits)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    st = m.lib().mla_decode_static_workspace(p(inp.q), p(inp.kv), p(inp.kv_scale), p(inp.qo_indptr),
                                             p(inp.kv_indptr), p(out), inp.kv_dtype, ctypes.byref(opts),
                                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, out


def _close(a, b):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(a))
    assert np.abs(a - b).max() <= MAX_ABS
    assert np.linalg.norm(a - b) <= REL_L2 * np.linalg.norm(b)


def test_static_workspace_two_calls_match_mla_decode():
    w1 = synth.Workload("a", 5, 1, 0, synth.BF16, synth.FP8_E4M3, seed=31)
    in1 = synth.make_inputs(w1, "cuda", kv_lens=[3000, 77, 1, 900, 4096])
    w2 = synth.Workload("b", 3, 1, 0, synth.FP8_E4M3, synth.FP8_E4M3, seed=32)
    in2 = synth.make_inputs(w2, "cuda", kv_lens=[500, 2048, 129])
    st1, o1 = _static(in1, 0)
    f1 = m.static_workspace_device_error()
    st2, o2 = _static(in2, 7)  # second call reuses the same scratch with other sizes
    f2 = m.static_workspace_device_error()
    torch.cuda.synchronize()
    assert st1 == m.MLA_OK and st2 == m.MLA_OK, (m.status_string(st1), m.status_string(st2))
    assert f1 == (m.MLA_OK, 0) and f2 == (m.MLA_OK, 0), (f1, f2)
    r1, r2 = _ref(in1, 0), _ref(in2, 7)
    _close(o1, r1)
    _close(o2, r2)
    assert torch.equal(o1, r1) and torch.equal(o2, r2)


def test_static_workspace_flags_are_readable():
    # a decreasing kv_indptr: the kernels skip the work and flag it in the fixed array
    w = synth.Workload("bad", 2, 1, 0, synth.BF16, synth.FP8_E4M3, seed=34)
    inp = synth.make_inputs(w, "cuda", kv_lens=[300, 200])
    bad = inp.kv_indptr.clone()
    bad[1] = 501  # kv_indptr = [0, 501, 500]: not monotone
    inp_bad = dataclasses.replace(inp, kv_indptr=bad)
    st, _ = _static(inp_bad, 3)
    assert st == m.MLA_OK
    status, flags = m.static_workspace_device_error()
    assert status == m.MLA_ERR_DEVICE_CHECK and flags & m.DEVFLAG_BAD_INDPTR, (status, flags)
    # the next good call clears them
    st, out = _static(inp, 3)
    assert st == m.MLA_OK
    assert m.static_workspace_device_error() == (m.MLA_OK, 0)
    assert torch.equal(out, _ref(inp, 3))


def test_static_workspace_with_token_pairs():
    # token pairs need 2 num_splits + total_q partial slots; the fixed array serves them too
    w = synth.Workload("pairs", 3, 1, 0, synth.FP8_E4M3, synth.FP8_E4M3, seed=33)
    inp = synth.make_inputs(w, "cuda", kv_lens=[2000, 64, 700], q_lens=[2, 3, 1])
    out = torch.full((inp.total_q, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    opts = m.make_opts(inp.batch, inp.total_q, inp.total_kv, q_dtype=inp.q_dtype, q_scale=inp.q_scale,
                       num_splits=9, token_pairs=True)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = m.lib().mla_decode_static_workspace(p(inp.q), p(inp.kv), p(inp.kv_scale), p(inp.qo_indptr),
                                             p(inp.kv_indptr), p(out), inp.kv_dtype, ctypes.byref(opts),
                                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == m.MLA_OK
    ref = torch.empty_like(out)
    ws = m.alloc_pairs_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, num_splits=9)
    m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, ref, inp.kv_dtype, workspace=ws,
             q_dtype=inp.q_dtype, q_scale=inp.q_scale, num_splits=9, token_pairs=True)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_static_workspace_with_token_groups_of_four():
    # groups of four need 4 num_splits + total_q partial slots; the fixed array serves them too
    w = synth.Workload("quad", 3, 1, 0, synth.FP8_E4M3, synth.FP8_E4M3, seed=34)
    inp = synth.make_inputs(w, "cuda", kv_lens=[2000, 64, 700], q_lens=[4, 5, 2])
    out = torch.full((inp.total_q, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    opts = m.make_opts(inp.batch, inp.total_q, inp.total_kv, q_dtype=inp.q_dtype, q_scale=inp.q_scale,
                       num_splits=9, token_group=4)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = m.lib().mla_decode_static_workspace(p(inp.q), p(inp.kv), p(inp.kv_scale), p(inp.qo_indptr),
                                             p(inp.kv_indptr), p(out), inp.kv_dtype, ctypes.byref(opts),
                                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == m.MLA_OK
    assert m.static_workspace_device_error() == (m.MLA_OK, 0)
    ref = torch.empty_like(out)
    ws = m.alloc_group_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, 4, num_splits=9)
    m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, ref, inp.kv_dtype, workspace=ws,
             q_dtype=inp.q_dtype, q_scale=inp.q_scale, num_splits=9, token_group=4)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_static_workspace_rejects_oversize_requests():
    # (num_splits + total_q) slots of 16 x 512 fp32 must fit in the fixed array
    slots = m.STATIC_WORKSPACE_BYTES // (16 * 512 * 4 + 64) + 1
    opts = m.make_opts(1, slots, 64, num_splits=1)
    st = m.lib().mla_decode_static_workspace(None, None, None, None, None, None, m.FP8_E4M3, ctypes.byref(opts),
                                             None)
    assert st == m.MLA_ERR_TOO_LARGE
    assert "fixed device array" in m.status_string(st)
