"""GPU parity of the four-token group decode (opts.token_group = 4: up to four
query tokens of a segment share each pass over its KV rows; fp8 KV with fp8 q,
given or quantised in the call).

Checked against the fp64 oracle (same tolerance as the other parity tests)
over ragged token counts (q_len 1 to 8, so groups of 1 to 4 tokens and
segments with two groups), ragged and empty KV runs and several partition
counts; a large multi-token case against the single-token decode and sampled
oracle rows; the workspace's counters left at zero; the dtype combinations it
does not take.
"""
import dataclasses

import numpy as np
import pytest
import torch

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
    m.lib()


def run_quad(inp, num_splits=0, quantize_q=False, sm_scale=0.0, ws=None):
    out = torch.full((inp.total_q, synth.HEADS, synth.D_V), float("nan"), dtype=torch.bfloat16, device="cuda")
    if ws is None:
        ws = m.alloc_group_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, 4, num_splits=num_splits)
    m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, inp.kv_dtype, workspace=ws,
             q_dtype=inp.q_dtype, q_scale=inp.q_scale, num_splits=num_splits, quantize_q=quantize_q,
             sm_scale=sm_scale, token_group=4)
    torch.cuda.synchronize()
    st, flags = m.device_error(ws)
    assert st == m.MLA_OK, (m.status_string(st), flags)
    return out


def caller_quantised(inp):
    """The a8w8 inputs whose codes the call's in-call quantisation computes: s = max(amax, 1e-12) / 448,
    codes = RNE(q / s) saturated (fp64 division rounded to fp32 = the correctly rounded fp32 quotient)."""
    qd = inp.q.float().cpu().double()
    scale = (torch.clamp(qd.abs().max(), min=1e-12) / 448.0).float().reshape(1)
    codes = (qd / scale.double()).float().clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).cuda()
    return dataclasses.replace(inp, q=codes, q_scale=scale.cuda(), q_dtype=synth.FP8_E4M3)


KV = [700, 64, 1301, 129, 50, 0, 257, 3000]
QL = [4, 3, 1, 5, 0, 2, 8, 6]


@pytest.mark.parametrize("q_dtype,quantize", [(synth.FP8_E4M3, False), (synth.BF16, True)])
@pytest.mark.parametrize("num_splits", [1, 7, 40, 0])
def test_quad_against_oracle(q_dtype, quantize, num_splits):
    w = synth.Workload("quad", len(KV), 1, 0, q_dtype, synth.FP8_E4M3, seed=71)
    inp = synth.make_inputs(w, "cuda", kv_lens=KV, q_lens=QL)
    got_t = run_quad(inp, num_splits=num_splits, quantize_q=quantize)
    if quantize:
        # the codes the call quantises to (the per-tensor rule in fp32); fed to
        # the same kernel they give the same bits, and the oracle takes them
        coded = caller_quantised(inp)
        assert torch.equal(got_t, run_quad(coded, num_splits=num_splits))
        ref = oracle_ref(coded)
    else:
        ref = oracle_ref(inp)
    got = got_t.float().cpu().numpy()
    qo = inp.qo_indptr.cpu().numpy()
    for b in np.nonzero(np.array(KV) == 0)[0]:  # empty KV: zeros
        assert np.array_equal(got[qo[b]:qo[b + 1]], np.zeros_like(got[qo[b]:qo[b + 1]]))
    check(got, ref)


@pytest.mark.parametrize("q_len", [1, 2, 3, 4, 5])
def test_quad_every_group_size(q_len):
    # every segment has q_len tokens: groups of 1-4 tokens, and 4 + 1 for q_len 5
    kv = [333, 1024, 77, 2048, 129]
    w = synth.Workload("quadq", len(kv), 1, 0, synth.FP8_E4M3, synth.FP8_E4M3, seed=72 + q_len)
    inp = synth.make_inputs(w, "cuda", kv_lens=kv, q_lens=[q_len] * len(kv))
    check(run_quad(inp, num_splits=9).float().cpu().numpy(), oracle_ref(inp))


def test_quad_large_against_single_token_decode():
    # 32 segments x 4 tokens x 8192 rows with the planner's partition: close to
    # the single-token decode, and within tolerance of the oracle on sampled rows
    w = synth.Workload("quadbig", 32, 4, 8192, synth.FP8_E4M3, synth.FP8_E4M3, seed=73)
    inp = synth.make_inputs(w, "cuda")
    got = run_quad(inp)
    check(got.float().cpu().numpy(), run_decode(inp).float().cpu().numpy().astype(np.float64))
    rng = np.random.default_rng(2)
    toks = rng.integers(0, inp.total_q, 16)
    heads = rng.integers(0, synth.HEADS, 16)
    check(got.float().cpu().numpy()[toks, heads], oracle_ref(inp, rows=(toks, heads)))


def test_quad_workspace_is_reused_and_left_clean():
    w = synth.Workload("quadws", 3, 1, 0, synth.FP8_E4M3, synth.FP8_E4M3, seed=74)
    inp = synth.make_inputs(w, "cuda", kv_lens=[3000, 17, 900], q_lens=[4, 7, 2])
    ws = m.alloc_group_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, 4, num_splits=13)
    outs = []
    for g in (4, 0, 2, 4):  # a group-of-four workspace also serves smaller groups
        out = torch.empty((inp.total_q, 16, 512), dtype=torch.bfloat16, device="cuda")
        m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, inp.kv_dtype, workspace=ws,
                 q_dtype=inp.q_dtype, q_scale=inp.q_scale, num_splits=13, token_group=g)
        torch.cuda.synchronize()
        assert m.device_error(ws)[0] == m.MLA_OK
        outs.append(out)
    assert torch.equal(outs[0], outs[3])
    cnt = ws[256:256 + 4 * inp.total_q].view(torch.int32)
    assert int(cnt.abs().sum()) == 0
    ref = oracle_ref(inp)
    for out in outs:
        check(out.float().cpu().numpy(), ref)


@pytest.mark.parametrize("q_dtype,kv_dtype", [(synth.BF16, synth.FP8_E4M3), (synth.BF16, synth.BF16),
                                              (synth.FP8_E4M3, synth.BF16), (synth.BF16, synth.MXFP4)])
def test_quad_needs_fp8_kv_and_fp8_q(q_dtype, kv_dtype):
    w = synth.Workload("quadno", 2, 4, 100, q_dtype, kv_dtype, seed=75)
    inp = synth.make_inputs(w, "cuda")
    out = torch.empty((inp.total_q, 16, 512), dtype=torch.bfloat16, device="cuda")
    ws = m.alloc_group_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, 4, num_splits=4)
    with pytest.raises(m.MlaError) as e:
        m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, inp.kv_dtype, workspace=ws,
                 q_dtype=inp.q_dtype, q_scale=inp.q_scale, num_splits=4, token_group=4)
    assert e.value.status == m.MLA_ERR_UNSUPPORTED
