"""GPU parity of the token-pair decode (opts.token_pairs: two query tokens of a
segment share each pass over its KV rows; fp8 and bf16 KV).

Checked against the fp64 oracle (same tolerance as the other parity tests)
over ragged token and row counts, odd q_len (a one-token last group), empty
segments and several partition counts; and bit for bit against the
single-token decode when each segment is one partition (num_splits = 1),
where both compute every token with the same tiles and arithmetic.
"""
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


def run_pairs(inp, num_splits=0, quantize_q=False, sm_scale=0.0):
    out = torch.full((inp.total_q, synth.HEADS, synth.D_V), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = m.alloc_pairs_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, num_splits=num_splits)
    m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, inp.kv_dtype, workspace=ws,
             q_dtype=inp.q_dtype, q_scale=inp.q_scale, num_splits=num_splits, quantize_q=quantize_q,
             sm_scale=sm_scale, token_pairs=True)
    torch.cuda.synchronize()
    st, flags = m.device_error(ws)
    assert st == m.MLA_OK, (m.status_string(st), flags)
    return out


KV = [700, 64, 1301, 129, 50, 0, 257]
QL = [2, 3, 1, 4, 0, 2, 5]


@pytest.mark.parametrize("q_dtype,quantize", [(synth.BF16, False), (synth.FP8_E4M3, False), (synth.BF16, True)])
def test_pairs_equal_single_token_decode_with_one_partition(q_dtype, quantize):
    # bf16 q: the token-pair kernel gives the single-token bits. fp8 q (given or quantised in the
    # call): the kernel that runs the two tokens' softmax in two warp groups does the same
    # arithmetic, but its compiled code may round an operation differently: one bf16 step on a
    # few elements at most, and the oracle decides
    w = synth.Workload("pairs1", len(KV), 1, 0, q_dtype, synth.FP8_E4M3, seed=61)
    inp = synth.make_inputs(w, "cuda", kv_lens=KV, q_lens=QL)
    got = run_pairs(inp, num_splits=1, quantize_q=quantize)
    out = torch.empty_like(got)
    ws = m.alloc_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, num_splits=1)
    m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, inp.kv_dtype, workspace=ws,
             q_dtype=inp.q_dtype, q_scale=inp.q_scale, num_splits=1, quantize_q=quantize)
    torch.cuda.synchronize()
    if q_dtype == synth.BF16 and not quantize:
        assert torch.equal(got, out)
    else:
        g, o = got.float(), out.float()
        step = torch.maximum(o.abs(), torch.full_like(o, 2.0 ** -126)) * 2.0 ** -7  # one bf16 step (upper bound)
        assert bool(((g - o).abs() <= step).all())
        assert int((g != o).sum()) <= 8
        if not quantize:
            check(got.float().cpu().numpy(), oracle_ref(inp))


@pytest.mark.parametrize("q_dtype", [synth.BF16, synth.FP8_E4M3])
@pytest.mark.parametrize("num_splits", [1, 7, 40, 0])
def test_pairs_against_oracle(q_dtype, num_splits):
    w = synth.Workload("pairs", len(KV), 1, 0, q_dtype, synth.FP8_E4M3, seed=62)
    inp = synth.make_inputs(w, "cuda", kv_lens=KV, q_lens=QL)
    got = run_pairs(inp, num_splits=num_splits).float().cpu().numpy()
    ref = oracle_ref(inp)
    qo = inp.qo_indptr.cpu().numpy()
    for b in np.nonzero(np.array(KV) == 0)[0]:  # empty KV: zeros
        assert np.array_equal(got[qo[b]:qo[b + 1]], np.zeros_like(got[qo[b]:qo[b + 1]]))
    check(got, ref)


def test_pairs_large_against_single_token_decode():
    # 64 segments x 2 tokens x 8192 rows with the planner's partition: each
    # token within tolerance of the oracle on sampled rows, and close to the
    # single-token decode
    w = synth.Workload("pairsbig", 64, 2, 8192, synth.BF16, synth.FP8_E4M3, seed=63)
    inp = synth.make_inputs(w, "cuda")
    got = run_pairs(inp)
    ref_single = run_decode(inp)
    check(got.float().cpu().numpy(), ref_single.float().cpu().numpy().astype(np.float64))
    rng = np.random.default_rng(1)
    toks = rng.integers(0, inp.total_q, 16)
    heads = rng.integers(0, synth.HEADS, 16)
    check(got.float().cpu().numpy()[toks, heads], oracle_ref(inp, rows=(toks, heads)))


def test_pairs_workspace_is_reused_and_left_clean():
    w = synth.Workload("pairsws", 3, 1, 0, synth.BF16, synth.FP8_E4M3, seed=64)
    inp = synth.make_inputs(w, "cuda", kv_lens=[3000, 17, 900], q_lens=[2, 3, 2])
    ws = m.alloc_pairs_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, num_splits=13)
    outs = []
    for pairs in (True, False, True):  # a pairs workspace also serves single-token calls
        out = torch.empty((inp.total_q, 16, 512), dtype=torch.bfloat16, device="cuda")
        m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, inp.kv_dtype, workspace=ws,
                 num_splits=13, token_pairs=pairs)
        torch.cuda.synchronize()
        assert m.device_error(ws)[0] == m.MLA_OK
        outs.append(out)
    assert torch.equal(outs[0], outs[2])
    cnt = ws[256:256 + 4 * inp.total_q].view(torch.int32)
    assert int(cnt.abs().sum()) == 0
    check(outs[0].float().cpu().numpy(), oracle_ref(inp))


@pytest.mark.parametrize("q_dtype", [synth.BF16, synth.FP8_E4M3])
@pytest.mark.parametrize("num_splits", [1, 7, 40, 0])
def test_pairs_bf16_kv_against_oracle(q_dtype, num_splits):
    w = synth.Workload("pairsbf", len(KV), 1, 0, q_dtype, synth.BF16, seed=66)
    inp = synth.make_inputs(w, "cuda", kv_lens=KV, q_lens=QL)
    got = run_pairs(inp, num_splits=num_splits).float().cpu().numpy()
    ref = oracle_ref(inp)
    qo = inp.qo_indptr.cpu().numpy()
    for b in np.nonzero(np.array(KV) == 0)[0]:  # empty KV: zeros
        assert np.array_equal(got[qo[b]:qo[b + 1]], np.zeros_like(got[qo[b]:qo[b + 1]]))
    check(got, ref)


@pytest.mark.parametrize("q_dtype", [synth.BF16, synth.FP8_E4M3])
def test_pairs_bf16_kv_equal_single_token_decode_with_one_partition(q_dtype):
    w = synth.Workload("pairsbf1", len(KV), 1, 0, q_dtype, synth.BF16, seed=67)
    inp = synth.make_inputs(w, "cuda", kv_lens=KV, q_lens=QL)
    got = run_pairs(inp, num_splits=1)
    assert torch.equal(got, run_decode(inp, num_splits=1))


def test_pairs_need_fp8_or_bf16_kv():
    w = synth.Workload("pairsmx", 2, 2, 100, synth.BF16, synth.MXFP4, seed=65)
    inp = synth.make_inputs(w, "cuda")
    out = torch.empty((inp.total_q, 16, 512), dtype=torch.bfloat16, device="cuda")
    ws = m.alloc_pairs_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, num_splits=4)
    with pytest.raises(m.MlaError) as e:
        m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, inp.kv_dtype, workspace=ws,
                 num_splits=4, token_pairs=True)
    assert e.value.status == m.MLA_ERR_UNSUPPORTED
