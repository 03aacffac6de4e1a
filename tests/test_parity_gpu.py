"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerance (the stated target for bf16 output): max |gpu - oracle| <= 2e-2 and
||gpu - oracle||_2 / ||oracle||_2 <= 1e-2 over the whole output. The expected
error of the design is far below that (bf16 output rounding ~1e-3 relative
plus bf16-precision softmax weights), so a tighter regression bound of 5e-3
rel-L2 is also asserted. Dequantisation is compared bit for bit.
"""
import dataclasses
import json
import os

import numpy as np
import pytest
import torch

import oracle
import oracle_parallel
import mla_decode_attention_split_gb300 as m
from mla_decode_attention_split_gb300 import synth

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2, REL_L2_TIGHT = 2e-2, 1e-2, 5e-3


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from mla_decode_attention_split_gb300 import build
    build.build()
    oracle.build()
    m.lib()


def run_decode(inp, num_splits=0, sm_scale=0.0):
    out = torch.full((inp.total_q, synth.HEADS, synth.D_V), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = m.alloc_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, num_splits=num_splits)
    m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, inp.kv_dtype, workspace=ws,
             q_dtype=inp.q_dtype, q_scale=inp.q_scale, num_splits=num_splits, sm_scale=sm_scale)
    torch.cuda.synchronize()
    st, flags = m.device_error(ws)
    assert st == m.MLA_OK, (m.status_string(st), flags)
    return out


def oracle_ref(inp, sm_scale=None, rows=None):
    h = synth.to_host_codes(inp)
    sm = synth.sm_scale_default() if sm_scale is None else sm_scale
    return oracle.mla_decode(h["q"], h["q_dtype"], h["q_scale"], h["kv"], h["kv_dtype"], h["kv_scale"],
                             h["qo_indptr"], h["kv_indptr"], heads=synth.HEADS, dqk=synth.D_QK, dv=synth.D_V,
                             sm_scale=sm, rows=rows)


def check(got, ref, tight=True):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref).max() if got.size else 0.0
    nrm = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / nrm if nrm > 0 else np.linalg.norm(got)
    assert err <= MAX_ABS, f"max abs {err:.3e} (rel-L2 {rel:.3e})"
    assert rel <= REL_L2, f"rel-L2 {rel:.3e}"
    if tight:
        assert rel <= REL_L2_TIGHT, f"rel-L2 {rel:.3e} above the regression bound"
    return err, rel


COMBOS = [(synth.BF16, synth.BF16), (synth.BF16, synth.FP8_E4M3), (synth.FP8_E4M3, synth.FP8_E4M3),
          (synth.FP8_E4M3, synth.BF16), (synth.BF16, synth.MXFP4), (synth.FP8_E4M3, synth.MXFP4)]
RAGGED = [1, 63, 64, 65, 700, 1301, 129, 2]


@pytest.mark.parametrize("q_dtype,kv_dtype", COMBOS)
@pytest.mark.parametrize("num_splits", [1, 3, 7, 40, 300])
def test_ragged_segments_all_split_counts(q_dtype, kv_dtype, num_splits):
    w = synth.Workload("ragged", len(RAGGED), 1, 0, q_dtype, kv_dtype, seed=21)
    inp = synth.make_inputs(w, "cuda", kv_lens=RAGGED)
    got = run_decode(inp, num_splits=num_splits)
    check(got.float().cpu().numpy(), oracle_ref(inp))


@pytest.mark.parametrize("kv_dtype", [synth.FP8_E4M3, synth.BF16, synth.MXFP4])
@pytest.mark.parametrize("num_splits", [9, 40, 151, 152, 300])
def test_more_splits_than_rows(kv_dtype, num_splits):
    # 9 KV rows in all: every CTA past the ninth gets none, and a token's pieces
    # are one row each (the merge of up to 5 one-row partials), for the
    # cooperative end-of-CTA merge (<= SM count) and the last-CTA merge (300)
    w = synth.Workload("tiny", 3, 1, 0, synth.BF16, kv_dtype, seed=23)
    inp = synth.make_inputs(w, "cuda", kv_lens=[3, 5, 1], q_lens=[1, 2, 1])
    ref = oracle_ref(inp)
    ws = m.alloc_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, num_splits=num_splits)
    for _ in range(2):  # the counters are left at zero for the next call
        out = torch.full((inp.total_q, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, inp.kv_dtype, workspace=ws,
                 q_dtype=inp.q_dtype, q_scale=inp.q_scale, num_splits=num_splits)
        torch.cuda.synchronize()
        assert m.device_error(ws)[0] == m.MLA_OK
        assert int(torch.count_nonzero(ws[256:512])) == 0
        check(out.float().cpu().numpy(), ref)


@pytest.mark.parametrize("q_dtype,kv_dtype", [(synth.BF16, synth.FP8_E4M3), (synth.BF16, synth.BF16),
                                              (synth.BF16, synth.MXFP4)])
def test_multi_token_and_empty_segments(q_dtype, kv_dtype):
    # q_len > 1 (non-causal: every token sees the whole segment), kv_len 0 -> zeros, q_len 0 segments
    w = synth.Workload("edge", 5, 1, 0, q_dtype, kv_dtype, seed=5)
    inp = synth.make_inputs(w, "cuda", kv_lens=[5, 0, 300, 64, 77], q_lens=[2, 1, 3, 0, 1])
    for ns in (1, 4, 16):
        got = run_decode(inp, num_splits=ns).float().cpu().numpy()
        ref = oracle_ref(inp)
        assert np.array_equal(got[2], np.zeros_like(got[2]))
        check(got, ref)


def _with_mxfp4_rows(inp, kvf):
    """The same inputs with the KV cache replaced by the mxfp4 quantisation of kvf."""
    kv, sc = synth.quantize_mxfp4(kvf)
    return dataclasses.replace(inp, kv=kv.contiguous(), kv_scale=sc.contiguous(), kv_dtype=synth.MXFP4)


def test_mxfp4_rows_of_very_different_magnitude():
    # per-row magnitudes 2^-6 .. 2^6 plus all-zero rows: the row exponents differ
    # across the tile, so the softmax weights carry 2^(x + r - mu) over a wide range
    lens = [700, 129, 1301, 64]
    w = synth.Workload("mxrows", len(lens), 1, 0, synth.BF16, synth.MXFP4, seed=31)
    inp = synth.make_inputs(w, "cuda", kv_lens=lens)
    g = torch.Generator(device="cuda").manual_seed(77)
    kvf = torch.randn((inp.total_kv, synth.D_QK), generator=g, device="cuda")
    e = torch.randint(-6, 7, (inp.total_kv, 1), generator=g, device="cuda").float()
    kvf = kvf * torch.pow(2.0, e)
    kvf[::37] = 0.0
    inp = _with_mxfp4_rows(inp, kvf)
    ref = oracle_ref(inp)
    # outputs reach |V| ~ 2^8 here: the absolute bound applies to out / max|out|
    s = np.abs(ref).max()
    for ns in (1, 9):
        check(run_decode(inp, num_splits=ns).float().cpu().numpy() / s, ref / s)


def test_mxfp4_blocks_far_below_the_row_maximum():
    # block magnitudes 2^0 .. 2^-40 inside each row: blocks more than 28 binades
    # below the row's largest scale are flushed by the kernel (elements under
    # 2^-28 of the row's largest block), which the oracle keeps exactly
    lens = [513, 77, 1000]
    w = synth.Workload("mxblocks", len(lens), 1, 0, synth.BF16, synth.MXFP4, seed=32)
    inp = synth.make_inputs(w, "cuda", kv_lens=lens)
    g = torch.Generator(device="cuda").manual_seed(78)
    kvf = torch.randn((inp.total_kv, synth.D_QK), generator=g, device="cuda")
    e = torch.randint(-40, 1, (inp.total_kv, synth.D_QK // 32, 1), generator=g, device="cuda").float()
    kvf = (kvf.view(inp.total_kv, -1, 32) * torch.pow(2.0, e)).view(inp.total_kv, synth.D_QK)
    inp = _with_mxfp4_rows(inp, kvf)
    assert int((inp.kv_scale.max(dim=1).values.int()[:, None] - inp.kv_scale.int() > 28).sum()) > 0
    check(run_decode(inp, num_splits=5).float().cpu().numpy(), oracle_ref(inp))


def test_mxfp4_deep_blocks_are_exact_within_28_binades():
    # V block 5 (dims 160..191) of every row 2^-16 .. 2^-22 below the rest, rope
    # block 17 2^-22 below: every block sits 13..28 binades under its row's
    # largest, where the old 15-binade operand flushed most of them. The output
    # dims 160..191 are that small too (a flushed block would leave them 0), so
    # they are also compared on their own scale.
    lens = [700, 129, 1301]
    w = synth.Workload("mxdeep", len(lens), 1, 0, synth.BF16, synth.MXFP4, seed=33)
    inp = synth.make_inputs(w, "cuda", kv_lens=lens)
    g = torch.Generator(device="cuda").manual_seed(79)
    kvf = torch.randn((inp.total_kv, synth.D_QK), generator=g, device="cuda")
    deep = torch.randint(16, 23, (inp.total_kv, 1), generator=g, device="cuda").float()
    kvf[:, 160:192] *= torch.pow(2.0, -deep)
    kvf[:, 544:576] *= 2.0 ** -22
    inp = _with_mxfp4_rows(inp, kvf)
    d = inp.kv_scale.max(dim=1).values.int()[:, None] - inp.kv_scale.int()
    assert int(d[:, 5].min()) >= 13 and int(d.max()) <= 28 and int((d[:, 5] > 15).sum()) > 0
    ref = oracle_ref(inp)
    for ns in (1, 7):
        got = run_decode(inp, num_splits=ns).float().cpu().numpy()
        check(got, ref)
        blk = ref[:, :, 160:192]
        s = np.abs(blk).max()
        assert s > 0
        check(got[:, :, 160:192] / s, blk / s)


def test_single_row_segments_return_v_rows():
    w = synth.Workload("one", 6, 1, 0, synth.BF16, synth.BF16, seed=9)
    inp = synth.make_inputs(w, "cuda", kv_lens=[1] * 6)
    got = run_decode(inp, num_splits=3)
    v = inp.kv[:, : synth.D_V]
    # softmax over a single row is exactly 1, so out = V row (bf16 in, bf16 out)
    for b in range(6):
        assert torch.equal(got[b], v[b].unsqueeze(0).expand(16, -1))


def test_sm_scale_override():
    w = synth.Workload("scale", 3, 1, 0, synth.BF16, synth.FP8_E4M3, seed=2)
    inp = synth.make_inputs(w, "cuda", kv_lens=[333, 1000, 64])
    got = run_decode(inp, num_splits=5, sm_scale=0.1)
    check(got.float().cpu().numpy(), oracle_ref(inp, sm_scale=0.1))


@pytest.mark.parametrize("kv_dtype", [synth.FP8_E4M3, synth.MXFP4])
def test_deterministic_bitwise(kv_dtype):
    w = synth.Workload("det", 4, 1, 0, synth.BF16, kv_dtype, seed=4)
    inp = synth.make_inputs(w, "cuda", kv_lens=[3000, 17, 900, 2048])
    a = run_decode(inp, num_splits=11)
    b = run_decode(inp, num_splits=11)
    assert torch.equal(a, b)


@pytest.mark.parametrize("kv_dtype", [synth.FP8_E4M3, synth.MXFP4])
def test_workspace_reuse_across_shapes(kv_dtype):
    # split tokens are merged by the CTA that finishes their last partial, through
    # per-token counters in the workspace that every call leaves at zero
    wa = synth.Workload("reuse_a", 3, 1, 0, synth.BF16, kv_dtype, seed=12)
    wb = synth.Workload("reuse_b", 5, 1, 0, synth.BF16, kv_dtype, seed=13)
    a = synth.make_inputs(wa, "cuda", kv_lens=[4000, 10, 2500])
    b = synth.make_inputs(wb, "cuda", kv_lens=[300, 0, 5000, 129, 1000])
    ws = m.alloc_workspace(5, 5, 20000, kv_dtype, num_splits=40)
    outs = []
    for inp in (a, b, a, b):
        out = torch.empty((inp.total_q, 16, 512), dtype=torch.bfloat16, device="cuda")
        m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, inp.kv_dtype, workspace=ws,
                 num_splits=40)
        outs.append(out)
    torch.cuda.synchronize()
    assert m.device_error(ws)[0] == m.MLA_OK
    assert int(torch.count_nonzero(ws[256:512])) == 0  # counters back at zero
    assert torch.equal(outs[0], outs[2]) and torch.equal(outs[1], outs[3])
    assert torch.equal(outs[0], run_decode(a, num_splits=40))
    assert torch.equal(outs[1], run_decode(b, num_splits=40))
    assert torch.count_nonzero(outs[1][1]) == 0  # the empty segment's token


def test_in_call_q_quantisation_equals_caller_quantised_a8w8():
    # quantize_q: the library computes the per-tensor scale and the e4m3 codes of the
    # bf16 q itself; the result must equal the a8w8 path fed with the same codes
    w = synth.Workload("qquant", 4, 1, 0, synth.BF16, synth.FP8_E4M3, seed=41)
    inp = synth.make_inputs(w, "cuda", kv_lens=[500, 1300, 64, 2000])
    # the rule in fp32 with IEEE division (fp64 then rounded to fp32 gives the
    # correctly rounded fp32 quotient); the e4m3 cast rounds to nearest even
    qd = inp.q.float().cpu().double()
    scale = (torch.clamp(qd.abs().max(), min=1e-12) / 448.0).float().reshape(1)
    codes = (qd / scale.double()).float().clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).cuda()
    scale = scale.cuda()
    ref = run_decode(dataclasses.replace(inp, q=codes, q_scale=scale, q_dtype=synth.FP8_E4M3), num_splits=9)
    ws = m.alloc_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, num_splits=9)
    for _ in range(2):  # the amax scratch in the header is left clean for the next call
        out = torch.empty_like(ref)
        m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, inp.kv_dtype, workspace=ws,
                 num_splits=9, quantize_q=True)
        torch.cuda.synchronize()
        assert m.device_error(ws)[0] == m.MLA_OK
        assert torch.equal(out, ref)
    hdr = ws[:32].view(torch.int32).cpu()
    assert int(hdr[2]) == 0 and int(hdr[4]) == 0
    assert abs(float(ws[12:16].view(torch.float32).cpu()[0]) - float(scale.cpu()[0])) == 0.0
    check(ref.float().cpu().numpy(), oracle_ref(dataclasses.replace(inp, q=codes, q_scale=scale, q_dtype=synth.FP8_E4M3)))


@pytest.mark.parametrize("q_mode", ["bf16", "fp8", "quantize"])
def test_later_token_runs_of_a_cta_equal_first_runs(q_mode):
    # 12 equal segments: with one CTA each, every token is its CTA's first run
    # (its Q operand set up by the softmax warps); with one CTA for all, runs
    # 1..11 get theirs from the Q-prep warps through the 4-slot scale ring
    # (wrapping twice). Each token's run lies inside one CTA either way, with
    # the same tiles, so the outputs must agree bit for bit.
    nseg = 12
    q_dtype = synth.FP8_E4M3 if q_mode == "fp8" else synth.BF16
    w = synth.Workload("qprep", nseg, 1, 0, q_dtype, synth.FP8_E4M3, seed=47)
    inp = synth.make_inputs(w, "cuda", kv_lens=[200] * nseg)
    outs = []
    for ns in (nseg, 1):
        out = torch.empty((inp.total_q, 16, 512), dtype=torch.bfloat16, device="cuda")
        ws = m.alloc_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, num_splits=ns)
        m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, inp.kv_dtype, workspace=ws,
                 q_dtype=inp.q_dtype, q_scale=inp.q_scale, num_splits=ns, quantize_q=q_mode == "quantize")
        torch.cuda.synchronize()
        assert m.device_error(ws)[0] == m.MLA_OK
        outs.append(out)
    assert torch.equal(outs[0], outs[1])
    if q_mode != "quantize":
        check(outs[1].float().cpu().numpy(), oracle_ref(inp))


def test_many_token_runs_per_cta_ragged():
    # 21 short ragged segments (one empty) over 1, 2 and 5 CTAs: up to 20 runs
    # per CTA, split and whole, for bf16 and fp8 q
    lens = [1, 7, 130, 0, 64, 65, 3, 300, 8, 9, 127, 128, 129, 2, 40, 17, 256, 5, 90, 11, 200]
    for q_dtype in (synth.BF16, synth.FP8_E4M3):
        w = synth.Workload("manyruns", len(lens), 1, 0, q_dtype, synth.FP8_E4M3, seed=48)
        inp = synth.make_inputs(w, "cuda", kv_lens=lens)
        ref = oracle_ref(inp)
        for ns in (1, 2, 5):
            check(run_decode(inp, num_splits=ns).float().cpu().numpy(), ref)


@pytest.mark.parametrize("q_dtype", [synth.BF16, synth.FP8_E4M3])
def test_piece_outputs_stored_during_the_next_piece(q_dtype):
    # Runs of 8, 6, 1, 16, 3 and 12 tiles: a run's output is stored one block
    # per tile of the next run (all of it when that run has four tiles or more,
    # the rest at its end when it is shorter), the CTA's last run at once. With
    # 2, 3 and 7 CTAs runs split at CTA boundaries, so partials are counted in
    # the middle of the next run; repeated calls give the same bits.
    lens = [1000, 700, 100, 2000, 300, 1500]
    w = synth.Workload("deferred", len(lens), 1, 0, q_dtype, synth.FP8_E4M3, seed=49)
    inp = synth.make_inputs(w, "cuda", kv_lens=lens)
    ref = oracle_ref(inp)
    for ns in (1, 2, 3, 7):
        a = run_decode(inp, num_splits=ns)
        assert torch.equal(a, run_decode(inp, num_splits=ns))
        check(a.float().cpu().numpy(), ref)


@pytest.mark.parametrize("amax_bits", [0x3F80, 0x3FFF, 0x42C9, 0x3B01])
def test_in_call_q_quantisation_codes_over_every_mantissa(amax_bits):
    # Every bf16 value within 13 binades below the tensor maximum (both signs) is
    # quantised in the call and must get the code of the fp32 rule RNE(q / s).
    # Each value sits at dim 0 of one (token, head); every segment holds two KV
    # rows that differ only in dim 0, so the output of that head is a mix of the
    # two V rows whose weight depends on that one code alone.
    amax = torch.tensor([amax_bits], dtype=torch.int16).view(torch.bfloat16).float()
    e = int(((amax_bits >> 7) & 0xFF))
    vals = []
    for be in range(e - 12, e + 1):
        for mant in range(128):
            bits = (be << 7) | mant
            if bits <= amax_bits:
                vals.append(bits)
    bits = torch.tensor(vals + [b | 0x8000 for b in vals], dtype=torch.int32).to(torch.int16)
    qv = bits.view(torch.bfloat16)
    ntok = (qv.numel() + 15) // 16
    qv = torch.cat([qv, torch.zeros(ntok * 16 - qv.numel(), dtype=torch.bfloat16)])
    q = torch.zeros((ntok, 16, 576), dtype=torch.bfloat16)
    q[:, :, 0] = qv.view(ntok, 16)
    kvf = torch.zeros((2 * ntok, 576))
    kvf[1::2, 0] = 3.0          # K differs in dim 0 only
    kvf[0::2, 1:512] = -1.0     # V rows: -1 and +1 (dims 1..511)
    kvf[1::2, 1:512] = 1.0
    kv, kv_scale = synth.quantize_fp8_per_tensor(kvf)
    qo = torch.arange(ntok + 1, dtype=torch.int32)
    kvp = 2 * qo
    inp = synth.Inputs(q=q.cuda(), q_scale=None, kv=kv.cuda(), kv_scale=kv_scale.cuda(), qo_indptr=qo.cuda(),
                       kv_indptr=kvp.cuda(), q_dtype=synth.BF16, kv_dtype=synth.FP8_E4M3)
    qd = q.double()
    scale = (torch.clamp(qd.abs().max(), min=1e-12) / 448.0).float().reshape(1)
    assert float(qd.abs().max()) == float(amax[0])
    codes = (qd / scale.double()).float().clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    sm = 1.0 / float(amax[0])  # scores within +-3: the head's output moves with every code
    ref = run_decode(dataclasses.replace(inp, q=codes.cuda(), q_scale=scale.cuda(), q_dtype=synth.FP8_E4M3),
                     num_splits=7, sm_scale=sm)
    out = torch.empty_like(ref)
    ws = m.alloc_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, num_splits=7)
    m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, inp.kv_dtype, workspace=ws,
             num_splits=7, sm_scale=sm, quantize_q=True)
    torch.cuda.synchronize()
    assert m.device_error(ws)[0] == m.MLA_OK
    # the mix weight moves with the code: distinct codes give distinct outputs
    o = ref[:, :, 1].float().cpu().reshape(-1)[: len(vals) * 2]
    c = codes[:, :, 0].reshape(-1)[: len(vals) * 2].int()
    assert len(set(o.tolist())) >= 0.5 * len(set(c.tolist()))
    assert torch.equal(out, ref)


def test_bad_indptr_sets_device_flag_and_skips_work():
    w = synth.Workload("bad", 3, 1, 0, synth.BF16, synth.FP8_E4M3, seed=8)
    inp = synth.make_inputs(w, "cuda", kv_lens=[100, 100, 100])
    bad = inp.kv_indptr.clone()
    bad[1] = 250  # not monotone: 0, 250, 200, 300
    out = torch.zeros((inp.total_q, 16, 512), dtype=torch.bfloat16, device="cuda")
    ws = m.alloc_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, num_splits=4)
    m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, bad, out, inp.kv_dtype, workspace=ws, num_splits=4)
    st, flags = m.device_error(ws)
    assert st == m.MLA_ERR_DEVICE_CHECK and flags & m.DEVFLAG_BAD_INDPTR
    assert torch.count_nonzero(out) == 0
    m.reset_device_error(ws)
    assert m.device_error(ws) == (m.MLA_OK, 0)


def test_validate_inputs_finds_the_first_bad_entry():
    w = synth.Workload("val", 4, 1, 0, synth.BF16, synth.MXFP4, seed=9)
    inp = synth.make_inputs(w, "cuda", kv_lens=[100, 0, 37, 64], q_lens=[1, 2, 0, 1])
    ok = m.validate_inputs(inp.qo_indptr, inp.kv_indptr, inp.total_q, inp.total_kv, inp.kv_dtype, inp.kv_scale)
    assert ok == (m.MLA_OK, -1)
    n = inp.batch + 1
    cases = []
    qo = inp.qo_indptr.clone()
    qo[2] = 0  # 0, 1, 0, 3, 3, 4: decreasing at 2
    cases.append((qo, inp.kv_indptr, inp.kv_scale, 2))
    kv = inp.kv_indptr.clone()
    kv[0] = 1
    cases.append((inp.qo_indptr, kv, inp.kv_scale, n + 0))
    kv = inp.kv_indptr.clone()
    kv[-1] -= 1  # the last offset is not total_kv
    cases.append((inp.qo_indptr, kv, inp.kv_scale, n + inp.batch))
    sc = inp.kv_scale.clone()
    sc.view(-1)[1000] = 0xFF  # an e8m0 NaN
    cases.append((inp.qo_indptr, inp.kv_indptr, sc, 2 * n + 1000))
    for qo_i, kv_i, sc_i, where in cases:
        st, bad = m.validate_inputs(qo_i, kv_i, inp.total_q, inp.total_kv, inp.kv_dtype, sc_i)
        assert (st, bad) == (m.MLA_ERR_DEVICE_CHECK, where), (m.status_string(st), bad, where)


def test_dequant_fp8_every_code_bit_exact():
    # Every finite code at many positions. The check multiplies by an identity
    # on the tensor core, where a NaN code would also poison the other outputs
    # of its MMA (0 * NaN), so the two NaN codes are checked on their own below.
    rows = 64
    r = np.arange(rows)[:, None]
    d = np.arange(576)[None, :]
    codes = ((r * 7 + d * 13) % 256).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x00
    kv = torch.from_numpy(codes).cuda()
    out = torch.empty((rows, 576), dtype=torch.float32, device="cuda")
    m.dequant_rows(kv, None, m.FP8_E4M3, 0, rows, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    ref = oracle.decode_array("e4m3fn", codes)
    assert np.array_equal(got, ref)
    assert len(np.unique(codes)) == 254
    # NaN codes decode to NaN in place
    nan_codes = np.zeros((8, 576), np.uint8)
    nan_codes[3, 100], nan_codes[5, 571] = 0x7F, 0xFF
    out2 = torch.empty((8, 576), dtype=torch.float32, device="cuda")
    m.dequant_rows(torch.from_numpy(nan_codes).cuda(), None, m.FP8_E4M3, 0, 8, out2)
    torch.cuda.synchronize()
    g2 = out2.cpu().numpy()
    assert np.isnan(g2[3, 100]) and np.isnan(g2[5, 571])


def test_dequant_bf16_bit_exact_with_offset_rows():
    g = torch.Generator().manual_seed(3)
    bits = torch.randint(0, 65536, (40, 576), generator=g, dtype=torch.int32).to(torch.int16)
    # keep finite values (exponent field != 0xFF)
    bits = torch.where((bits.to(torch.int32) & 0x7F80) == 0x7F80, torch.zeros_like(bits), bits)
    kv = bits.view(torch.bfloat16).cuda()
    out = torch.empty((30, 576), dtype=torch.float32, device="cuda")
    m.dequant_rows(kv, None, m.BF16, 7, 30, out)
    torch.cuda.synchronize()
    ref = oracle.decode_array("bf16", bits[7:37].numpy().view(np.uint16))
    got = out.cpu().numpy().astype(np.float64)
    # subnormal bf16 inputs may be flushed by the tensor core; compare the rest exactly
    normal = (np.abs(ref) >= 2.0 ** -126) | (ref == 0)
    assert np.array_equal(got[normal], ref[normal])


def test_dequant_mxfp4_bit_exact_through_the_stage1_conversion():
    # Every byte (two e2m1 codes) meets block exponents 0..40 binades below its
    # row's largest: within 28 the value is code * 2^(s - 127) exactly (that
    # covers the e5m2 subnormals at 26..28 below), beyond it the block is
    # flushed to zero as in the decode. Two more rows: every scale 254 (values
    # from 2^128 up overflow fp32 on both sides) and every scale 0 (fp32
    # subnormals).
    rows, nb = 66, 18
    r = np.arange(rows)[:, None]
    codes = ((r * 7 + np.arange(288)[None, :] * 13) % 256).astype(np.uint8)
    base = 120 + (np.arange(rows) % 9)
    down = (np.arange(rows)[:, None] * 5 + np.arange(nb)[None, :] * 3) % 41
    down[:, 0] = 0  # block 0 holds the row's largest exponent
    scales = (base[:, None] - down).astype(np.uint8)
    scales[64], scales[65] = 254, 0
    kv = torch.from_numpy(codes).cuda()
    sc = torch.from_numpy(scales).cuda()
    out = torch.empty((rows - 2, 576), dtype=torch.float32, device="cuda")
    m.dequant_rows(kv, sc, m.MXFP4, 2, rows - 2, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    nib = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(rows, 576)
    elem = oracle.decode_array("e2m1", nib)
    scale = oracle.decode_array("e8m0", scales)
    with np.errstate(over="ignore"):
        ref = (elem * np.repeat(scale, 32, axis=1)).astype(np.float32)[2:]
    depth = scales.max(axis=1, keepdims=True) - scales.astype(np.int32)
    flushed = np.repeat(depth > 28, 32, axis=1)[2:]
    assert flushed.any() and (~flushed).any()
    assert set(np.unique(depth[:64])) == set(range(41))  # every block distance 0..40 occurs
    bad = np.argwhere((got != ref) & ~flushed & ~(np.isnan(got) & np.isnan(ref)))
    rs, ds = bad[:, 0] + 2, bad[:, 1]
    assert len(bad) == 0, (len(bad), [(int(a), int(d), int(nib[a, d]), int(scales[a, d // 32]),
                                        int(scales[a].max()), float(got[a - 2, d]), float(ref[a - 2, d]))
                                       for a, d in zip(rs[:12], ds[:12])])
    assert np.all(got[flushed] == 0)
    assert np.isinf(got[62]).any() and np.isfinite(got[62]).any()
    assert ((np.abs(got[63]) < 2.0 ** -126) & (got[63] != 0)).any()
    assert len(np.unique(codes[2:])) == 256


def test_host_buffer_entry_matches_device_entry():
    w = synth.Workload("host", 3, 1, 0, synth.FP8_E4M3, synth.FP8_E4M3, seed=6)
    inp = synth.make_inputs(w, "cuda", kv_lens=[500, 64, 1500])
    ref = run_decode(inp, num_splits=6)
    h = {"q": inp.q.cpu().pin_memory(), "kv": inp.kv.cpu().pin_memory(), "kv_scale": inp.kv_scale.cpu().pin_memory(),
         "q_scale": inp.q_scale.cpu().pin_memory(), "qo_indptr": inp.qo_indptr.cpu().pin_memory(),
         "kv_indptr": inp.kv_indptr.cpu().pin_memory(),
         "out": torch.empty(ref.shape, dtype=torch.bfloat16).pin_memory()}
    dev = {k: torch.empty_like(v, device="cuda") for k, v in h.items()}
    ws = m.alloc_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, num_splits=6)
    m.decode_from_host(h, dev, inp.kv_dtype, q_dtype=inp.q_dtype, workspace=ws, num_splits=6)
    torch.cuda.synchronize()
    assert torch.equal(h["out"], ref.cpu())


# ---- the benchmark workloads --------------------------------------------------

def test_workload_bf16_bs4_kv1024_full():
    inp = synth.make_inputs(synth.WORKLOADS["bf16_bs4_kv1024"], "cuda")
    got = run_decode(inp)
    check(got.float().cpu().numpy(), oracle_ref(inp))


def test_workload_a8w8_bs64_kv1024_full():
    inp = synth.make_inputs(synth.WORKLOADS["a8w8_bs64_kv1024"], "cuda")
    got = run_decode(inp)
    check(got.float().cpu().numpy(), oracle_ref(inp))


@pytest.mark.parametrize("name", ["fp8kv_bs32_kv8192", "fp8kv_bs256_kv8192", "mxfp4_bs128_ragged16384"])
def test_workload_large_full(name):
    """Full size, the benchmark's launch configuration (planner default), compared
    with the oracle over the whole output; the oracle runs one segment per host
    thread. Every segment must also meet the rel-L2 bound on its own (the
    per-segment diagnostic). With MLA_PARITY_REPORT_DIR set, the figures are
    written there as JSON."""
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w, "cuda")
    got = run_decode(inp).float().cpu().numpy().astype(np.float64)
    h = synth.to_host_codes(inp)
    ref = oracle_parallel.decode_segments(h, synth.sm_scale_default())
    err, rel = check(got, ref)
    seg = oracle_parallel.per_segment_rel_l2(got, ref, h["qo_indptr"])
    seg = seg[np.isfinite(seg)]
    assert seg.size == inp.batch
    assert seg.max() <= REL_L2, f"worst segment rel-L2 {seg.max():.3e} (segment {int(np.argmax(seg))})"
    report_dir = os.environ.get("MLA_PARITY_REPORT_DIR")
    if report_dir:
        os.makedirs(report_dir, exist_ok=True)
        kvp = h["kv_indptr"].astype(np.int64)
        worst = int(np.argmax(seg))
        with open(os.path.join(report_dir, f"parity_{name}.json"), "w") as f:
            json.dump({"workload": name, "elements": int(got.size), "max_abs": float(err), "rel_l2": float(rel),
                       "segments": int(seg.size), "segment_rel_l2_min": float(seg.min()),
                       "segment_rel_l2_median": float(np.median(seg)), "segment_rel_l2_max": float(seg.max()),
                       "worst_segment": worst, "worst_segment_kv_len": int(kvp[worst + 1] - kvp[worst]),
                       "num_splits": m.plan(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype)}, f, indent=1)


def _rising_inputs(q_dtype, kv_dtype, q_lens, kv_lens, seed):
    """Scores that rise along each segment (rope dim 512 of K, which is not a V dim, is a ramp
    0..300 and q's dim 512 is 1 in every head) with N(0,1) elsewhere, plus one spike row in the
    middle: in log2 units the softmax reference of a head moves several times within a segment,
    and after the spike it stays above the rising rows."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    qo = torch.tensor([0] + list(np.cumsum(q_lens)), dtype=torch.int32)
    kvp = torch.tensor([0] + list(np.cumsum(kv_lens)), dtype=torch.int32)
    qf = torch.randn((int(qo[-1]), 16, 576), generator=g)
    qf[:, :, 512] = 1.0
    kvf = torch.randn((int(kvp[-1]), 576), generator=g)
    for b, n in enumerate(kv_lens):
        k0 = int(kvp[b])
        kvf[k0:k0 + n, 512] = torch.linspace(0.0, 300.0, n)
        kvf[k0 + n // 2, 512] = 330.0
    if q_dtype == synth.BF16:
        q, q_scale = qf.to(torch.bfloat16), None
    else:
        q, q_scale = synth.quantize_fp8_per_tensor(qf)
    if kv_dtype == synth.BF16:
        kv, kv_scale = kvf.to(torch.bfloat16), None
    elif kv_dtype == synth.FP8_E4M3:
        kv, kv_scale = synth.quantize_fp8_per_tensor(kvf)
    else:
        kv, kv_scale = synth.quantize_mxfp4(kvf)
    dev = lambda t: None if t is None else t.contiguous().cuda()  # noqa: E731
    return synth.Inputs(q=dev(q), q_scale=dev(q_scale), kv=dev(kv), kv_scale=dev(kv_scale), qo_indptr=qo.cuda(),
                        kv_indptr=kvp.cuda(), q_dtype=q_dtype, kv_dtype=kv_dtype)


@pytest.mark.parametrize("q_dtype,kv_dtype,group", [
    (synth.BF16, synth.FP8_E4M3, 0), (synth.BF16, synth.BF16, 0), (synth.BF16, synth.MXFP4, 0),
    (synth.BF16, synth.FP8_E4M3, 2), (synth.FP8_E4M3, synth.FP8_E4M3, 2), (synth.BF16, synth.BF16, 2),
    (synth.FP8_E4M3, synth.FP8_E4M3, 4)])
def test_rising_scores_move_the_softmax_reference(q_dtype, kv_dtype, group):
    # the kernels keep a lazy reference max per head (it moves only when a tile's max exceeds it
    # by more than 3.5 in log2 units); the output must still be the softmax of the oracle
    inp = _rising_inputs(q_dtype, kv_dtype, [3, 4], [2000, 1300], seed=91)
    out = torch.full((inp.total_q, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    for ns in (1, 5):
        ws = m.alloc_group_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, group, num_splits=ns)
        m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, inp.kv_dtype, workspace=ws,
                 q_dtype=inp.q_dtype, q_scale=inp.q_scale, num_splits=ns, token_group=group)
        torch.cuda.synchronize()
        assert m.device_error(ws)[0] == m.MLA_OK
        check(out.float().cpu().numpy(), oracle_ref(inp))
