"""Pins for the oracle's attention arithmetic (CPU only).

The oracle is checked against: brute force in 50-digit arithmetic (mpmath,
no max subtraction) on tiny inputs; the naive reference formula of
kernelbot-amd-mixed-mla-675627 (`custom_kernel_bf16`: per segment
softmax((q*sm_scale) @ k^T) @ v) re-evaluated by torch in float64; and
invariants that fix the result without any implementation (one KV row,
identical keys, zero query, permutation of rows, split + LSE merge, a dominant
key). Small dims (D=8, DV=6) keep the "V = first DV dims" rule visible.
"""
import math

import mpmath
import numpy as np
import pytest
import torch

from mla_decode_attention_split_gb300 import synth

RNG = np.random.default_rng(1234)


def _segments(lens_q, lens_kv):
    return (np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32),
            np.concatenate([[0], np.cumsum(lens_kv)]).astype(np.int32))


def _rand_case(lens_q, lens_kv, H=2, D=8, scale=1.0):
    qo, kvp = _segments(lens_q, lens_kv)
    q = RNG.standard_normal((qo[-1], H, D)) * scale
    kv = RNG.standard_normal((kvp[-1], D)) * scale
    return q, kv, qo, kvp


def _brute(q, kv, qo, kvp, sm_scale, DV):
    mpmath.mp.dps = 50
    total_q, H, D = q.shape
    out = np.zeros((total_q, H, DV))
    for b in range(len(qo) - 1):
        for t in range(qo[b], qo[b + 1]):
            for h in range(H):
                ws, acc = [], [mpmath.mpf(0)] * DV
                for j in range(kvp[b], kvp[b + 1]):
                    s = mpmath.mpf(sm_scale) * mpmath.fsum(
                        mpmath.mpf(q[t, h, d]) * mpmath.mpf(kv[j, d]) for d in range(D))
                    w = mpmath.exp(s)
                    ws.append(w)
                    acc = [acc[d] + w * mpmath.mpf(kv[j, d]) for d in range(DV)]
                if ws:
                    z = mpmath.fsum(ws)
                    out[t, h] = [float(a / z) for a in acc]
    return out


def test_brute_force_50_digits(oracle_mod):
    q, kv, qo, kvp = _rand_case([1, 2, 1, 1], [3, 1, 8, 5])
    sm = 1.0 / math.sqrt(8)
    ours = oracle_mod.attention_f64(q, kv, qo, kvp, sm, 6)
    ref = _brute(q, kv, qo, kvp, sm, 6)
    assert np.allclose(ours, ref, rtol=1e-13, atol=1e-15)


def test_torch_float64_naive_reference_formula(oracle_mod):
    q, kv, qo, kvp = _rand_case([1, 3, 2, 1], [37, 64, 1, 200], H=4, D=24)
    sm = 1.0 / math.sqrt(24)
    DV = 16
    ours = oracle_mod.attention_f64(q, kv, qo, kvp, sm, DV)
    qt, kt = torch.from_numpy(q), torch.from_numpy(kv)
    for b in range(len(qo) - 1):
        qi = qt[qo[b]:qo[b + 1]].permute(1, 0, 2)          # (H, seq_q, D)
        ki = kt[kvp[b]:kvp[b + 1]]
        scores = torch.softmax(torch.matmul(qi * sm, ki.T), dim=-1)
        oi = torch.matmul(scores, ki[:, :DV]).permute(1, 0, 2)
        assert np.allclose(ours[qo[b]:qo[b + 1]], oi.numpy(), rtol=1e-12, atol=1e-14)


def test_single_kv_row_returns_that_v_exactly(oracle_mod):
    q, kv, qo, kvp = _rand_case([1, 1], [1, 1], H=3, D=8)
    out = oracle_mod.attention_f64(q, kv, qo, kvp, 0.3, 6)
    for b in range(2):
        for h in range(3):
            assert np.array_equal(out[b, h], kv[b, :6])


def test_identical_keys_and_zero_query_give_mean_of_v(oracle_mod):
    # Every score equal: the query is zero on the V dims and the rows agree on
    # the remaining (rope) dims, so all keys look identical to the query.
    n, D, DV = 50, 8, 6
    v = RNG.standard_normal((n, D))
    q = np.zeros((1, 1, D))
    q[0, 0, DV:] = RNG.standard_normal(D - DV)
    kv = v.copy()
    kv[:, DV:] = v[0, DV:]
    out = oracle_mod.attention_f64(q, kv, [0, 1], [0, n], 0.7, DV)
    assert np.allclose(out[0, 0], kv[:, :DV].mean(axis=0), rtol=1e-13, atol=1e-15)
    qz = np.zeros((1, 1, D))
    outz = oracle_mod.attention_f64(qz, v, [0, 1], [0, n], 0.7, DV)
    assert np.allclose(outz[0, 0], v[:, :DV].mean(axis=0), rtol=1e-13, atol=1e-15)


def test_rope_dims_enter_scores_but_not_values(oracle_mod):
    q, kv, qo, kvp = _rand_case([1], [40], H=2, D=8)
    base = oracle_mod.attention_f64(q, kv, qo, kvp, 0.5, 6)
    kv2 = kv.copy()
    kv2[:, 6:] += RNG.standard_normal((40, 2))
    moved = oracle_mod.attention_f64(q, kv2, qo, kvp, 0.5, 6)
    assert np.abs(moved - base).max() > 1e-3          # dims >= DV change the weights
    q3 = q.copy()
    q3[..., 6:] = 0.0                                  # ... and with q zero there, nothing
    a = oracle_mod.attention_f64(q3, kv, qo, kvp, 0.5, 6)
    b = oracle_mod.attention_f64(q3, kv2, qo, kvp, 0.5, 6)
    assert np.array_equal(a, b)


def test_permutation_invariance(oracle_mod):
    q, kv, qo, kvp = _rand_case([2, 1], [300, 77], H=3, D=16)
    out = oracle_mod.attention_f64(q, kv, qo, kvp, 0.25, 12)
    kvp_perm = kv.copy()
    kvp_perm[0:300] = kv[0:300][RNG.permutation(300)]
    kvp_perm[300:] = kv[300:][RNG.permutation(77)]
    out2 = oracle_mod.attention_f64(q, kvp_perm, qo, kvp, 0.25, 12)
    assert np.abs(out - out2).max() < 1e-12


@pytest.mark.parametrize("cuts", [[1], [150], [299], [10, 20, 250], [1, 2, 3, 4, 5]])
def test_split_and_lse_merge_equals_unsplit(oracle_mod, cuts):
    n, D, DV = 300, 16, 12
    q = RNG.standard_normal((1, 1, D)) * 2
    kv = RNG.standard_normal((n, D))
    full, full_lse = oracle_mod.attention_f64(q, kv, [0, 1], [0, n], 0.4, DV, want_lse=True)
    edges = [0] + cuts + [n]
    parts, lses = [], []
    for a, b in zip(edges[:-1], edges[1:]):
        o, l = oracle_mod.attention_f64(q, kv[a:b], [0, 1], [0, b - a], 0.4, DV, want_lse=True)
        parts.append(o[0, 0])
        lses.append(l[0, 0])
    merged, mlse = oracle_mod.lse_combine(np.array(parts), np.array(lses))
    assert np.abs(merged - full[0, 0]).max() < 1e-12
    assert abs(mlse - full_lse[0, 0]) < 1e-12


def test_lse_merge_ignores_empty_splits(oracle_mod):
    o = RNG.standard_normal((3, 5))
    merged, lse = oracle_mod.lse_combine(o, np.array([-np.inf, 0.5, -np.inf]))
    assert np.array_equal(merged, o[1]) and lse == 0.5
    merged0, lse0 = oracle_mod.lse_combine(o, np.full(3, -np.inf))
    assert np.array_equal(merged0, np.zeros(5)) and lse0 == -np.inf


def test_dominant_key_selects_its_value(oracle_mod):
    n, D, DV = 64, 8, 6
    q = RNG.standard_normal((1, 1, D))
    kv = RNG.standard_normal((n, D)) * 0.1
    kv[17] = q[0, 0] * 40.0                     # score gap >> 40 nats
    out = oracle_mod.attention_f64(q, kv, [0, 1], [0, n], 1.0, DV)
    assert np.allclose(out[0, 0], kv[17, :DV], rtol=1e-14, atol=1e-14)


def test_empty_segments_and_non_causal_multi_token(oracle_mod):
    # kv_len 0 -> zeros, lse -inf; q_len 0 -> nothing; q_len 3 -> each token alone
    q, kv, qo, kvp = _rand_case([1, 0, 3, 2], [5, 4, 9, 0], H=2, D=8)
    out, lse = oracle_mod.attention_f64(q, kv, qo, kvp, 0.5, 6, want_lse=True)
    assert np.array_equal(out[4:6], np.zeros((2, 2, 6))) and np.all(lse[4:6] == -np.inf)
    for t in range(1, 4):
        single = oracle_mod.attention_f64(q[t:t + 1], kv[9:18], [0, 1], [0, 9], 0.5, 6)
        assert np.array_equal(out[t], single[0])


# ---- raw encodings -> the decode path (pins the dequant plumbing)

def _unpack_mx(packed, scales):
    lo, hi = packed & 0xF, packed >> 4
    nib = np.empty((packed.shape[0], packed.shape[1] * 2), np.uint8)
    nib[:, 0::2], nib[:, 1::2] = lo, hi
    table = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])
    return table[nib] * np.repeat(2.0 ** (scales.astype(np.float64) - 127), 32, axis=1)


@pytest.mark.parametrize("q_dtype,kv_dtype", [(synth.BF16, synth.BF16), (synth.BF16, synth.FP8_E4M3),
                                              (synth.FP8_E4M3, synth.FP8_E4M3), (synth.BF16, synth.MXFP4)])
def test_raw_decode_path_matches_decoded_arrays(oracle_mod, q_dtype, kv_dtype):
    w = synth.Workload("t", 3, 1, 0, q_dtype, kv_dtype, seed=3)
    inp = synth.make_inputs(w, "cpu", kv_lens=[5, 33, 64], q_lens=[1, 2, 1])
    h = synth.to_host_codes(inp)
    sm = synth.sm_scale_default()
    out = oracle_mod.mla_decode(h["q"], q_dtype, h["q_scale"], h["kv"], kv_dtype, h["kv_scale"],
                                h["qo_indptr"], h["kv_indptr"], heads=16, dqk=576, dv=512, sm_scale=sm)
    if q_dtype == synth.BF16:
        qd = inp.q.double().numpy()
    else:
        qd = inp.q.view(torch.float8_e4m3fn).double().numpy() * float(inp.q_scale[0])
    if kv_dtype == synth.BF16:
        kd = inp.kv.double().numpy()
    elif kv_dtype == synth.FP8_E4M3:
        kd = inp.kv.view(torch.float8_e4m3fn).double().numpy() * float(inp.kv_scale[0])
    else:
        kd = _unpack_mx(inp.kv.numpy(), inp.kv_scale.numpy())
    ref = oracle_mod.attention_f64(qd, kd, h["qo_indptr"], h["kv_indptr"], sm, 512)
    assert np.array_equal(out, ref)
    # sampled rows give the same numbers as the full pass
    rows = (np.array([3, 0, 2]), np.array([15, 0, 7]))
    part = oracle_mod.mla_decode(h["q"], q_dtype, h["q_scale"], h["kv"], kv_dtype, h["kv_scale"],
                                 h["qo_indptr"], h["kv_indptr"], heads=16, dqk=576, dv=512,
                                 sm_scale=sm, rows=rows)
    for i in range(3):
        assert np.array_equal(part[i], out[rows[0][i], rows[1][i]])
