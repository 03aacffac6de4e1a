"""The threaded per-segment driver of the oracle (used by the full-size parity
tests) gives exactly what one oracle call over the whole batch gives."""
import numpy as np
import pytest

import oracle
import oracle_parallel
from mla_decode_attention_split_gb300 import synth


@pytest.mark.parametrize("q_dtype,kv_dtype", [(synth.BF16, synth.BF16), (synth.BF16, synth.FP8_E4M3),
                                              (synth.FP8_E4M3, synth.FP8_E4M3), (synth.BF16, synth.MXFP4)])
def test_threaded_segments_equal_one_call(oracle_mod, q_dtype, kv_dtype):
    w = synth.Workload("threads", 6, 1, 0, q_dtype, kv_dtype, seed=4)
    inp = synth.make_inputs(w, "cpu", kv_lens=[40, 0, 7, 130, 1, 65], q_lens=[2, 1, 0, 3, 1, 1])
    h = synth.to_host_codes(inp)
    sm = synth.sm_scale_default()
    whole = oracle.mla_decode(h["q"], h["q_dtype"], h["q_scale"], h["kv"], h["kv_dtype"], h["kv_scale"],
                              h["qo_indptr"], h["kv_indptr"], heads=16, dqk=576, dv=512, sm_scale=sm)
    got = oracle_parallel.decode_segments(h, sm, workers=4)
    assert np.array_equal(got, whole)
    rel = oracle_parallel.per_segment_rel_l2(got, whole, h["qo_indptr"])
    assert np.isnan(rel[2]) and np.all(rel[np.isfinite(rel)] == 0)
