"""Pins for the oracle's number-format decoders (CPU only).

Each decoder is checked against something other than itself: torch's CPU
float8 dtypes (a library routine), every code of each format, and the generic
minifloat decoder that e2m1 reuses is pinned on two 8-bit formats torch knows.
"""
import math
import os

import numpy as np
import pytest
import torch

from mla_decode_attention_split_gb300 import synth


def _torch_decode(codes_u8, dtype):
    return torch.from_numpy(codes_u8.copy()).view(dtype).double().numpy()


def _same(a, b):
    return np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(a[~np.isnan(a)], b[~np.isnan(b)])


def test_e4m3fn_all_codes_match_torch(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle_mod.decode_array("e4m3fn", codes)
    ref = _torch_decode(codes, torch.float8_e4m3fn)
    assert _same(ours, ref)
    # spot values of the OCP E4M3 definition: max 448, min subnormal 2^-9, min normal 2^-6
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6
    assert math.isnan(ours[0x7F]) and math.isnan(ours[0xFF])


def test_e8m0_all_codes_match_torch(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle_mod.decode_array("e8m0", codes)
    ref = _torch_decode(codes, torch.float8_e8m0fnu)
    assert _same(ours, ref)
    assert ours[127] == 1.0 and ours[0] == 2.0 ** -127


def test_bf16_all_bit_patterns_match_torch(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle_mod.decode_array("bf16", bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    assert _same(ours, ref)


@pytest.mark.parametrize("ebits,mbits,bias,tdtype", [(4, 3, 7, torch.float8_e4m3fn),
                                                     (5, 2, 15, torch.float8_e5m2)])
def test_generic_minifloat_matches_torch(oracle_mod, ebits, mbits, bias, tdtype):
    codes = np.arange(256, dtype=np.uint32)
    ours = oracle_mod.decode_array("minifloat", codes, params=(ebits, mbits, bias))
    ref = _torch_decode(codes.astype(np.uint8), tdtype)
    finite = np.isfinite(ref)
    # the generic decoder has no special codes: compare every finite code
    assert finite.sum() >= 240
    assert np.array_equal(ours[finite], ref[finite])


def test_e2m1_is_the_pinned_minifloat_with_ocp_grid(oracle_mod):
    nib = np.arange(16, dtype=np.uint8)
    ours = oracle_mod.decode_array("e2m1", nib)
    generic = oracle_mod.decode_array("minifloat", nib.astype(np.uint32), params=(2, 1, 1))
    assert np.array_equal(ours, generic)
    # OCP MX v1.0, FP4 E2M1: max normal 6.0, min subnormal 0.5, sign in bit 3
    assert ours.max() == 6.0 and ours.min() == -6.0
    assert sorted(set(np.abs(ours).tolist())) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert np.array_equal(ours[8:], -ours[:8])


def test_golden_constants_match_pages():
    path = os.path.join(os.path.dirname(__file__), "golden", "mla_config.txt")
    vals = {}
    for line in open(path):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = float(v)
    assert vals["num_heads"] == synth.HEADS
    assert vals["qk_head_dim"] == synth.D_QK == vals["kv_lora_rank"] + vals["qk_rope_head_dim"]
    assert vals["v_head_dim"] == synth.D_V == vals["kv_lora_rank"]
    assert abs(vals["sm_scale"] - synth.sm_scale_default()) < 1e-15
    assert abs(vals["log2e"] - 1.0 / math.log(2.0)) < 1e-8


# ---- the input generator's quantisers (not oracle code, but inputs depend on them)

def test_fp8_quantizer_rounds_to_nearest_and_saturates(oracle_mod):
    g = torch.Generator().manual_seed(5)
    x = torch.randn(4096, generator=g) * 3
    codes, scale = synth.quantize_fp8_per_tensor(x)
    dec = oracle_mod.decode_array("e4m3fn", codes.numpy()) * float(scale[0])
    assert float(scale[0]) == pytest.approx(float(x.abs().max()) / 448.0, rel=1e-7)
    assert np.abs(dec).max() == pytest.approx(float(x.abs().max()), rel=1e-6)
    # nearest: no other e4m3 code is closer to x / scale
    grid = oracle_mod.decode_array("e4m3fn", np.arange(256, dtype=np.uint8))
    grid = np.unique(grid[np.isfinite(grid)])
    xs = (x.double() / float(scale[0])).numpy()
    best = np.abs(grid[None, :] - xs[:, None]).min(axis=1)
    got = np.abs(dec / float(scale[0]) - xs)
    assert np.all(got <= best + 1e-12)


def test_mxfp4_quantizer_roundtrip_and_nearest(oracle_mod):
    g = torch.Generator().manual_seed(7)
    x = torch.randn(64, 576, generator=g)
    packed, sc = synth.quantize_mxfp4(x)
    assert packed.shape == (64, 288) and sc.shape == (64, 18)
    lo = (packed & 0xF).numpy()
    hi = (packed >> 4).numpy()
    nib = np.empty((64, 576), np.uint8)
    nib[:, 0::2], nib[:, 1::2] = lo, hi
    el = oracle_mod.decode_array("e2m1", nib)
    scale = oracle_mod.decode_array("e8m0", sc.numpy())
    dec = el * np.repeat(scale, 32, axis=1)
    # per block: amax maps into [4, 8) * 2^X, so no element saturates, and each
    # element is the nearest grid point of x / 2^X
    xs = x.double().numpy() / np.repeat(scale, 32, axis=1)
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -.5, -1, -1.5, -2, -3, -4, -6])
    best = np.abs(grid[None, :] - xs.reshape(-1, 1)).min(axis=1).reshape(xs.shape)
    got = np.abs(dec / np.repeat(scale, 32, axis=1) - xs)
    assert np.all(got <= best + 1e-12)
    # values already on the grid survive exactly
    onto = torch.from_numpy(dec).float()
    p2, s2 = synth.quantize_mxfp4(onto)
    assert torch.equal(p2, packed) and torch.equal(s2, sc)
