"""FP8 (E4M3) KV, host side: the oracle's decoding of the format and its
dequantised decode, pinned to the format definition, a library conversion and
closed forms.

FD++ §4 (quantisation-friendly fusion): the K/V cache is held in FP8 in HBM
and dequantised in registers before the attention arithmetic.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from workloads import make_small, to_fp8


def test_e4m3_matches_the_library_conversion_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_float(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    ok = ~np.isnan(lib)
    assert np.array_equal(ours[ok], lib[ok])
    assert np.array_equal(np.signbit(ours[ok]), np.signbit(lib[ok]))


def test_e4m3_format_landmarks():
    v = oracle.e4m3_to_float(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x7E, 0x7F, 0x80, 0xFE, 0xFF],
                                      dtype=np.uint8))
    assert v[0] == 0.0 and v[1] == 2.0 ** -9 and v[2] == 7 * 2.0 ** -9   # subnormals m/8 * 2^-6
    assert v[3] == 2.0 ** -6                                             # smallest normal
    assert v[4] == 1.0 and v[5] == 448.0 and math.isnan(v[6])
    assert v[7] == 0.0 and np.signbit(v[7]) and v[8] == -448.0 and math.isnan(v[9])
    pos = oracle.e4m3_to_float(np.arange(0, 127, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0), "codes 0..126 are increasing magnitudes"


def test_dequant_takes_each_heads_own_scale():
    codes = np.full((3, 2, 4), 0x38, dtype=np.uint8)          # every code is 1.0
    out = oracle.dequant_fp8(codes, np.array([0.5, 3.0], dtype=np.float32))
    assert np.all(out[:, 0] == 0.5) and np.all(out[:, 1] == 3.0)


def _fp8_case(seed=3):
    inp = make_small(2, 8, 2, 128, [70, 33], seed=seed)
    return to_fp8(inp)


def test_decode_fp8_is_decode_on_the_dequantised_values():
    f = _fp8_case()
    o, lse = oracle.decode_fp8(f["q"], f["k_fp8"], f["v_fp8"], f["k_scale"], f["v_scale"],
                               f["kv_indptr"], f["scale"])
    k = torch.from_numpy(oracle.dequant_fp8(f["k_fp8"], f["k_scale"]))
    v = torch.from_numpy(oracle.dequant_fp8(f["v_fp8"], f["v_scale"]))
    o2, lse2 = oracle.decode(f["q"].double(), k, v, f["kv_indptr"], f["scale"])
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_scales_enter_as_logit_and_output_factors():
    """s_j = scale * q . (c_k K_j) and O = c_v sum p_j V_j: doubling every K
    scale equals doubling q; doubling every V scale doubles O, LSE unchanged."""
    f = _fp8_case(5)
    args = (f["kv_indptr"], f["scale"])
    o, lse = oracle.decode_fp8(f["q"], f["k_fp8"], f["v_fp8"], f["k_scale"], f["v_scale"], *args)
    ok, lk = oracle.decode_fp8(f["q"], f["k_fp8"], f["v_fp8"], f["k_scale"] * 2, f["v_scale"], *args)
    oq, lq = oracle.decode_fp8(f["q"].double() * 2, f["k_fp8"], f["v_fp8"], f["k_scale"],
                               f["v_scale"], *args)
    assert np.allclose(ok, oq, rtol=0, atol=1e-12) and np.allclose(lk, lq, rtol=0, atol=1e-12)
    ov, lv = oracle.decode_fp8(f["q"], f["k_fp8"], f["v_fp8"], f["k_scale"], f["v_scale"] * 2, *args)
    assert np.allclose(ov, 2 * o, rtol=0, atol=1e-12) and np.allclose(lv, lse, rtol=0, atol=1e-12)


def test_quantisation_error_is_within_half_an_e4m3_step():
    f = _fp8_case(7)
    for name in ("k", "v"):
        x = f[name].double().numpy()
        deq = oracle.dequant_fp8(f[name + "_fp8"], f[name + "_scale"])
        s = f[name + "_scale"].double().numpy().reshape(1, -1, 1)
        # relative 2^-4 for normals (3 mantissa bits), absolute 2^-10 * scale below 2^-6
        bound = np.maximum(np.abs(x) * 2.0 ** -4, s * 2.0 ** -10)
        assert np.all(np.abs(deq - x) <= bound * (1 + 1e-9))
        assert not np.any(np.isnan(deq))
        assert np.isclose(np.abs(deq).max(axis=(0, 2)), 448 * s.reshape(-1)).all()
