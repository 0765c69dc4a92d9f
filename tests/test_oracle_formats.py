"""Pins of the oracle's number formats against library routines.

The oracle's own bf16 rounding and E4M3 encoder/decoder (written from the
format definitions) are checked against torch's bfloat16 and float8_e4m3fn
conversions, which are independent implementations of the same formats.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _torch_bf16_bits(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_round_matches_torch_random_and_ties():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),  # subnormals
    ])
    # exact ties: low 16 bits == 0x8000, with even and odd kept parts
    base = rng.integers(0, 0x7f7f, 500, dtype=np.uint32) << 16
    ties = (base | 0x8000).view(np.float32)
    vals = np.concatenate([vals, ties, -ties])
    ref = _torch_bf16_bits(vals)
    got = np.array([oracle.f32_to_bf16(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_specials():
    assert oracle.f32_to_bf16(float("inf")) == 0x7F80
    assert oracle.f32_to_bf16(float("-inf")) == 0xFF80
    assert math.isnan(oracle.bf16_to_f32(oracle.f32_to_bf16(float("nan"))))
    assert oracle.f32_to_bf16(0.0) == 0 and oracle.f32_to_bf16(-0.0) == 0x8000
    # largest finite fp32 rounds up to inf in bf16, as RNE demands
    assert oracle.f32_to_bf16(3.4028234663852886e38) == 0x7F80


def test_bf16_widen_is_exact():
    for b in [0x0000, 0x3F80, 0xBF80, 0x0001, 0x7F7F, 0x4049]:
        f = np.array([b], np.uint16).view(np.int16)
        ref = torch.from_numpy(f).view(torch.bfloat16).float().item()
        assert oracle.bf16_to_f32(b) == ref


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    got = np.array([oracle.e4m3_to_f32(int(c)) for c in codes], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert nan.sum() == 2  # S.1111.111
    assert np.array_equal(got[~nan], ref[~nan])
    assert oracle.e4m3_to_f32(0x7E) == 448.0 and oracle.e4m3_to_f32(0x08) == 2.0 ** -6
    assert oracle.e4m3_to_f32(0x01) == 2.0 ** -9


def test_e4m3_encode_every_bf16_value_matches_torch():
    # every bf16 bit pattern with |v| <= 464 (above that torch does not saturate)
    bits = np.arange(65536, dtype=np.uint32)
    vals = (bits << 16).astype(np.uint32).view(np.float32)
    keep = np.isfinite(vals) & (np.abs(vals) <= 464.0)
    vals = vals[keep]
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.f32_to_e4m3(float(v)) for v in vals], np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_encode_random_fp32_and_midpoints_match_torch():
    rng = np.random.default_rng(2)
    vals = np.concatenate([
        (rng.standard_normal(6000) * 100).astype(np.float32),
        (rng.standard_normal(3000) * 1e-2).astype(np.float32),
        rng.uniform(-464, 464, 3000).astype(np.float32),
    ])
    # exact midpoints between neighbouring finite codes (ties go to even)
    finite = np.array([oracle.e4m3_to_f32(c) for c in range(0, 0x7E + 1)], np.float64)
    mids = ((finite[:-1] + finite[1:]) / 2).astype(np.float32)
    vals = np.concatenate([vals, mids, -mids])
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.f32_to_e4m3(float(v)) for v in vals], np.uint8)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("v,code", [(448.0, 0x7E), (464.0, 0x7E), (470.0, 0x7E), (1e9, 0x7E),
                                    (-1e9, 0xFE), (float("inf"), 0x7E), (float("-inf"), 0xFE)])
def test_e4m3_satfinite(v, code):
    # saturation to the largest finite magnitude, by the format's definition
    assert oracle.f32_to_e4m3(v) == code


def test_e4m3_nan_maps_to_nan_code():
    assert oracle.f32_to_e4m3(float("nan")) & 0x7F == 0x7F
