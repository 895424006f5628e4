"""Pins of the oracle's number-format decoders and its E4M3 encoder.

The decoders are pinned to the published format tables (golden files) and to
PyTorch's independent float8 / bfloat16 conversions; the encoder to PyTorch's
float8_e4m3fn rounding inside the finite range and to the OFP8 "satfinite"
rule outside it.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden


def _val(s):
    return float("nan") if s == "nan" else float(s)


def test_e4m3_spec_points():
    for code, value, *_ in read_golden("ofp8_e4m3.txt"):
        got = oracle.e4m3_decode(np.array([int(code, 16)], np.uint8))[0]
        want = _val(value)
        if math.isnan(want):
            assert math.isnan(got), code
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), code


def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # exactly two NaN codes and no infinities in E4M3
    assert nan.sum() == 2 and not np.isinf(ours).any()


def test_e4m3_encode_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    back = oracle.e4m3_encode(vals)
    assert np.array_equal(back, codes)


def test_e4m3_encode_matches_torch_rne():
    rng = np.random.default_rng(7)
    # all midpoints between neighbouring finite positive codes (ties to even),
    # values just around them, a log-uniform sweep and subnormals
    pos = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (pos[1:] + pos[:-1]) / 2
    vals = np.concatenate([mids, np.nextafter(mids, 0), np.nextafter(mids, 1000),
                           np.exp(rng.uniform(np.log(1e-4), np.log(460), 20000)),
                           rng.uniform(0, 2 ** -6, 2000)]).astype(np.float32)
    vals = np.concatenate([vals, -vals])
    vals = vals[np.abs(vals) <= 464]  # torch does not saturate beyond the last tie
    ours = oracle.e4m3_encode(vals)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_encode_saturates():
    vals = np.array([464.0001, 479.0, 480.0, 1e6, np.inf], np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), np.full(5, 0x7E, np.uint8))
    assert np.array_equal(oracle.e4m3_encode(-vals), np.full(5, 0xFE, np.uint8))


def test_e2m1_e8m0_tables():
    for kind, code, value in read_golden("mx_e2m1_e8m0.txt"):
        c = int(code, 16)
        got = oracle.e2m1_decode(c) if kind == "e2m1" else oracle.e8m0_decode(c)
        want = _val(value)
        if math.isnan(want):
            assert math.isnan(got)
        else:
            assert got == want, (kind, code)


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 65536, 97, dtype=np.int64).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    ours = np.array([oracle.bf16_decode(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_is_exact_in_f16_and_bf16():
    """Every finite E4M3 value is exactly representable in fp16 and bf16 (the
    sparse-attention kernel lifts latents into 16-bit operands)."""
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    v = oracle.e4m3_decode(codes)
    assert np.array_equal(v.astype(np.float16).astype(np.float64), v)
    assert np.array_equal(torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy(), v)
