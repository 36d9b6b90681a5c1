"""Pins for the oracle's number formats (fp16, bf16, E4M3FN) against
independent library conversions and the format definitions."""
import numpy as np
import pytest
import torch

import oracle as O
from quantized_self_speculative_gb300 import synth


def test_f32_to_f16_matches_numpy_rne():
    g = synth.rng(11)
    x = np.concatenate([
        g.standard_normal(200_000).astype(np.float32) * np.float32(1000),
        g.standard_normal(50_000).astype(np.float32) * np.float32(1e-5),    # subnormal range
        np.array([0.0, -0.0, 65504, 65519.996, 65520, 1e9, -1e9, 2**-24, 2**-25, 3 * 2**-26,
                  1.0 + 2**-11, 1.0 + 3 * 2**-11, 2048 + 1, 2048 + 3], np.float32),
    ])
    ours = O.f32_to_f16_bits(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_f16_to_f32_exhaustive():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = O.f16_bits_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_decode_exhaustive_against_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = O.e4m3_to_f32(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2                      # S.1111.111 only
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_e4m3_encode_rne_in_range_against_torch():
    # every value in range: all codes, midpoints between neighbours, random values
    vals = O.e4m3_to_f32(np.arange(256, dtype=np.uint8))
    finite = np.sort(vals[np.isfinite(vals)])
    mids = ((finite[1:].astype(np.float64) + finite[:-1]) / 2).astype(np.float32)
    g = synth.rng(12)
    rnd = (g.standard_normal(200_000) * 100).astype(np.float32)
    rnd = rnd[np.abs(rnd) <= 448]
    x = np.concatenate([finite, mids, np.nextafter(mids, np.float32(np.inf)),
                        np.nextafter(mids, np.float32(-np.inf)), rnd]).astype(np.float32)
    ours = O.f32_to_e4m3(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_encode_saturates():
    x = np.array([448, 449, 463.9, 464, 480, 1e9, np.inf, -449, -1e9, -np.inf, np.nan], np.float32)
    out = O.f32_to_e4m3(x)
    assert list(out[:7]) == [0x7E] * 7
    assert list(out[7:10]) == [0xFE] * 3
    assert out[10] == 0x7F


def test_bf16_helper_matches_torch():
    g = synth.rng(13)
    x = g.standard_normal(100_000).astype(np.float32) * np.float32(7)
    ours = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = synth.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())
