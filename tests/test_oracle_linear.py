"""Pins for the oracle's dequantised linear (C2).

Draft pass: base plane only; verify pass: both planes, i.e. the 8-bit target
(BitNest, Fig. 2 and Fig. 3).  FP8 / FP16 tiers: SpecQuant Sec. III.A.
The pins decode the packed planes by the format definition (bit operations in
this file) and multiply with a library matmul -- a different route from the
oracle's grouped fp64 loop.
"""
import numpy as np
import pytest
import torch

import oracle as O
from quantized_self_speculative_gb300 import synth
from test_oracle_pack import nibbles


def decoded(base, resid, scales, n, k, g, verify):
    s = np.repeat(O.f16_bits_to_f32(scales).reshape(n, k // g).astype(np.float64), g, axis=1)
    q4 = nibbles(base).astype(np.float64)
    if not verify:
        return s * q4
    return s / 16 * (16 * q4 + nibbles(resid))


@pytest.mark.parametrize("g,M", [(128, 1), (128, 5), (64, 16), (64, 3)])
def test_nested_linear_equals_decoded_matmul(g, M):
    n, k = 72, 768
    w = synth.weights(31, n, k)
    base, resid, scales = O.pack_nested(w, g)
    x = synth.activations_bf16(32, M, k)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    for verify in (False, True):
        y = O.linear(O.FMT_NESTED44, n, k, g, base, resid, scales, x, verify)
        ref = xf @ decoded(base, resid, scales, n, k, g, verify).T
        assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_one_hot_returns_decoded_column_exactly():
    n, k, g = 16, 256, 128
    w = synth.weights(33, n, k)
    base, resid, scales = O.pack_nested(w, g)
    one = synth.f32_to_bf16_bits(np.float32([1.0]))[0]
    for col in (0, 1, 127, 128, 255):
        x = np.zeros((1, k), np.uint16)
        x[0, col] = one
        for verify in (False, True):
            y = O.linear(O.FMT_NESTED44, n, k, g, base, resid, scales, x, verify)
            assert np.array_equal(y[0], decoded(base, resid, scales, n, k, g, verify)[:, col])


def test_zero_weights_give_zero():
    n, k, g = 8, 256, 64
    base, resid, scales = O.pack_nested(np.zeros((n, k), np.float32), g)
    x = synth.activations_bf16(34, 2, k)
    assert np.all(O.linear(O.FMT_NESTED44, n, k, g, base, resid, scales, x, True) == 0)


def test_row_subset_matches_full():
    n, k, g = 50, 512, 128
    w = synth.weights(35, n, k)
    base, resid, scales = O.pack_nested(w, g)
    x = synth.activations_bf16(36, 5, k)
    full = O.linear(O.FMT_NESTED44, n, k, g, base, resid, scales, x, True)
    rows = np.array([49, 0, 17, 17, 3], np.int32)
    sub = O.linear(O.FMT_NESTED44, n, k, g, base, resid, scales, x, True, rows=rows)
    assert np.array_equal(sub, full[:, rows])


def test_verify_tracks_fp32_weights_better_than_draft():
    n, k, g = 64, 1024, 128
    w = synth.weights(37, n, k)
    base, resid, scales = O.pack_nested(w, g)
    x = synth.activations_bf16(38, 5, k)
    true = synth.bf16_bits_to_f32(x).astype(np.float64) @ w.astype(np.float64).T
    yd = O.linear(O.FMT_NESTED44, n, k, g, base, resid, scales, x, False)
    yv = O.linear(O.FMT_NESTED44, n, k, g, base, resid, scales, x, True)
    assert np.abs(yv - true).max() < np.abs(yd - true).max() / 8


def test_int4_equals_nested_draft():
    n, k, g = 40, 512, 128
    w = synth.weights(39, n, k)
    base, resid, scales = O.pack_nested(w, g)
    x = synth.activations_bf16(40, 3, k)
    a = O.linear(O.FMT_INT4, n, k, g, base, None, scales, x, False)
    b = O.linear(O.FMT_NESTED44, n, k, g, base, resid, scales, x, False)
    assert np.array_equal(a, b)
    with pytest.raises(ValueError):
        O.linear(O.FMT_INT4, n, k, g, base, None, scales, x, True)


def test_fp8_linear_equals_library_decode():
    n, k = 24, 512
    w = synth.weights(41, n, k)
    codes, scale = O.pack_fp8(w)
    x = synth.activations_bf16(42, 7, k)
    y = O.linear(O.FMT_FP8, n, k, 0, codes, None, scale, x, True)
    wdec = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy() * scale[:, None].astype(np.float64)
    ref = synth.bf16_bits_to_f32(x).astype(np.float64) @ wdec.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_fp16_linear_equals_library_decode():
    n, k = 24, 512
    w = synth.weights(43, n, k)
    w16 = O.pack_fp16(w)
    x = synth.activations_bf16(44, 9, k)
    y = O.linear(O.FMT_FP16, n, k, 0, w16, None, None, x, True)
    ref = synth.bf16_bits_to_f32(x).astype(np.float64) @ w16.view(np.float16).astype(np.float64).T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
