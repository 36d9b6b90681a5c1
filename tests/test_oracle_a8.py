"""Pins for the oracle's int8-activation linears (BitNest Table 1, "W4A8 ->
W8A8": the draft multiplies 4-bit base codes, the target the 8-bit codes,
both against int8 activations; Table 12).  Reading: per activation row
s = fp32(absmax / 127), code = clamp(rint(x / s), -127, 127).  Pins: the
quantiser's range and half-step bound; a one-hot row returns the decoded
weight column; the result stays within the activation rounding bound
(sum_k |w_k| s / 2) of the bf16 linear, for both planes."""
import numpy as np
import pytest

import oracle as O
from quantized_self_speculative_gb300 import synth


def test_activation_quantiser():
    x = synth.activations_bf16(1200, 6, 512)
    x[2] = 0                                            # a zero row
    xq, sx = O.quantize_act_int8(x)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    assert sx[2] == 0 and not xq[2].any()
    for m in (0, 1, 3, 4, 5):
        assert np.abs(xq[m]).max() == 127
        # half a step, plus the fp32 rounding of x / s (|x / s| <= 127, so one
        # unit of 2^-16 covers it)
        err = np.abs(xf[m] - np.float64(sx[m]) * xq[m].astype(np.float64))
        assert np.all(err <= np.float64(sx[m]) * (0.5 + 2.0 ** -16))


@pytest.mark.parametrize("verify", [False, True])
def test_one_hot_and_rounding_bound(verify):
    n, k, g = 64, 512, 128
    w = synth.weights(1201, n, k)
    base, resid, scales = O.pack_nested(w, g)
    cols = [0, 129, 511]
    x = np.zeros((3, k), np.uint16)
    for i, c in enumerate(cols):
        x[i, c] = synth.f32_to_bf16_bits(np.float32([2.5]))[0]
    xq, sx = O.quantize_act_int8(x)
    y = O.linear_a8(O.FMT_NESTED44, n, k, g, base, resid, scales, xq, sx, verify)
    ref = O.linear(O.FMT_NESTED44, n, k, g, base, resid, scales, x, verify)
    assert np.allclose(y, ref, rtol=1e-6, atol=0)
    xr = synth.activations_bf16(1202, 5, k)
    xq, sx = O.quantize_act_int8(xr)
    y = O.linear_a8(O.FMT_NESTED44, n, k, g, base, resid, scales, xq, sx, verify)
    ref = O.linear(O.FMT_NESTED44, n, k, g, base, resid, scales, xr, verify)
    # |w_deq| from one-hot columns of the same linear
    eye = np.zeros((k, k), np.uint16)
    eye[np.arange(k), np.arange(k)] = synth.f32_to_bf16_bits(np.float32([1.0]))[0]
    wd = O.linear(O.FMT_NESTED44, n, k, g, base, resid, scales, eye, verify)   # [k][n]
    bound = np.abs(wd).sum(axis=0)[None, :] * (sx[:, None] / 2)
    assert np.all(np.abs(y - ref) <= bound * (1 + 1e-9))
    assert np.abs(y - ref).max() > 0
