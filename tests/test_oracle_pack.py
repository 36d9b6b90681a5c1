"""Pins for the oracle's nested quantise/pack (C1).

BitNest, Fig. 2: a b-bit base plus an r-bit refinement of the remaining error;
Fig. 3: two independent 4-bit planes of N/2 bytes each, the target recovers
the full 8-bit representation.  The pages fix neither the scale nor the
rounding; the reading pinned here: s = fp16(absmax / 7) per group, rint
(half to even), refinement step s/16.
"""
import numpy as np
import pytest

import oracle as O
from quantized_self_speculative_gb300 import synth


def nibbles(plane: np.ndarray) -> np.ndarray:
    """Signed two's-complement nibbles of a packed plane, element 2j = low nibble."""
    lo = (plane & 0x0F).astype(np.int16)
    hi = (plane >> 4).astype(np.int16)
    out = np.empty(plane.shape[:-1] + (plane.shape[-1] * 2,), np.int16)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return np.where(out >= 8, out - 16, out)


def test_every_nibble_pair_reconstructs_a_unique_8bit_code():
    # all 256 (base, refinement) nibble pairs -> 16*q4 + r covers 256 distinct
    # integers in [-136, 119]: the two planes together carry a full 8-bit code
    codes = set()
    for bn in range(16):
        for rn in range(16):
            q4, r = O.nibble_value(bn), O.nibble_value(rn)
            assert -8 <= q4 <= 7 and -8 <= r <= 7
            assert (q4 & 15) == bn and (r & 15) == rn
            codes.add(16 * q4 + r)
    assert len(codes) == 256 and min(codes) == -136 and max(codes) == 119


@pytest.mark.parametrize("g", [64, 128])
def test_exact_multiples_round_trip(g):
    """Weights that are exact multiples of s/16 (s a power of two, so fp16(absmax/7)
    is exact) must come back as the very codes they were built from."""
    s = 2.0 ** -6
    gen = synth.rng(21)
    n = 12
    q4 = gen.integers(-7, 8, size=(n, g))
    r = gen.integers(-7, 8, size=(n, g))
    q4[:, 0], r[:, 0] = 7, 0                    # absmax = 7 s exactly -> scale s
    # keep |16 q4 + r| <= 112 so no weight exceeds the group absmax 7 s
    over = np.abs(16 * q4 + r) > 112
    r[over] = 0
    w = ((16 * q4 + r) * (s / 16)).astype(np.float32)
    base, resid, scales = O.pack_nested(w, g)
    assert np.all(O.f16_bits_to_f32(scales) == np.float32(s))
    assert np.array_equal(nibbles(base), q4)
    assert np.array_equal(nibbles(resid), r)


@pytest.mark.parametrize("g", [64, 128])
def test_plane_sizes_and_error_bounds(g):
    n, k = 96, 1024
    w = synth.weights(3, n, k)
    base, resid, scales = O.pack_nested(w, g)
    assert base.nbytes == n * k // 2 and resid.nbytes == n * k // 2      # N/2 bytes per plane
    assert scales.shape == (n, k // g)
    s = np.repeat(O.f16_bits_to_f32(scales).reshape(n, k // g), g, axis=1).astype(np.float64)
    q4 = nibbles(base).astype(np.float64)
    r = nibbles(resid).astype(np.float64)
    wd = w.astype(np.float64)
    # base: round-to-nearest on the group grid
    assert np.all(np.abs(wd - s * q4) <= s * (0.5 + 1e-6))
    # target (8-bit): within half a refinement step, except where the signed
    # refinement saturates at +7 (16 (x - q4) rounds to +8, i.e. the base's
    # rounding error lies in [15/32, 1/2] of a step); there it is within s/16
    err_t = np.abs(wd - s / 16 * (16 * q4 + r))
    x = wd / s
    saturated = 16 * (x - q4) >= 7.5 - 1e-4
    assert np.all(err_t[~saturated] <= s[~saturated] / 32 * (1 + 1e-5))
    assert np.all(err_t[saturated] <= s[saturated] / 16 * (1 + 1e-5))
    assert np.all(r[saturated] == 7)
    assert 0.02 < saturated.mean() < 0.045                       # about 1/32 of N(0, .02) weights
    # the target is far closer to W than the draft (higher precision recovered by refinement)
    assert np.linalg.norm(wd - s / 16 * (16 * q4 + r)) < np.linalg.norm(wd - s * q4) / 8


def test_scale_is_fp16_of_absmax_over_7():
    w = synth.weights(4, 8, 256)
    _, _, scales = O.pack_nested(w, 128)
    amax = np.abs(w.reshape(8, 2, 128)).max(axis=2)
    expect = (amax / np.float32(7)).astype(np.float32).astype(np.float16).view(np.uint16)
    assert np.array_equal(scales, expect)


def test_zero_group_and_single_nonzero():
    w = np.zeros((2, 128), np.float32)
    w[1, 5] = -0.3
    base, resid, scales = O.pack_nested(w, 128)
    assert np.all(base[0] == 0) and np.all(resid[0] == 0) and scales[0, 0] == 0
    q4 = nibbles(base)[1]
    assert q4[5] == -7 and np.count_nonzero(q4) == 1


def test_int4_tier_is_the_base_plane():
    w = synth.weights(5, 40, 512)
    b1, _, s1 = O.pack_nested(w, 128)
    b2, r2, s2 = O.pack_nested(w, 128, with_resid=False)
    assert r2 is None and np.array_equal(b1, b2) and np.array_equal(s1, s2)


def test_fp8_pack_pins():
    w = synth.weights(6, 16, 512)
    codes, scale = O.pack_fp8(w)
    amax = np.abs(w).max(axis=1)
    assert np.array_equal(scale, (amax / np.float32(448)).astype(np.float32))
    dec = O.e4m3_to_f32(codes.ravel()).reshape(codes.shape)
    assert np.all(np.isfinite(dec)) and np.abs(dec).max() <= 448
    # RNE relative error of E4M3 (3 mantissa bits) is at most 2^-4 for normals
    recon = dec * scale[:, None]
    big = np.abs(w) > scale[:, None] * 2 ** -6
    assert np.all(np.abs(recon[big] - w[big]) <= np.abs(w[big]) * 2 ** -4 * (1 + 1e-6))
    # the row maximum maps to +-448 exactly
    idx = np.abs(w).argmax(axis=1)
    assert np.all(np.abs(dec[np.arange(16), idx]) == 448)


def test_fp16_pack_is_rne():
    w = synth.weights(7, 8, 256)
    assert np.array_equal(O.pack_fp16(w), w.astype(np.float16).view(np.uint16))


def test_non_finite_weights_rejected():
    w = synth.weights(8, 4, 128)
    w[2, 7] = np.nan
    with pytest.raises(ValueError):
        O.pack_nested(w, 128)
