"""Pins for the oracle's nested-KV attention (BitNest, Fig. 4: the draft reads
the low-bit base view of the cache, verification the full view; the rows are
quantised like the weights, Fig. 2).  Closed forms: one visible row returns
that row's value vector; zero queries weight the visible rows uniformly; a
dominant score selects its row; causal rows see one more row each; the
8-bit view stays within s/16 of the stored values, the 4-bit view within s/2."""
import math

import numpy as np
import pytest

import oracle as O
from quantized_self_speculative_gb300 import synth


def make_cache(B, Hkv, L, d, G, seed):
    g = synth.rng(seed)
    K = g.standard_normal((B, Hkv, L, d)).astype(np.float32)
    V = g.standard_normal((B, Hkv, L, d)).astype(np.float32)
    kb, kr, ks = O.kv_rows_pack(K, G)
    vb, vr, vs = O.kv_rows_pack(V, G)
    return K, V, dict(k_base=kb, k_resid=kr, k_scales=ks, v_base=vb, v_resid=vr, v_scales=vs)


def dequant(base, resid, scales, G, planes):
    lo = (base & 15).astype(np.int32)
    hi = (base >> 4).astype(np.int32)
    q4 = np.stack([lo, hi], -1).reshape(*base.shape[:-1], -1)
    q4 = np.where(q4 > 7, q4 - 16, q4)
    s = np.repeat(O.f16_bits_to_f32(scales.reshape(-1)).reshape(scales.shape).astype(np.float64), G, axis=-1)
    if planes == 1:
        return s * q4
    lo = (resid & 15).astype(np.int32)
    hi = (resid >> 4).astype(np.int32)
    r = np.stack([lo, hi], -1).reshape(*resid.shape[:-1], -1)
    r = np.where(r > 7, r - 16, r)
    return s / 16 * (16 * q4 + r)


@pytest.mark.parametrize("planes", [1, 2])
def test_uniform_scores_average_the_visible_rows(planes):
    B, Hkv, L, d, G, M = 2, 2, 40, 64, 64, 3
    K, V, c = make_cache(B, Hkv, L, d, G, 900)
    lens = np.array([40, 17], np.int32)
    q = np.zeros((B, M, Hkv * 3, d), np.float32)            # GQA: three query heads per kv head
    out = O.attn_decode(q, c, lens, planes, 0.125)
    Vd = dequant(c["v_base"], c["v_resid"], c["v_scales"], G, planes)
    for b in range(B):
        for m in range(M):
            lim = lens[b] - (M - 1 - m)                       # causal: one more row per query row
            for h in range(Hkv * 3):
                ref = Vd[b, h // 3, :lim].mean(axis=0)
                assert np.allclose(out[b, m, h], ref, rtol=1e-6, atol=1e-7)
    # the 8-bit view is within s/16 of the stored rows, the 4-bit view within s/2
    s = np.repeat(O.f16_bits_to_f32(c["v_scales"].reshape(-1)).reshape(c["v_scales"].shape), G, axis=-1)
    bound = s / 16 if planes == 2 else s / 2
    assert np.all(np.abs(Vd - V) <= bound + 1e-7)


def test_one_visible_row_and_a_dominant_score():
    B, Hkv, L, d, G = 1, 1, 9, 128, 128
    K, V, c = make_cache(B, Hkv, L, d, G, 901)
    Vd = dequant(c["v_base"], c["v_resid"], c["v_scales"], G, 2)
    q = synth.rng(902).standard_normal((1, 1, 1, d)).astype(np.float32)
    out = O.attn_decode(q, c, np.array([1], np.int32), 2, 0.1)   # only row 0 visible
    assert np.allclose(out[0, 0, 0], Vd[0, 0, 0], rtol=1e-6, atol=1e-7)
    Kd = dequant(c["k_base"], c["k_resid"], c["k_scales"], G, 2)
    q = (Kd[0, 0, 5] * 1000.0).astype(np.float32)[None, None, None]   # row 5's score dominates
    out = O.attn_decode(q, c, np.array([9], np.int32), 2, 1.0)
    assert np.allclose(out[0, 0, 0], Vd[0, 0, 5], rtol=1e-5, atol=1e-6)


def test_softmax_weights_closed_form_two_rows():
    """Two visible rows with scores a and b: out = (e^a v0 + e^b v1) / (e^a + e^b)."""
    B, Hkv, L, d, G = 1, 1, 2, 64, 64
    K, V, c = make_cache(B, Hkv, L, d, G, 903)
    Kd = dequant(c["k_base"], c["k_resid"], c["k_scales"], G, 1)
    Vd = dequant(c["v_base"], c["v_resid"], c["v_scales"], G, 1)
    q = synth.rng(904).standard_normal((1, 1, 1, d)).astype(np.float32)
    out = O.attn_decode(q, c, np.array([2], np.int32), 1, 0.3)
    a, b = (0.3 * Kd[0, 0] @ q[0, 0, 0].astype(np.float64))
    w0 = 1.0 / (1.0 + math.exp(b - a))
    assert np.allclose(out[0, 0, 0], w0 * Vd[0, 0, 0] + (1 - w0) * Vd[0, 0, 1], rtol=1e-6, atol=1e-7)
