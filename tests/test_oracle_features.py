"""Pins for the oracle's draft features (SpecKV, "How it works": the mean and
maximum draft entropy and the mean and minimum draft confidence over a
step's drafted positions, fed to the acceptance-rate predictor that picks
gamma).  Closed forms: a uniform draft has entropy ln V and confidence 1/V;
a two-point draft has the binary entropy; temperature divides the logits."""
import math

import numpy as np
import pytest

import oracle as O
from quantized_self_speculative_gb300 import synth


def test_uniform_and_point_mass():
    V, k = 1000, 3
    dl = np.zeros((1, k, V), np.float32)
    f = O.draft_features(np.zeros((1, k), np.int32), dl)
    assert np.allclose(f[0], [math.log(V), 1 / V, math.log(V), 1 / V], rtol=1e-12)
    dl[0, :, 17] = 200.0                      # all mass on token 17
    f = O.draft_features(np.full((1, k), 17, np.int32), dl)
    assert f[0, 0] < 1e-60 and f[0, 1] == 1.0 and f[0, 3] == 1.0


@pytest.mark.parametrize("p", [0.5, 0.9, 0.99])
def test_two_point_binary_entropy_and_aggregates(p):
    V, k = 8, 4
    dl = np.full((1, k, V), -1e4, np.float32)
    dl[0, :, 2] = math.log(p)
    dl[0, :, 5] = math.log(1 - p)
    dl[0, 3, :] = 0.0                         # the last position is uniform
    d = np.array([[2, 5, 2, 0]], np.int32)
    f = O.draft_features(d, dl)[0]
    hb = -p * math.log(p) - (1 - p) * math.log(1 - p)
    hs = [hb, hb, hb, math.log(V)]
    cs = [p, 1 - p, p, 1 / V]
    assert np.allclose(f, [np.mean(hs), np.mean(cs), max(hs), min(cs)], rtol=1e-6)


def test_temperature_scales_the_logits():
    dl = synth.target_logits(800, 2, 2, 300, 2.0)[:, :2]
    d = synth.draft_tokens_greedy(dl)
    a = O.draft_features(d, dl, temperature=0.5)
    b = O.draft_features(d, (dl * 2.0).astype(np.float32), temperature=1.0)
    assert np.allclose(a, b, rtol=1e-6)
    hot = O.draft_features(d, dl, temperature=1e4)
    assert np.allclose(hot[:, 0], math.log(300), rtol=1e-3)
