"""Pins for the oracle's sampled acceptance (C4) and its canonical arithmetic.

"How Speculative Decoding Speeds Up Inference": speculative sampling
(Leviathan et al.; Chen et al.) accepts each draft token with a probability
set by both models' scores, resamples from a corrected distribution after a
rejection, and then follows the target distribution exactly; Eq. (1) gives the
expected tokens per pass under i.i.d. acceptance.  Philox4x32-10 is pinned to
its published known-answer vectors.
"""
import os
from fractions import Fraction

import mpmath
import numpy as np
import pytest
from scipy import stats

import oracle as O
from conftest import GOLDEN
from quantized_self_speculative_gb300 import synth

ULP = 2.0 ** -23


# ------------------------------------------------------------------ Philox
def test_philox_known_answer_vectors():
    n = 0
    for line in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")):
        if line.startswith("#") or not line.strip():
            continue
        v = [int(t, 16) for t in line.split()]
        assert list(O.philox4x32_10(v[0:4], v[4:6])) == v[6:10]
        n += 1
    assert n == 3


def test_uniform_layout_and_range():
    seeds = synth.rng(80).integers(0, 2**63, size=2000, dtype=np.uint64)
    u = O.uniforms(seeds, 3, 1, 77)
    assert np.all((u >= 0) & (u < 1))
    assert np.all(u * 2**24 == np.floor(u * 2**24))             # multiples of 2^-24
    assert abs(u.mean() - 0.5) < 0.03
    # the uniform is word 0 of Philox(key = seed halves, ctr = (j, purpose, round lo, hi)) >> 8
    s = int(seeds[5])
    w = O.philox4x32_10([3, 1, 77, 0], [s & 0xFFFFFFFF, s >> 32])
    assert u[5] == (w[0] >> 8) * 2.0**-24
    # each counter field and the round's high word matter
    base = O.uniform(12345, 2, 0, 9)
    assert len({base, O.uniform(12346, 2, 0, 9), O.uniform(12345, 3, 0, 9),
                O.uniform(12345, 2, 1, 9), O.uniform(12345, 2, 0, 10),
                O.uniform(12345, 2, 0, 9 + 2**32)}) == 6


# ------------------------------------------------------------------ exp2
def test_exp2_coefficients_are_correctly_rounded_taylor_terms():
    with mpmath.workprec(200):
        ln2 = mpmath.log(2)
        exact = [ln2 ** i / mpmath.factorial(i) for i in range(7)]
    with mpmath.workprec(24):                      # binary32 significand, round to nearest
        rn = [float(+e) for e in exact]
    assert [O.exp2_coef(i) for i in range(7)] == [np.float32(v) for v in rn]


def test_exp2_accuracy_and_special_values():
    t = np.concatenate([np.linspace(-125, 0.5, 400_001, dtype=np.float32),
                        -synth.rng(81).random(100_000).astype(np.float32) * 20])
    e = O.exp2c(t)
    ref = np.exp2(t.astype(np.float64))
    rel = np.abs(e - ref) / ref
    assert rel.max() < 3 * ULP
    assert O.exp2c([0.0])[0] == 1.0
    assert np.all(O.exp2c([-125.0001, -126, -1000, -3.0e38]) == 0.0)
    assert O.exp2c([-125.0])[0] == np.float32(2.0 ** -125)
    assert O.exp2c([-1.0])[0] == 0.5 and O.exp2c([-10.0])[0] == 2.0 ** -10


# ------------------------------------------------------------------ softmax / trees
def softmax64(l, T=1.0):
    z = l.astype(np.float64) / T
    z -= z.max()
    p = np.exp(z)
    return p / p.sum()


@pytest.mark.parametrize("V", [1, 5, 15, 16, 17, 255, 4096, 32000, 152064])
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_canonical_softmax_matches_fp64(V, T):
    l = synth.target_logits(90 + V, 1, 0, V, 3.0)[0, 0]
    p = O.softmax_canonical(l, T)
    ref = softmax64(l, T)
    big = ref > 1e-30
    assert np.all(np.abs(p[big] - ref[big]) <= ref[big] * 2e-6)
    assert abs(p.astype(np.float64).sum() - 1.0) < 1e-5


def test_canonical_softmax_underflow_is_exact_zero():
    l = np.array([0.0, -1000.0, 3.0, -500.0], np.float32)
    p = O.softmax_canonical(l)
    assert p[1] == 0 and p[3] == 0 and p[0] > 0 and p[2] > p[0]


def test_tree_sample_is_inverse_cdf_away_from_boundaries():
    g = synth.rng(91)
    for V in (1, 7, 16, 33, 1000, 4096, 5000, 20000):
        w = g.random(V).astype(np.float32) * (g.random(V) < 0.7)
        if w.sum() == 0:
            w[0] = 1
        us = g.random(150).astype(np.float32)
        cdf = np.cumsum(w.astype(np.float64))       # textbook inverse CDF, index order
        tot = cdf[-1]
        for u in us:
            got = O.tree_sample(w, float(u))
            t = float(u) * tot
            if np.min(np.abs(cdf - t)) < 1e-5 * tot:
                continue
            want = int(np.searchsorted(cdf, t, side="right"))
            assert got == want, (V, u)
            assert w[got] > 0


def test_tree_sample_distribution_chi_square():
    g = synth.rng(92)
    V = 40000                                      # three blocks, the last one partial
    w = np.zeros(V, np.float32)
    hot = g.choice(V, 12, replace=False)
    w[hot] = g.random(12).astype(np.float32) + 0.2
    us = ((np.arange(12000) + 0.5) / 12000).astype(np.float32)
    got = np.array([O.tree_sample(w, float(u)) for u in us])
    assert np.all(np.isin(got, hot))
    obs = np.array([(got == h).sum() for h in hot])
    wh = w[hot].astype(np.float64)
    exp = wh / wh.sum() * us.size
    assert stats.chisquare(obs, exp).pvalue > 1e-3


def test_tree_sample_zero_total_and_extreme_u():
    assert O.tree_sample(np.zeros(20, np.float32), 0.5) == -1
    w = np.zeros(40, np.float32)
    w[[3, 37]] = [1.0, 2.0]
    # entry 3 sits in leaf 0, entry 37 in leaf 2: the first and the last positive weight
    assert O.tree_sample(w, 0.0) == 3
    assert O.tree_sample(w, float(np.float32(1 - 2**-24))) == 37


# ------------------------------------------------------------------ the round
def fixed_position_round(rows, k, p_logits, q_logits, seed, T=1.0, round_=0):
    """rows independent rounds where every row has the same per-position logits."""
    V = p_logits.shape[-1]
    tl = np.broadcast_to(p_logits, (rows, k + 1, V)).copy()
    dl = np.broadcast_to(q_logits, (rows, k, V)).copy()
    d = synth.draft_tokens_sampled(q_logits[None].repeat(rows, 0), seed, T)
    seeds = synth.rng(seed + 1).integers(0, 2**63, size=rows, dtype=np.uint64)
    return d, O.accept_sample(d, dl, tl, T, seeds, round_)


@pytest.mark.parametrize("V,k,seed", [(5, 4, 100), (8, 3, 101)])
def test_chi_square_emitted_tokens_follow_target(V, k, seed):
    g = synth.rng(seed)
    p_logits = (g.standard_normal((k + 1, V)) * 1.0).astype(np.float32)
    q_logits = (p_logits[:k] + g.standard_normal((k, V)) * 1.2).astype(np.float32)
    rows = 120_000
    _, (out, cnt) = fixed_position_round(rows, k, p_logits, q_logits, seed)
    assert np.all((cnt >= 1) & (cnt <= k + 1))
    for i in range(k + 1):
        emitted = out[cnt > i, i]
        obs = np.bincount(emitted, minlength=V)
        exp = softmax64(p_logits[i]) * emitted.size
        assert exp.min() > 5
        pval = stats.chisquare(obs, exp).pvalue
        assert pval > 1e-3 / (k + 1), (i, pval, obs, exp)


@pytest.mark.parametrize("alpha", [0.6, 0.95])
@pytest.mark.parametrize("k", [2, 4, 6, 8])
def test_eq1_expected_tokens_per_round(alpha, k):
    """Eq. (1): with q = (1, 0) and p = (alpha, 1 - alpha) every position is
    accepted independently with probability alpha."""
    rows = 100_000
    p_logits = np.tile(np.log(np.array([alpha, 1 - alpha])).astype(np.float32), (k + 1, 1))
    q_logits = np.tile(np.array([0.0, -1000.0], np.float32), (k, 1))
    d, (out, cnt) = fixed_position_round(rows, k, p_logits, q_logits, 200 + k)
    assert np.all(d == 0)
    E = (1 - alpha ** (k + 1)) / (1 - alpha)
    se = cnt.std() / np.sqrt(rows)
    assert abs(cnt.mean() - E) < 4 * se, (cnt.mean(), E, se)


def test_acceptance_probability_is_sum_of_min():
    V, k = 6, 2
    g = synth.rng(300)
    p_logits = g.standard_normal((k + 1, V)).astype(np.float32)
    q_logits = (p_logits[:k] + g.standard_normal((k, V)) * 1.5).astype(np.float32)
    rows = 100_000
    _, (out, cnt) = fixed_position_round(rows, k, p_logits, q_logits, 301)
    beta = np.minimum(softmax64(p_logits[0]), softmax64(q_logits[0])).sum()
    acc = (cnt > 1).mean()
    assert abs(acc - beta) < 4 * np.sqrt(beta * (1 - beta) / rows)


def test_identical_models_always_accept():
    V, k = 50, 5
    l = synth.target_logits(310, 1, k, V, 2.0)[0]
    _, (out, cnt) = fixed_position_round(2000, k, l, l[:k], 311)
    assert np.all(cnt == k + 1)


def test_disjoint_supports_always_reject_first():
    k = 3
    p_logits = np.tile(np.array([0.0, 0.0, -1000.0, -1000.0], np.float32), (k + 1, 1))
    q_logits = np.tile(np.array([-1000.0, -1000.0, 0.0, 0.0], np.float32), (k, 1))
    d, (out, cnt) = fixed_position_round(20_000, k, p_logits, q_logits, 320)
    assert np.all(np.isin(d, [2, 3]))
    assert np.all(cnt == 1) and np.all(np.isin(out[:, 0], [0, 1]))
    assert abs((out[:, 0] == 0).mean() - 0.5) < 0.02


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_canonical_round_agrees_with_fp64_round(T):
    """Config-1-shaped round (V = 4096, target ~ N(0, 2), draft = target +
    N(0, 0.5)); the canonical fp32 recipe must take the same decisions as
    plain fp64 arithmetic except at near-ties."""
    B, k, V = 256, 4, 4096
    tl = synth.target_logits(400, B, k, V, 2.0)
    dl = synth.draft_logits_from(tl, 401, 0.5)
    d = synth.draft_tokens_sampled(dl, 402, T)
    seeds = synth.seeds_for(1, B)
    out, cnt = O.accept_sample(d, dl, tl, T, seeds, 3)
    out64, cnt64, margin = O.accept_sample_f64(d, dl, tl, T, seeds, 3)
    differ = np.any(out != out64, axis=1) | (cnt != cnt64)
    assert np.all(margin[differ] < 1e-5)
    assert differ.sum() <= 1
    assert 1.5 < cnt.mean() < k + 1


def test_invalid_inputs_rejected():
    B, k, V = 2, 2, 10
    tl = synth.target_logits(410, B, k, V, 1.0)
    dl = synth.draft_logits_from(tl, 411, 0.5)
    d = np.zeros((B, k), np.int32)
    seeds = synth.seeds_for(0, B)
    with pytest.raises(ValueError):
        O.accept_sample(d, dl, tl, 0.0, seeds, 0)
    d[1, 1] = V
    with pytest.raises(ValueError):
        O.accept_sample(d, dl, tl, 1.0, seeds, 0)
    d[1, 1] = 0
    tl[0, 2, 3] = np.nan
    with pytest.raises(ValueError):
        O.accept_sample(d, dl, tl, 1.0, seeds, 0)


@pytest.mark.parametrize("k,noise", [(4, 1.05), (8, 0.132)])
def test_canonical_round_agrees_with_fp64_round_sweep_shape(k, noise):
    """Acceptance-sweep shape (V = 152064, target ~ N(0, 3), draft noise at the
    two calibrated levels): the canonical recipe and the textbook fp64 round
    (index-order inverse CDF) emit the same ids and counts on every row whose
    decisions are not near-ties."""
    B, V = 12, 152064
    tl = synth.target_logits(430 + k, B, k, V, 3.0)
    dl = synth.draft_logits_from(tl, 431 + k, noise)
    d = synth.draft_tokens_sampled(dl, 432 + k)
    seeds = synth.seeds_for(2, B)
    for rnd in (0, 7):
        out, cnt = O.accept_sample(d, dl, tl, 1.0, seeds, rnd)
        out64, cnt64, margin = O.accept_sample_f64(d, dl, tl, 1.0, seeds, rnd)
        differ = np.any(out != out64, axis=1) | (cnt != cnt64)
        assert np.all(margin[differ] < 1e-5)
        assert differ.sum() == 0


@pytest.mark.parametrize("V", [1, 5, 1023, 1024, 1025, 4096, 40000, 152064])
def test_sample_p_is_inverse_cdf_of_softmax(V):
    """The bonus draw's two-level rule (segment weights from the (max, sum)
    pass, then the chosen segment's leaves) picks the textbook fp64 inverse
    CDF of softmax(l / T) over the vocabulary in index order, except where
    u * total lies within fp32 rounding (1e-6 of the total) of a boundary."""
    g = synth.rng(700 + V)
    l = (g.standard_normal(V) * 3.0).astype(np.float32)
    for T in (1.0, 0.7):
        cdf = np.cumsum(softmax64(l, T))
        us = g.random(60).astype(np.float32)
        checked = 0
        for u in us:
            got = O.sample_p(l, T, float(u))
            t = float(u) * cdf[-1]
            if np.min(np.abs(cdf - t)) < 1e-6:
                continue
            assert got == int(np.searchsorted(cdf, t, side="right")), (V, T, u)
            checked += 1
        assert checked >= 50


def test_sample_p_extremes_and_underflow():
    l = np.array([0.0, -1000.0, 3.0, -500.0, 3.0], np.float32)
    assert O.sample_p(l, 1.0, 0.0) == 0                       # u = 0: the first entry with p > 0
    assert O.sample_p(l, 1.0, float(np.float32(1 - 2**-24))) == 4   # the last entry with p > 0
    draws = {O.sample_p(l, 1.0, float(u)) for u in np.linspace(0, 0.999, 400, dtype=np.float32)}
    assert draws <= {0, 2, 4}                                  # underflowed entries are never drawn
