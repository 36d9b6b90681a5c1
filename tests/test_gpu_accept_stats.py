"""Sampled acceptance on the GPU against what the mathematics fixes, with no
structure shared with the kernels.

"How Speculative Decoding Speeds Up Inference", "The same output as the large
model alone": speculative sampling (Leviathan et al.; Chen et al.) accepts
each draft token with probability min(1, p/q), resamples from the normalised
residual after a rejection, and so emits tokens that follow the target
distribution; Eq. (1) gives the expected tokens per pass when every position
is accepted independently with probability alpha.  The per-position
acceptance probability is sum_x min(p, q) (Leviathan et al.).

The first test compares the kernels' ids and counts with the oracle's plain
fp64 round (libm exp, serial sums, the textbook inverse CDF over the
vocabulary in index order) at the acceptance-sweep shape; the others are
distributional: chi-square of emitted tokens against softmax(p), Eq. (1), and
the acceptance probability.
"""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle as O
from quantized_self_speculative_gb300 import synth

pytestmark = pytest.mark.gpu


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def seeds_dev(s):
    return torch.from_numpy(np.ascontiguousarray(s).view(np.int64)).cuda()


def softmax64(l):
    z = l.astype(np.float64)
    z = z - z.max()
    p = np.exp(z)
    return p / p.sum()


@pytest.mark.parametrize("k,noise", [(4, 1.05), (8, 0.132), (2, 1.05)])
def test_gpu_matches_fp64_textbook_round(nq, k, noise):
    """Acceptance-sweep shape: B = 64, V = 152064, target ~ N(0, 3), draft =
    target + N(0, noise) at the noise levels that give alpha ~ 0.6 and ~ 0.95.
    Every row must get the same count and ids as the fp64 round unless one of
    its uniforms lies within fp32 rounding of a decision boundary: the fp32
    recipe's probabilities and tree sums carry a relative error of a few
    units of 2^-24 (about 1e-6 of the total at most), so a row may differ
    only where the fp64 margin is below 1e-6."""
    B, V = 64, 152064
    tl = synth.target_logits(9100 + k, B, k, V, 3.0)
    dl = synth.draft_logits_from(tl, 9101 + k, noise)
    d = synth.draft_tokens_sampled(dl, 9102 + k)
    seeds = synth.seeds_for(11, B)
    near, total = 0, 0
    for rnd in (0, 1, 2):
        out, cnt = nq.accept_sample(dev(d), dev(dl), dev(tl), 1.0, seeds_dev(seeds), rnd)
        out, cnt = out.cpu().numpy(), cnt.cpu().numpy()
        out64, cnt64, margin = O.accept_sample_f64(d, dl, tl, 1.0, seeds, rnd)
        differ = np.any(out != out64, axis=1) | (cnt != cnt64)
        assert np.all(margin[differ] < 1e-6), (rnd, np.nonzero(differ), margin[differ])
        near += int((margin < 1e-6).sum())
        total += int(differ.sum())
    assert nq.device_status() == 0
    assert total <= near, (total, near)


def gpu_rounds(nq, p_logits, q_logits, rows, seed, calls=2, T=1.0):
    """`rows` rounds per call, every row with the same per-position logits;
    draft tokens drawn from softmax(q) in fp64 (the draft model's behaviour)."""
    k, V = q_logits.shape
    tl = dev(np.broadcast_to(p_logits, (rows, k + 1, V)).copy())
    dl = dev(np.broadcast_to(q_logits, (rows, k, V)).copy())
    seeds = seeds_dev(synth.rng(seed).integers(0, 2**63, size=rows, dtype=np.uint64))
    outs, cnts = [], []
    for c in range(calls):
        d = synth.draft_tokens_sampled(np.broadcast_to(q_logits, (rows, k, V)), seed + 1 + c, T)
        out, cnt = nq.accept_sample(dev(d), dl, tl, T, seeds, 1000 + c)
        outs.append(out.cpu().numpy())
        cnts.append(cnt.cpu().numpy())
    assert nq.device_status() == 0
    return np.concatenate(outs), np.concatenate(cnts)


@pytest.mark.parametrize("V,k,seed", [(5, 4, 9200), (8, 3, 9201)])
def test_gpu_chi_square_emitted_tokens_follow_target(nq, V, k, seed):
    g = synth.rng(seed)
    p_logits = g.standard_normal((k + 1, V)).astype(np.float32)
    q_logits = (p_logits[:k] + g.standard_normal((k, V)) * 1.2).astype(np.float32)
    out, cnt = gpu_rounds(nq, p_logits, q_logits, 60_000, seed)
    assert cnt.size >= 100_000
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
def test_gpu_eq1_expected_tokens_per_round(nq, alpha, k):
    """V = 2, q = (1, 0), p = (alpha, 1 - alpha): each position is accepted
    independently with probability alpha, so the mean count per round is
    (1 - alpha^(k+1)) / (1 - alpha)."""
    p_logits = np.tile(np.log(np.array([alpha, 1 - alpha])).astype(np.float32), (k + 1, 1))
    q_logits = np.tile(np.array([0.0, -1000.0], np.float32), (k, 1))
    out, cnt = gpu_rounds(nq, p_logits, q_logits, 50_000, 9300 + k)
    E = (1 - alpha ** (k + 1)) / (1 - alpha)
    se = cnt.std() / np.sqrt(cnt.size)
    assert abs(cnt.mean() - E) < 4 * se, (cnt.mean(), E, se)
    # a rejected position is replaced by token 1, the only one with p > q
    rej = cnt <= k
    assert np.all(out[rej, cnt[rej] - 1] == 1)


def test_gpu_acceptance_probability_is_sum_of_min(nq):
    V, k = 6, 2
    g = synth.rng(9400)
    p_logits = g.standard_normal((k + 1, V)).astype(np.float32)
    q_logits = (p_logits[:k] + g.standard_normal((k, V)) * 1.5).astype(np.float32)
    out, cnt = gpu_rounds(nq, p_logits, q_logits, 50_000, 9401)
    beta = np.minimum(softmax64(p_logits[0]), softmax64(q_logits[0])).sum()
    acc = (cnt > 1).mean()
    assert abs(acc - beta) < 4 * np.sqrt(beta * (1 - beta) / cnt.size)


@pytest.mark.parametrize("B,k,V,T", [(64, 4, 152064, 1.0), (5, 8, 32000, 0.7), (3, 2, 4099, 1.3)])
def test_gpu_draft_features_match_fp64(nq, B, k, V, T):
    """SpecKV's step features from the acceptance pass (mean / max draft
    entropy, mean / min draft confidence) against the oracle's fp64
    definition; the token outputs equal spec_accept_sample's bit for bit."""
    tl = synth.target_logits(9500 + V, B, k, V, 3.0)
    dl = synth.draft_logits_from(tl, 9501 + V, 0.5)
    d = synth.draft_tokens_sampled(dl, 9502 + V, T)
    seeds = synth.seeds_for(12, B)
    out, cnt, feat = nq.accept_sample_features(dev(d), dev(dl), dev(tl), T, seeds_dev(seeds), 4)
    out2, cnt2 = nq.accept_sample(dev(d), dev(dl), dev(tl), T, seeds_dev(seeds), 4)
    assert torch.equal(out, out2) and torch.equal(cnt, cnt2)
    ref = O.draft_features(d, dl, T)
    got = feat.cpu().numpy().astype(np.float64)
    assert np.allclose(got, ref, rtol=2e-5, atol=1e-6), np.abs(got - ref).max()
    assert nq.device_status() == 0
