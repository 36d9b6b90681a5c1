"""Pins for the oracle's greedy acceptance (C3).

"How Speculative Decoding Speeds Up Inference": the round (draft k tokens,
check all k positions in one target pass, keep the matching prefix, replace
the first mismatch by the target's choice, 1..k+1 tokens per pass), Table 1
(k = 4 worked round) and the greedy equivalence ("every kept token is the
target model's own top choice").
"""
import itertools
import os

import numpy as np
import pytest

import oracle as O
from conftest import GOLDEN
from quantized_self_speculative_gb300 import synth


def load_worked_round():
    rows, added = [], None
    for line in open(os.path.join(GOLDEN, "erge_table1_k4.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        f = line.split()
        if f[0] == "added":
            added = (int(f[1]), f[2:])
        else:
            rows.append((int(f[0]), f[1], f[2], f[3]))
    return rows, added


def one_hot_logits(choices, V, rest=0.0, peak=5.0):
    l = np.full((len(choices), V), rest, np.float32)
    for j, c in enumerate(choices):
        l[j, c] = peak
    return l


def test_worked_round_table1():
    rows, (n_added, added_words) = load_worked_round()
    vocab = sorted({w for r in rows for w in r[1:3] if w != "-"})
    V = len(vocab) + 3
    ids = {w: i for i, w in enumerate(vocab)}
    draft = np.array([[ids[r[1]] for r in rows]], np.int32)
    k = draft.shape[1]
    known = [ids[r[2]] for r in rows if r[2] != "-"]
    results = set()
    # the page leaves the target's choice at position 4 blank and does not show
    # the choice after the last draft token: sweep every value of both
    for t4, t5 in itertools.product(range(V), range(V)):
        tl = one_hot_logits(known + [t4, t5], V)[None]
        out, cnt = O.accept_greedy(draft, tl)
        results.add((tuple(out[0]), int(cnt[0])))
    assert len(results) == 1
    (out, cnt), = results
    assert cnt == n_added == 3
    assert [vocab[i] for i in out[:cnt]] == added_words
    assert list(out[cnt:]) == [-1] * (k + 1 - cnt)
    # per-row results: accepted, accepted, replaced, discarded
    assert [r[3] for r in rows] == ["accepted", "accepted", "replaced", "discarded"]


@pytest.mark.parametrize("k", [1, 4, 8])
def test_all_accepted_and_first_mismatch(k):
    V = 11
    g = synth.rng(50 + k)
    t = g.integers(0, V, size=k + 1)
    tl = one_hot_logits(list(t), V)[None]
    out, cnt = O.accept_greedy(t[None, :k].astype(np.int32), tl)
    assert cnt[0] == k + 1 and list(out[0]) == list(t)             # bonus token t_k
    d = t[:k].copy()
    d[0] = (d[0] + 1) % V
    out, cnt = O.accept_greedy(d[None].astype(np.int32), tl)
    assert cnt[0] == 1 and out[0, 0] == t[0] and np.all(out[0, 1:] == -1)


def test_ties_take_lowest_index_and_nonfinite_rejected():
    V = 9
    tl = np.zeros((1, 2, V), np.float32)
    tl[0, 0, [3, 7]] = 2.0
    tl[0, 1, :] = 1.0
    out, cnt = O.accept_greedy(np.array([[3]], np.int32), tl)
    assert list(out[0]) == [3, 0] and cnt[0] == 2
    tl[0, 1, 4] = np.inf
    with pytest.raises(ValueError):
        O.accept_greedy(np.array([[3]], np.int32), tl)


def test_counts_are_within_1_to_k_plus_1_on_random_rounds():
    B, k, V = 64, 6, 300
    tl = synth.target_logits(60, B, k, V, 2.0)
    dl = synth.draft_logits_from(tl, 61, 1.0)
    d = synth.draft_tokens_greedy(dl)
    out, cnt = O.accept_greedy(d, tl)
    assert np.all((cnt >= 1) & (cnt <= k + 1))
    for b in range(B):
        c = cnt[b]
        assert np.array_equal(out[b, :c - 1], d[b, :c - 1])
        assert out[b, c - 1] == np.argmax(tl[b, c - 1])
        assert np.all(out[b, c:] == -1)


def test_speculative_greedy_equals_target_only_greedy():
    """Brute force on a toy bigram LM: the draft uses the base plane only, the
    target both planes; speculative rounds must emit exactly the target's own
    greedy sequence."""
    V, d, g = 128, 64, 64
    E = synth.weights(70, V, d, std=1.0)          # token embeddings -> activations
    Wlm = synth.weights(71, V, d, std=0.5)         # lm head
    base, resid, scales = O.pack_nested(Wlm, g)
    emb = synth.f32_to_bf16_bits(E)

    def logits(tokens, verify):
        y = O.linear(O.FMT_NESTED44, V, d, g, base, resid, scales, emb[np.asarray(tokens)], verify)
        return y.astype(np.float32)

    start, n_tokens, k = 5, 40, 4
    ref = [start]
    while len(ref) < n_tokens + 1:
        ref.append(int(np.argmax(logits([ref[-1]], True)[0])))
    seq = [start]
    rounds = 0
    while len(seq) < n_tokens + 1:
        draft = []
        cur = seq[-1]
        for _ in range(k):
            cur = int(np.argmax(logits([cur], False)[0]))
            draft.append(cur)
        tl = logits([seq[-1]] + draft, True)[None]          # k+1 positions in one pass
        out, cnt = O.accept_greedy(np.array([draft], np.int32), tl)
        seq.extend(int(t) for t in out[0, :cnt[0]])
        rounds += 1
    assert seq[:n_tokens + 1] == ref
    assert rounds < n_tokens                                   # speculation saved passes
