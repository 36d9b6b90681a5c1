"""Pins for the oracle's round bookkeeping.

"How Speculative Decoding Speeds Up Inference", "Drafting and checking
tokens": the draft proposes k tokens one at a time, the target checks the
k+1 positions in one pass, the kept prefix plus the target's replacement
extend the sequence and that last token starts the next round; Table 1 (the
k = 4 worked round adds three tokens).  BitNest, Fig. 4: the cache entries of
the rejected suffix are dropped, so the cache keeps one entry per committed
token but the last.
"""
import numpy as np

import oracle as O
from quantized_self_speculative_gb300 import synth
from test_oracle_greedy import load_worked_round, one_hot_logits


def test_draft_argmax_is_lowest_index_argmax():
    g = synth.rng(500)
    l = g.standard_normal((40, 333)).astype(np.float32)
    l[3, [5, 200]] = 50.0                    # a tie: the lower index wins
    l[7, :] = 1.0                            # all equal: index 0
    tok = O.draft_argmax(l)
    assert tok[3] == 5 and tok[7] == 0
    for m in range(40):
        assert tok[m] == min(np.flatnonzero(l[m] == l[m].max()))


def test_commit_worked_round_table1():
    """Table 1's round after a two-token prefix: A and B kept, E replaces the
    third draft; three tokens are appended and E starts the next round."""
    rows, (n_added, words) = load_worked_round()
    vocab = sorted({w for r in rows for w in r[1:3] if w != "-"})
    V = len(vocab) + 3
    ids = {w: i for i, w in enumerate(vocab)}
    draft = np.array([[ids[r[1]] for r in rows]], np.int32)
    known = [ids[r[2]] for r in rows if r[2] != "-"]
    out, cnt = O.accept_greedy(draft, one_hot_logits(known + [0, 0], V)[None])
    seq = np.full((1, 16), -9, np.int32)
    seq[0, :2] = [V - 1, V - 2]
    seq2, len2, x0, rc = O.round_commit(out, cnt, seq, np.array([2], np.int32), np.array([V - 2], np.int32))
    assert rc == 0 and len2[0] == 2 + n_added == 5
    assert [vocab[i] for i in seq2[0, 2:5]] == words
    assert x0[0] == ids[words[-1]]
    assert np.all(seq2[0, 5:] == -9) and list(seq2[0, :2]) == [V - 1, V - 2]
    # the cache keeps the first cnt of the k+1 verified positions: length
    # (seq_len - 1) grows by cnt, the rejected suffix (k + 1 - cnt entries) goes
    k = draft.shape[1]
    assert (len2[0] - 1) - (2 - 1) == cnt[0] and k + 1 - cnt[0] == 2


def test_commit_lengths_truncation_and_bad_counts():
    g = synth.rng(501)
    B, k, L = 50, 6, 20
    cnt = g.integers(1, k + 2, size=B).astype(np.int32)
    out = np.full((B, k + 1), -1, np.int32)
    for b in range(B):
        out[b, :cnt[b]] = g.integers(0, 1000, size=cnt[b])
    seq_len = g.integers(0, L + 1, size=B).astype(np.int32)
    seq = np.full((B, L), 7, np.int32)
    seq2, len2, x0, rc = O.round_commit(out, cnt, seq, seq_len, np.zeros(B, np.int32))
    full = seq_len + cnt > L
    assert rc == (1 if full.any() else 0)
    for b in range(B):
        n = min(cnt[b], L - seq_len[b])
        assert len2[b] == seq_len[b] + n
        assert np.array_equal(seq2[b, seq_len[b]:seq_len[b] + n], out[b, :n])
        assert np.all(seq2[b, :seq_len[b]] == 7) and np.all(seq2[b, seq_len[b] + n:] == 7)
        assert x0[b] == out[b, cnt[b] - 1]
    bad = cnt.copy()
    bad[3] = 0
    bad[4] = k + 2
    seq3, len3, x03, rc3 = O.round_commit(out, bad, seq, seq_len, np.full(B, -5, np.int32))
    assert rc3 == -1 and len3[3] == seq_len[3] and len3[4] == seq_len[4] and x03[3] == -5 and x03[4] == -5


def test_rounds_through_the_bookkeeping_equal_target_greedy():
    """Brute force on a toy bigram model: rounds driven only by draft_argmax,
    embed_round, the linears, accept_greedy and round_commit emit the target's
    own greedy sequence."""
    V, d, g, k = 96, 64, 64, 3
    E = synth.f32_to_bf16_bits(synth.weights(502, V, d, std=1.0))
    base, resid, scales = O.pack_nested(synth.weights(503, V, d, std=0.5), g)
    lin = lambda x, verify: O.linear(O.FMT_NESTED44, V, d, g, base, resid, scales, x, verify).astype(np.float32)
    B, max_len, rounds = 3, 64, 12
    starts = np.array([4, 50, 77], np.int32)
    seq = np.full((B, max_len), -1, np.int32)
    seq[:, 0] = starts
    seq_len = np.ones(B, np.int32)
    x0 = starts.copy()
    for _ in range(rounds):
        draft = np.zeros((B, k), np.int32)
        cur = x0
        for j in range(k):
            cur = O.draft_argmax(lin(O.embed_rows(E, cur), False))
            draft[:, j] = cur
        tl = lin(O.embed_round(E, x0, draft), True).reshape(B, k + 1, V)
        out, cnt = O.accept_greedy(draft, tl)
        seq, seq_len, x0, rc = O.round_commit(out, cnt, seq, seq_len, x0)
        assert rc == 0
    for b in range(B):
        ref = [int(starts[b])]
        while len(ref) < seq_len[b]:
            ref.append(int(O.draft_argmax(lin(O.embed_rows(E, [ref[-1]]), True))[0]))
        assert list(seq[b, :seq_len[b]]) == ref
    assert seq_len.sum() > B * (rounds + 1)          # some drafts survived
