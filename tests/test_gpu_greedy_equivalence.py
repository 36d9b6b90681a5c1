"""Greedy speculative decoding through the GPU kernels emits exactly the
target's own greedy sequence, by brute force on a toy language model.

"How Speculative Decoding Speeds Up Inference", "The same output as the large
model alone": with greedy decoding, the drafted tokens that survive the check
are the ones the target would have picked itself, and the token that replaces
the first mismatch is the target's own choice, so the output equals plain
target-only greedy decoding whatever the draft proposes.  "Drafting and
checking tokens": the draft proposes k tokens one at a time, the target checks
all of them in one pass over k+1 positions.

Toy model: vocabulary V = 4096, width d = 1024.  The input row of a position
is bf16(E[token] + P[position mod 97]) (E, P ~ N(0, 1)); the logits are that
row times a nested 4+4-bit matrix W [V][d] (N(0, 0.02) weights, group 128,
packed by the oracle).  The draft reads W's base plane (nq_draft_gemv, one
position per call); the target reads both planes (nq_verify_gemm over the k+1
positions of a round); spec_accept_greedy keeps the matching prefix.  The
property rests on the verify kernel being batch-invariant: row m of a call
over M rows is bit-identical to a call over that row alone, so the target's
logits for a position do not depend on how many positions share the pass.
The target-only sequence is also compared with the oracle's fp64 greedy
decoding over its first tokens.
"""
import numpy as np
import pytest
import torch

import oracle as O
from quantized_self_speculative_gb300 import synth

from gpu_helpers import oracle_packed

pytestmark = pytest.mark.gpu

V, D, G, NPOS = 4096, 1024, 128, 97


class ToyLM:
    def __init__(self, nq):
        self.nq = nq
        w = synth.weights(8100, V, D)
        self.pl, (self.base, self.resid, self.scales) = oracle_packed(nq, w, nq.FMT_NESTED44, G)
        self.E = torch.from_numpy(synth.rng(8101).standard_normal((V, D), dtype=np.float32)).cuda()
        self.P = torch.from_numpy(synth.rng(8102).standard_normal((NPOS, D), dtype=np.float32)).cuda()

    def rows(self, tokens, positions):
        """Input rows, bf16 [len(tokens)][D]."""
        t = torch.as_tensor(np.asarray(tokens, dtype=np.int64), device="cuda")
        p = torch.as_tensor(np.asarray(positions, dtype=np.int64) % NPOS, device="cuda")
        return (self.E[t] + self.P[p]).to(torch.bfloat16).contiguous()

    def rows_host(self, tokens, positions):
        return self.rows(tokens, positions).view(torch.int16).cpu().numpy().view(np.uint16)


def target_only(lm, start, pos0, n):
    """Plain greedy decoding with the target: one position per verify call (M = 1)."""
    seq = [start]
    for i in range(n):
        y = lm.nq.verify_gemm(lm.pl, lm.rows([seq[-1]], [pos0 + i]))
        seq.append(int(torch.argmax(y[0]).item()))
    return seq


def speculative(lm, starts, k, rounds):
    """B sequences decoded together: per round, k draft calls over the B
    current positions (M = B), one verify call over the B (k+1) positions,
    one greedy acceptance call; the emitted tokens are appended."""
    nq = lm.nq
    B = len(starts)
    seqs = [[s] for s in starts]
    passes = 0
    for _ in range(rounds):
        cur = [s[-1] for s in seqs]
        pos = [len(s) - 1 for s in seqs]
        draft = [[] for _ in range(B)]
        for j in range(k):
            y = nq.draft_gemv(lm.pl, lm.rows(cur, [p + j for p in pos]))
            nxt = torch.argmax(y, dim=1).cpu().numpy()
            for b in range(B):
                draft[b].append(int(nxt[b]))
            cur = [int(t) for t in nxt]
        toks, poss = [], []
        for b in range(B):
            toks += [seqs[b][-1]] + draft[b]
            poss += [pos[b] + j for j in range(k + 1)]
        tl = nq.verify_gemm(lm.pl, lm.rows(toks, poss)).view(B, k + 1, V)
        out, cnt = nq.accept_greedy(torch.tensor(draft, dtype=torch.int32, device="cuda"), tl)
        out, cnt = out.cpu().numpy(), cnt.cpu().numpy()
        for b in range(B):
            assert 1 <= cnt[b] <= k + 1
            assert np.all(out[b, cnt[b]:] == -1)
            seqs[b].extend(int(t) for t in out[b, :cnt[b]])
        passes += 1
    return seqs, passes


@pytest.fixture(scope="module")
def lm(nq):
    return ToyLM(nq)


@pytest.mark.parametrize("B,k,rounds", [(1, 4, 256), (4, 4, 64), (2, 8, 64)])
def test_speculative_greedy_equals_target_only_greedy(lm, B, k, rounds):
    starts = [int(s) for s in synth.rng(8200 + B).integers(0, V, size=B)]
    seqs, passes = speculative(lm, starts, k, rounds)
    emitted = sum(len(s) - 1 for s in seqs)
    assert passes == rounds and emitted >= B * rounds
    for b in range(B):
        ref = target_only(lm, starts[b], 0, len(seqs[b]) - 1)
        assert seqs[b] == ref, f"sequence {b} departs from target-only greedy at {next(i for i, (a, c) in enumerate(zip(seqs[b], ref)) if a != c)}"
    # the draft is a 4-bit copy of the target: some drafted tokens survive
    assert emitted > B * rounds


def test_target_only_greedy_matches_oracle(lm):
    """The GPU target-only sequence equals the oracle's fp64 greedy decoding
    (same packed planes, same bf16 rows) wherever the oracle's top-two logit
    margin exceeds the linears' 2e-3 normwise tolerance times max |logit|."""
    start, n = 1234, 48
    gpu = target_only(lm, start, 0, n)
    seq = [start]
    compared = 0
    for i in range(n):
        x = lm.rows_host([seq[-1]], [i])
        y = O.linear(O.FMT_NESTED44, V, D, G, lm.base, lm.resid, lm.scales, x, True)[0]
        top2 = np.sort(y)[-2:]
        if top2[1] - top2[0] <= 2e-3 * np.abs(y).max():
            break   # a near-tie: the fp32 kernel may legitimately pick the other token
        seq.append(int(np.argmax(y)))
        compared += 1
    assert compared >= 40
    assert gpu[:len(seq)] == seq
