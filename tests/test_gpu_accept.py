"""GPU acceptance (K6 greedy, K7 sampled) vs the CPU oracle: bit-exact token
ids and counts on the same seeded inputs and Philox seeds."""
import numpy as np
import pytest
import torch

import oracle as O
from quantized_self_speculative_gb300 import synth
from test_oracle_greedy import load_worked_round, one_hot_logits

pytestmark = pytest.mark.gpu


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def seeds_dev(s):
    return torch.from_numpy(np.ascontiguousarray(s).view(np.int64)).cuda()


def greedy_case(B, k, V, seed, tstd=2.0, dstd=0.5):
    tl = synth.target_logits(seed, B, k, V, tstd)
    dl = synth.draft_logits_from(tl, seed + 1, dstd)
    return synth.draft_tokens_greedy(dl), tl


def sample_case(B, k, V, seed, T=1.0, tstd=2.0, dstd=0.5):
    tl = synth.target_logits(seed, B, k, V, tstd)
    dl = synth.draft_logits_from(tl, seed + 1, dstd)
    return synth.draft_tokens_sampled(dl, seed + 2, T), dl, tl


def check_greedy(nq, d, tl):
    out, cnt = nq.accept_greedy(dev(d), dev(tl))
    ref_out, ref_cnt = O.accept_greedy(d, tl)
    assert np.array_equal(cnt.cpu().numpy(), ref_cnt)
    assert np.array_equal(out.cpu().numpy(), ref_out)
    assert nq.device_status() == 0
    return ref_cnt


def check_sample(nq, d, dl, tl, T, seeds, rnd):
    out, cnt = nq.accept_sample(dev(d), dev(dl), dev(tl), T, seeds_dev(seeds), rnd)
    ref_out, ref_cnt = O.accept_sample(d, dl, tl, T, seeds, rnd)
    assert np.array_equal(cnt.cpu().numpy(), ref_cnt)
    assert np.array_equal(out.cpu().numpy(), ref_out)
    assert nq.device_status() == 0
    return ref_cnt


def test_greedy_worked_round_table1(nq):
    rows, (n_added, words) = load_worked_round()
    vocab = sorted({w for r in rows for w in r[1:3] if w != "-"})
    V = len(vocab) + 3
    ids = {w: i for i, w in enumerate(vocab)}
    d = np.array([[ids[r[1]] for r in rows]], np.int32)
    known = [ids[r[2]] for r in rows if r[2] != "-"]
    blanks = [(a, b) for a in range(V) for b in range(V)]
    tl = np.stack([one_hot_logits(known + [a, b], V) for a, b in blanks])
    out, cnt = nq.accept_greedy(dev(np.repeat(d, len(blanks), 0)), dev(tl))
    out, cnt = out.cpu().numpy(), cnt.cpu().numpy()
    assert np.all(cnt == n_added)
    assert all([vocab[i] for i in row[:n_added]] == words for row in out)
    assert np.all(out[:, n_added:] == -1)


@pytest.mark.parametrize("B,k,V", [(256, 4, 4096), (1, 4, 4096), (64, 2, 152064), (64, 8, 152064),
                                   (3, 16, 4099), (7, 1, 5), (5, 3, 1), (9, 5, 32000), (2, 6, 20000)])
def test_greedy_parity(nq, B, k, V):
    d, tl = greedy_case(B, k, V, 7000 + B + k + V)
    cnt = check_greedy(nq, d, tl)
    assert np.all((cnt >= 1) & (cnt <= k + 1))


def test_greedy_ties_and_all_accept(nq):
    B, k, V = 4, 3, 8200
    tl = np.zeros((B, k + 1, V), np.float32)
    tl[:, :, [17, 4100, 8199]] = 1.0                 # three-way tie spread over chunks -> lowest index
    d = np.full((B, k), 17, np.int32)
    d[1, 2] = 4100
    cnt = check_greedy(nq, d, tl)
    assert list(cnt) == [4, 3, 4, 4]


@pytest.mark.parametrize("B,k,V,T", [(256, 4, 4096, 1.0), (1, 4, 4096, 1.0), (64, 2, 152064, 1.0),
                                     (64, 8, 152064, 1.0), (16, 4, 32000, 0.7), (3, 16, 4099, 1.3),
                                     (7, 1, 5, 1.0), (5, 3, 1, 1.0), (2, 6, 20000, 1.0), (8, 4, 2048, 1.0)])
def test_sample_parity(nq, B, k, V, T):
    d, dl, tl = sample_case(B, k, V, 8000 + B + k + V, T)
    seeds = synth.seeds_for(3, B)
    for rnd in (0, 1, 2**33 + 5):
        cnt = check_sample(nq, d, dl, tl, T, seeds, rnd)
        assert np.all((cnt >= 1) & (cnt <= k + 1))


def test_sample_identical_models_and_disjoint_supports(nq):
    B, k, V = 32, 5, 3000
    tl = synth.target_logits(8100, B, k, V, 2.0)
    dl = tl[:, :k].copy()
    d = synth.draft_tokens_sampled(dl, 8101)
    cnt = check_sample(nq, d, dl, tl, 1.0, synth.seeds_for(4, B), 0)
    assert np.all(cnt == k + 1)
    tl2 = np.full((B, k + 1, V), -1000.0, np.float32)
    tl2[:, :, :100] = 0.0
    dl2 = np.full((B, k, V), -1000.0, np.float32)
    dl2[:, :, 2000:2100] = 0.0
    d2 = synth.draft_tokens_sampled(dl2, 8102)
    cnt = check_sample(nq, d2, dl2, tl2, 1.0, synth.seeds_for(5, B), 0)
    assert np.all(cnt == 1)


def test_sample_config5_alpha_sweep_small(nq):
    """Acceptance-sweep shape at reduced batch: many rounds, mean tokens per
    round consistent between GPU and oracle (bit-exact) and within 1..k+1."""
    B, k, V = 64, 4, 152064
    d, dl, tl = sample_case(B, k, V, 8200, 1.0, 3.0, 0.3)
    seeds = synth.seeds_for(6, B)
    cnt = check_sample(nq, d, dl, tl, 1.0, seeds, 11)
    assert cnt.mean() > 1.5


def test_device_status_flags(nq):
    B, k, V = 2, 3, 1000
    d, tl = greedy_case(B, k, V, 8300)
    tl[1, 2, 500] = np.nan
    nq.accept_greedy(dev(d), dev(tl))
    assert nq.device_status() & nq.NQ_DEV_NONFINITE
    assert nq.device_status() == 0                   # read-and-clear
    d[0, 1] = V + 3
    _, tl = greedy_case(B, k, V, 8301)
    nq.accept_greedy(dev(d), dev(tl))
    assert nq.device_status() & nq.NQ_DEV_BAD_TOKEN
    d2, dl2, tl2 = sample_case(B, k, V, 8302)
    dl2[0, 0, 3] = np.inf
    nq.accept_sample(dev(d2), dev(dl2), dev(tl2), 1.0, seeds_dev(synth.seeds_for(7, B)), 0)
    assert nq.device_status() & nq.NQ_DEV_NONFINITE
    # an out-of-range draft id in the sampled path: flagged, and treated as a
    # rejection at its position (the row keeps at most that many drafts)
    d3, dl3, tl3 = sample_case(B, k, V, 8303)
    d3[1, 1] = V
    tok, cnt = nq.accept_sample(dev(d3), dev(dl3), dev(tl3), 1.0, seeds_dev(synth.seeds_for(9, B)), 0)
    assert nq.device_status() & nq.NQ_DEV_BAD_TOKEN
    tok, cnt = tok.cpu().numpy(), cnt.cpu().numpy()
    assert 1 <= cnt[1] <= 2 and np.all((tok[1, :cnt[1]] >= 0) & (tok[1, :cnt[1]] < V))


def test_workspace_and_argument_checks(nq):
    B, k, V = 4, 4, 5000
    d, dl, tl = sample_case(B, k, V, 8400)
    small = torch.zeros(nq.workspace_bytes(B, k, V) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(nq.NQError) as e:
        nq.accept_greedy(dev(d), dev(tl), ws=small)
    assert e.value.status == nq.NQ_ERR_WORKSPACE
    with pytest.raises(nq.NQError) as e:
        nq.accept_sample(dev(d), dev(dl), dev(tl), 0.0, seeds_dev(synth.seeds_for(8, B)), 0)
    assert e.value.status == nq.NQ_ERR_ARG
    # a reused workspace gives the same answers call after call
    ws = nq.accept_workspace(B, k, V)
    a = [nq.accept_sample(dev(d), dev(dl), dev(tl), 1.0, seeds_dev(synth.seeds_for(9, B)), 3, ws=ws)[0].cpu()
         for _ in range(3)]
    assert torch.equal(a[0], a[1]) and torch.equal(a[1], a[2])


def test_sample_zero_residual_falls_back_to_p(nq):
    """Degenerate residual (Erge, "The same output as the large model alone";
    the reading for sum max(0, p - q) = 0): when rounding leaves p <= q at every
    entry of a rejected position, the replacement is drawn from p.  Built from
    the oracle: canonical p from logits (0, 0, -eps) is elementwise <= the
    uniform q and one ulp below it at the draft id, and a seed whose accept
    uniform lands in the one-ulp rejection window is found by search."""
    V = 3
    q_logits = np.zeros(V, np.float32)
    q = O.softmax_canonical(q_logits, 1.0)
    case = None
    for e in range(14, 30):
        p_logits = np.array([0.0, 0.0, -np.float32(2.0) ** -e], np.float32)
        p = O.softmax_canonical(p_logits, 1.0)
        if np.all(p <= q) and p[2] < q[2]:
            ratio = np.float32(p[2]) / np.float32(q[2])
            if ratio < np.float32(1.0) and (case is None or ratio < case[1]):
                case = (p_logits, ratio)
    assert case is not None
    p_logits, ratio = case
    seed = None
    for start in range(0, 1 << 27, 1 << 22):
        s = np.arange(start, start + (1 << 22), dtype=np.uint64)
        u = O.uniforms(s, 0, 0, 0)
        hit = np.nonzero(u >= ratio)[0]
        if hit.size:
            seed = int(s[hit[0]])
            break
    assert seed is not None
    d = np.array([[2]], np.int32)
    dl = q_logits.reshape(1, 1, V)
    tl = np.stack([p_logits, np.array([1.0, 2.0, 3.0], np.float32)]).reshape(1, 2, V)
    seeds = np.array([seed], np.uint64)
    cnt = check_sample(nq, d, dl, tl, 1.0, seeds, 0)
    assert list(cnt) == [1]
