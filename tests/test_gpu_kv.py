"""Nested KV cache on the GPU vs the oracle (BitNest, Fig. 4: the draft reads
the low-bit base view, verification the full b_kv + r_kv-bit view of the same
cache; accepted entries stay, the rejected suffix is discarded).

Appending quantises rows exactly like the weights (bit-exact against the
oracle's pack of the same rows); attention over either view agrees with the
oracle's fp64 attention over the same dequantised rows (normwise, per output
vector, within the linears' 2e-3: the kernel feeds the tensor cores fp16
queries and fp16 probabilities, about 2^-11 relative each, and accumulates in
fp32).
"""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_helpers import normwise_err
from quantized_self_speculative_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = 2e-3


def rows(seed, *shape):
    return synth.rng(seed).standard_normal(shape).astype(np.float32)


def fill(nq, B, Hkv, d, G, L, lens, seed):
    """A cache holding lens[b] rows per sequence, appended in two chunks."""
    cache = nq.KVCache(B, Hkv, d, G, L)
    K = rows(seed, B, Hkv, L, d)
    V = rows(seed + 1, B, Hkv, L, d)
    first = min(lens) // 2
    for lo, hi in ((0, first), (first, max(lens))):
        k = torch.from_numpy(np.ascontiguousarray(K[:, :, lo:hi])).cuda()
        v = torch.from_numpy(np.ascontiguousarray(V[:, :, lo:hi])).cuda()
        cache.append(k, v, torch.full((B,), lo, dtype=torch.int32, device="cuda"))
    return cache, K, V


@pytest.mark.parametrize("d,G", [(128, 128), (128, 64), (64, 64)])
def test_append_matches_oracle_pack(nq, d, G):
    B, Hkv, L = 2, 3, 300
    cache, K, V = fill(nq, B, Hkv, d, G, L, [300, 300], 1000 + d + G)
    h = cache.host_dict()
    for name, X in (("k", K), ("v", V)):
        base, resid, scales = O.kv_rows_pack(X, G)
        assert np.array_equal(h[name + "_base"], base)
        assert np.array_equal(h[name + "_resid"], resid)
        assert np.array_equal(h[name + "_scales"], scales)
    assert nq.device_status() == 0


@pytest.mark.parametrize("B,Hq,Hkv,d,G,M,lens", [
    (1, 4, 4, 128, 128, 1, [700]),            # MHA draft step, ragged last split
    (1, 4, 4, 128, 128, 5, [700]),            # MHA verify over k + 1 = 5 positions
    (3, 8, 2, 64, 64, 9, [257, 40, 1000]),    # GQA (4 query heads per kv head), batch of unequal lengths
    (2, 28, 4, 128, 128, 3, [513, 600]),      # Qwen2.5-7B head layout
    (2, 28, 4, 128, 128, 1, [513, 600]),      # its draft step: 7 query vectors per kv head (keys-as-rows kernel)
    (1, 8, 2, 128, 64, 2, [333]),             # two groups per row, exactly 8 query vectors per kv head
    (1, 8, 2, 128, 64, 3, [450]),             # two groups per row, 12 query vectors per kv head (query tiles)
])
@pytest.mark.parametrize("planes", [1, 2])
def test_attention_matches_oracle(nq, B, Hq, Hkv, d, G, M, lens, planes):
    L = 1024
    cache, _, _ = fill(nq, B, Hkv, d, G, L, lens, 2000 + Hq + M)
    q = rows(3000 + M, B, M, Hq, d)
    ln = torch.tensor(lens, dtype=torch.int32, device="cuda")
    scale = 1.0 / np.sqrt(d)
    out = cache.attention(torch.from_numpy(q).cuda(), ln, planes, scale).cpu().numpy()
    ref = O.attn_decode(q, cache.host_dict(), np.array(lens, np.int32), planes, scale)
    err = max(normwise_err(out[b, m, h][None], ref[b, m, h][None])
              for b in range(B) for m in range(M) for h in range(Hq))
    assert err <= TOL, err
    assert nq.device_status() == 0


@pytest.mark.parametrize("planes,M", [(1, 1), (2, 5)])
def test_attention_long_splits_match_oracle(nq, planes, M):
    """Enough (sequence, kv head) pairs that the kernel takes its longest
    splits (1024 cache rows per CTA, 16 blocks per warp through the four-stage
    ring), with lengths that end inside a block and inside a split."""
    B, H, d, G, L = 4, 16, 128, 128, 4096
    lens = [4000, 3077, 1025, 4096]
    cache, _, _ = fill(nq, B, H, d, G, L, lens, 5000 + planes)
    q = rows(5100 + M, B, M, H, d)
    ln = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = cache.attention(torch.from_numpy(q).cuda(), ln, planes, 0.09).cpu().numpy()
    ref = O.attn_decode(q, cache.host_dict(), np.array(lens, np.int32), planes, 0.09)
    err = max(normwise_err(out[b, m, h][None], ref[b, m, h][None])
              for b in range(B) for m in range(M) for h in range(H))
    assert err <= TOL, err
    assert nq.device_status() == 0


def test_draft_view_differs_from_target_view_and_suffix_discard(nq):
    """The 4-bit and 8-bit views give different attention (the base alone is
    a coarser copy); rows past a sequence's length are never read, so after a
    rejected suffix is dropped (a shorter length) the result equals a cache
    that never held those rows."""
    B, H, d, G, L = 1, 2, 128, 128, 512
    cache, K, V = fill(nq, B, H, d, G, L, [400], 4000)
    q = torch.from_numpy(rows(4001, B, 1, H, d)).cuda()
    ln = torch.tensor([400], dtype=torch.int32, device="cuda")
    a4 = cache.attention(q, ln, 1, 0.1)
    a8 = cache.attention(q, ln, 2, 0.1)
    assert (a4 - a8).abs().max().item() > 1e-3
    # five verified rows appended at 400..404; three rejected -> the length becomes 402
    extra = torch.from_numpy(rows(4002, B, H, 5, d)).cuda()
    cache.append(extra, extra, torch.tensor([400], dtype=torch.int32, device="cuda"))
    short = cache.attention(q, torch.tensor([402], dtype=torch.int32, device="cuda"), 2, 0.1)
    ref_cache, _, _ = fill(nq, B, H, d, G, L, [400], 4000)
    ref_cache.append(extra[:, :, :2].contiguous(), extra[:, :, :2].contiguous(),
                     torch.tensor([400], dtype=torch.int32, device="cuda"))
    ref = ref_cache.attention(q, torch.tensor([402], dtype=torch.int32, device="cuda"), 2, 0.1)
    assert torch.equal(short, ref)
    assert nq.device_status() == 0


@pytest.mark.parametrize("Hq,Hkv,kv_sel", [(32, 32, [0, 9, 22, 31]), (28, 4, [0, 3])])
def test_attention_32k_bench_workload_sampled_heads(nq, Hq, Hkv, kv_sel):
    """The benchmark's attention workload at full size: one sequence of 32768
    cached rows in a cache of 32768 + 16, d = 128, G = 128, LLaMA-2-7B-32K
    (MHA) and Qwen2.5-7B (GQA) heads; the draft read of the KV4 view at M = 1
    and the verify read of the KV8 view at M = k + 1 = 5, through the same
    entry point and split rule.  The oracle recomputes every query head of a
    few kv heads (the heads are independent)."""
    B, d, G, ctx = 1, 128, 128, 32768
    cache, _, _ = fill(nq, B, Hkv, d, G, ctx + 16, [ctx], 6000 + Hkv)
    sub = {n: np.ascontiguousarray(a[:, kv_sel]) for n, a in cache.host_dict().items()}
    g = Hq // Hkv
    q_sel = [kv * g + j for kv in kv_sel for j in range(g)]
    ln = torch.tensor([ctx], dtype=torch.int32, device="cuda")
    for M, planes in ((1, 1), (5, 2)):
        q = rows(6100 + 10 * M + Hkv, B, M, Hq, d)
        out = cache.attention(torch.from_numpy(q).cuda(), ln, planes, d ** -0.5).cpu().numpy()[:, :, q_sel]
        ref = O.attn_decode(np.ascontiguousarray(q[:, :, q_sel]), sub, np.array([ctx], np.int32), planes, d ** -0.5)
        err = max(normwise_err(out[0, m, i][None], ref[0, m, i][None]) for m in range(M) for i in range(len(q_sel)))
        assert err <= TOL, (M, planes, err)
    assert nq.device_status() == 0
