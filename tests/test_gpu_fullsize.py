"""Parity at the benchmark's full sizes, in the launch configuration the bench
times, on sampled outputs.

"How Speculative Decoding Speeds Up Inference", Eq. (2): a round is k draft
passes and one verify pass over every linear of the model.  The bench times
each pass as one persistent launch over all of them: the LLaMA-2-7B round
(32 layers x q, k, v, o, gate, up, down, then lm_head; draft M = 1 on the
base plane, verify M = k + 1 = 5 on both planes), and the batched rounds of
LLaMA-3-8B on the tensor-memory kernel (draft M = 16, verify M = 144).

Output row j of a linear depends only on weight row j and the activations
(BitNest Fig. 3 packs the planes row by row, groups along the row), so the
oracle recomputes a few rows of every linear one by one: it packs the same
seeded float rows itself (the device's packed bytes of those rows must be
identical) and multiplies them with the same activations; the device's rows
must agree within the linears' normwise tolerance.
"""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_helpers import TOL, bf16_dev, normwise_err
from quantized_self_speculative_gb300 import synth

pytestmark = pytest.mark.gpu

G = 128
ROWS_PER_LINEAR = 4


def model_shapes(spec):
    layer, lm, n_layers = spec()
    return [(n, k) for _ in range(n_layers) for _, n, k in layer] + [(lm[1], lm[2])]


def build(nq, shapes, seed):
    """Pack every linear (float weights drawn on the device, as the bench
    does); keep the float rows sampled for the oracle."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    pick = np.random.default_rng(seed + 1)
    layers, picked = [], []
    for n, k in shapes:
        w = torch.randn((n, k), generator=gen, device="cuda", dtype=torch.float32).mul_(0.02)
        rows = np.unique(np.concatenate([[0, n - 1], pick.integers(0, n, ROWS_PER_LINEAR - 2)]))
        picked.append((rows, w[torch.from_numpy(rows).cuda()].cpu().numpy()))
        layers.append(nq.pack_weights(w, nq.FMT_NESTED44, G))
        del w
    torch.cuda.synchronize()
    return layers, picked


def check_pass(nq, layers, picked, M, verify, tensor_cores, seed):
    xs_bits = [synth.activations_bf16(seed + i, M, L.k_in) for i, L in enumerate(layers)]
    xs = [bf16_dev(b) for b in xs_bits]
    ys = [torch.empty((M, L.n_out), dtype=torch.float32, device="cuda") for L in layers]
    nq.LinearBatch(verify, layers, xs, ys, tensor_cores=tensor_cores)()
    torch.cuda.synchronize()
    worst = 0.0
    for L, (rows, wrows), xb, y in zip(layers, picked, xs_bits, ys):
        base, resid, scales = O.pack_nested(wrows, G)
        idx = torch.from_numpy(rows).cuda()
        kb, ks = L.k_in // 2, (L.k_in // G) * 2
        assert np.array_equal(L.base.view(L.n_out, kb)[idx].cpu().numpy(), base)
        assert np.array_equal(L.resid.view(L.n_out, kb)[idx].cpu().numpy(), resid)
        assert np.array_equal(L.scales.view(L.n_out, ks)[idx].cpu().numpy().view(np.uint16), scales)
        ref = O.linear(O.FMT_NESTED44, len(rows), L.k_in, G, base, resid, scales, xb, verify)
        err = normwise_err(y[:, idx].cpu().numpy(), ref)
        worst = max(worst, err)
        assert err <= TOL, (L.n_out, L.k_in, M, verify, err)
    assert nq.device_status() == 0
    return worst


def test_llama2_7b_round_passes_sampled_rows(nq):
    """The round's draft pass (M = 1) and verify pass (M = 5): 225 linears in
    one streaming launch each, as timed by the bench."""
    layers, picked = build(nq, model_shapes(synth.llama2_7b_linears), 811)
    check_pass(nq, layers, picked, 1, False, False, 900)
    check_pass(nq, layers, picked, 5, True, False, 1900)
    del layers
    torch.cuda.empty_cache()


def test_llama3_8b_batched_round_passes_sampled_rows(nq):
    """Batched rounds (B = 16, k = 8): draft M = 16 and verify M = 144 over
    the 225 linears of LLaMA-3-8B on the tensor-memory kernel, one launch each."""
    layers, picked = build(nq, model_shapes(synth.llama3_8b_linears), 812)
    check_pass(nq, layers, picked, 16, False, True, 2900)
    check_pass(nq, layers, picked, 144, True, True, 3900)
    del layers
    torch.cuda.empty_cache()
