"""Int8-activation linears on the GPU vs the oracle (BitNest Table 1, "W4A8
-> W8A8"; Table 12).  The activation codes and row scales are bit-exact; the
products of codes are exact integers on both sides, so the outputs differ
only by the fp32 order of the scaling (normwise below 1e-5); each output row
is independent of the other activation rows (bit for bit)."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_helpers import bf16_dev, normwise_err, oracle_packed
from quantized_self_speculative_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K", [(1, 4096), (5, 11008), (9, 64), (3, 1000 * 8)])
def test_activation_codes_bit_exact(nq, M, K):
    x = synth.activations_bf16(1300 + M, M, K, std=2.0)
    if M > 2:
        x[1] = 0
    xq, sx = nq.quantize_act_int8(bf16_dev(x))
    rq, rs = O.quantize_act_int8(x)
    assert np.array_equal(xq.cpu().numpy(), rq)
    assert np.array_equal(sx.cpu().numpy(), rs)
    assert nq.device_status() == 0


@pytest.mark.parametrize("n,k,g", [(4096, 4096, 128), (130, 11008, 128), (77, 512, 64), (1000, 3584, 64)])
@pytest.mark.parametrize("M", [1, 5, 9])
@pytest.mark.parametrize("verify", [False, True])
def test_a8_linear_matches_oracle(nq, n, k, g, M, verify):
    w = synth.weights(1400 + n + k, n, k)
    pl, (base, resid, scales) = oracle_packed(nq, w, nq.FMT_NESTED44, g)
    x = synth.activations_bf16(1500 + M + k, M, k)
    xq, sx = nq.quantize_act_int8(bf16_dev(x))
    y = nq.linear_a8(pl, xq, sx, verify).cpu().numpy()
    rq, rs = O.quantize_act_int8(x)
    ref = O.linear_a8(O.FMT_NESTED44, n, k, g, base, resid, scales, rq, rs, verify)
    assert normwise_err(y, ref) <= 1e-5
    # row independence: the last activation row alone gives the same bits
    y1 = nq.linear_a8(pl, xq[M - 1:].contiguous(), sx[M - 1:].contiguous(), verify).cpu().numpy()
    assert np.array_equal(y1[0], y[M - 1])


def test_int4_draft_and_batched_call(nq):
    shapes = [(256, 1024), (96, 2048), (1000, 512)]
    layers, xs, refs = [], [], []
    for i, (n, k) in enumerate(shapes):
        w = synth.weights(1600 + i, n, k)
        pl, (base, resid, scales) = oracle_packed(nq, w, nq.FMT_INT4, 128)
        x = synth.activations_bf16(1610 + i, 5, k)
        xq, sx = nq.quantize_act_int8(bf16_dev(x))
        layers.append(pl)
        xs.append((xq, sx))
        rq, rs = O.quantize_act_int8(x)
        refs.append(O.linear_a8(O.FMT_INT4, n, k, 128, base, None, scales, rq, rs, False))
    ys = [torch.empty((5, n), dtype=torch.float32, device="cuda") for n, _ in shapes]
    nq.LinearA8Batch(False, layers, [a for a, _ in xs], [b for _, b in xs], ys)()
    for y, ref, L, (xq, sx) in zip(ys, refs, layers, xs):
        assert normwise_err(y.cpu().numpy(), ref) <= 1e-5
        assert torch.equal(y, nq.linear_a8(L, xq, sx, False))       # batched = single calls, bit for bit
