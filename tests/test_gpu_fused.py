"""Fused linears of one layer input (q|k|v, gate|up) on the GPU.

"How Speculative Decoding Speeds Up Inference", Eq. (2): a round's time is
the k draft passes plus the verify pass, so each pass should stream its
weights once; q, k and v (and gate and up) read the same input, and BitNest
Fig. 3 packs the planes row by row, so one matrix of the concatenated rows
streams all of them in one linear.  Its outputs are the separate linears'
rows: packed bytes identical to the oracle's pack of the concatenated matrix,
outputs equal to the separate calls bit for bit (per-row accumulation) and
to the oracle within the linears' normwise tolerance.
"""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_helpers import TOL, bf16_dev, normwise_err
from quantized_self_speculative_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shapes,d,M", [
    ([512, 128, 128], 512, 5),        # q | k | v of a grouped-query layer (4:1)
    ([1376, 1376], 512, 1),           # gate | up
    ([256, 64, 64], 256, 16),         # q | k | v at a batched-round width
])
def test_fused_linear_equals_the_separate_linears_and_the_oracle(nq, shapes, d, M):
    G = 128
    parts = [synth.weights(7000 + i, n, d) for i, n in enumerate(shapes)]
    W = np.concatenate(parts)
    fused = nq.pack_weights(torch.from_numpy(W).cuda(), nq.FMT_NESTED44, G)
    sep = [nq.pack_weights(torch.from_numpy(p).cuda(), nq.FMT_NESTED44, G) for p in parts]
    base, resid, scales = O.pack_nested(W, G)
    host = lambda t: t.cpu().numpy().reshape(-1)
    assert np.array_equal(host(fused.base), np.ascontiguousarray(base).reshape(-1).view(np.uint8))
    assert np.array_equal(host(fused.resid), np.ascontiguousarray(resid).reshape(-1).view(np.uint8))
    assert np.array_equal(host(fused.scales), np.ascontiguousarray(scales).reshape(-1).view(np.uint8))
    # the fused planes are the separate planes stacked row by row
    assert torch.equal(fused.base, torch.cat([p.base for p in sep]))
    assert torch.equal(fused.scales, torch.cat([p.scales for p in sep]))
    x_bits = synth.activations_bf16(7100 + M, M, d)
    x = bf16_dev(x_bits)
    for verify in (False, True):
        run = nq.verify_gemm if verify else nq.draft_gemv
        y = run(fused, x).cpu().numpy()
        ys = np.concatenate([run(p, x).cpu().numpy() for p in sep], axis=1)
        assert np.array_equal(y, ys)                       # the same rows, bit for bit
        ref = O.linear(O.FMT_NESTED44, W.shape[0], d, G, base, resid, scales, x_bits, verify)
        assert normwise_err(y, ref) <= TOL
    assert nq.device_status() == 0
