"""GPU draft GEMV / verify GEMM (K2-K5) vs the fp64-accumulated oracle.

Tolerance: normwise max relative error <= 2e-3 with bf16 activations.
Planes are packed by the oracle on the CPU and uploaded, so these tests do
not depend on the GPU packer.
"""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_helpers import TOL, bf16_dev, normwise_err, oracle_fmt, oracle_packed
from quantized_self_speculative_gb300 import synth

pytestmark = pytest.mark.gpu

CASES = [  # (n, k, group): several 64-row units, ragged tails, K segments
    (1024, 1024, 128),      # the tiny single-layer workload
    (200, 640, 64),         # ragged last unit
    (77, 1152, 128),
    (130, 4096, 64),
    (40, 11008, 128),       # long K: activation staging in several segments at M > 1
]


def run_and_compare(nq, fmt, verify, n, k, g, M, seed):
    w = synth.weights(seed, n, k)
    pl, (base, resid, scales) = oracle_packed(nq, w, fmt, g)
    x = synth.activations_bf16(seed + 1, M, k)
    fn = nq.verify_gemm if verify else nq.draft_gemv
    y = fn(pl, bf16_dev(x))
    torch.cuda.synchronize()
    ref = O.linear(oracle_fmt(nq, fmt), n, k, g, base, resid, scales, x, verify)
    err = normwise_err(y.cpu().numpy(), ref)
    assert err <= TOL, (fmt, verify, n, k, g, M, err)
    return err


@pytest.mark.parametrize("n,k,g", CASES)
@pytest.mark.parametrize("M", [1, 5, 16])
def test_nested_draft_and_verify(nq, n, k, g, M):
    run_and_compare(nq, nq.FMT_NESTED44, False, n, k, g, M, 1000 + n + M)
    run_and_compare(nq, nq.FMT_NESTED44, True, n, k, g, M, 2000 + n + M)


@pytest.mark.parametrize("M", [2, 3, 7, 8, 9, 13, 17, 33])
def test_nested_other_batch_sizes(nq, M):
    run_and_compare(nq, nq.FMT_NESTED44, False, 150, 768, 128, M, 3000 + M)
    run_and_compare(nq, nq.FMT_NESTED44, True, 150, 768, 64, M, 3100 + M)


@pytest.mark.parametrize("n,k", [(300, 512), (64, 3584), (129, 1024)])
@pytest.mark.parametrize("M", [1, 3, 5, 7, 9, 16])
def test_int4_fp8_fp16_tiers(nq, n, k, M):
    run_and_compare(nq, nq.FMT_INT4, False, n, k, 128, M, 4000 + n + M)
    run_and_compare(nq, nq.FMT_FP8E4M3_ROW, True, n, k, 0, M, 4100 + n + M)
    run_and_compare(nq, nq.FMT_FP16, True, n, k, 0, M, 4200 + n + M)


def test_one_hot_columns_are_exact(nq):
    n, k, g = 96, 512, 128
    w = synth.weights(4300, n, k)
    pl, (base, resid, scales) = oracle_packed(nq, w, nq.FMT_NESTED44, g)
    cols = [0, 1, 127, 128, 300, 511]
    x = np.zeros((len(cols), k), np.uint16)
    one = synth.f32_to_bf16_bits(np.float32([1.0]))[0]
    for i, c in enumerate(cols):
        x[i, c] = one
    for verify in (False, True):
        y = (nq.verify_gemm if verify else nq.draft_gemv)(pl, bf16_dev(x))
        ref = O.linear(O.FMT_NESTED44, n, k, g, base, resid, scales, x, verify)
        assert np.array_equal(y.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("fmt", ["NESTED44", "FP8E4M3_ROW", "FP16"])
def test_batch_invariance_and_batched_call(nq, fmt):
    """Each output row is bit-identical whatever M is and whether the layer
    runs alone or inside a batched launch."""
    f = getattr(nq, "FMT_" + fmt)
    shapes = [(256, 1024), (96, 2048), (1000, 512)]
    layers, xs = [], []
    for i, (n, k) in enumerate(shapes):
        pl, _ = oracle_packed(nq, synth.weights(4400 + i, n, k), f, 128 if fmt == "NESTED44" else 0)
        layers.append(pl)
        xs.append(bf16_dev(synth.activations_bf16(4410 + i, 9, k)))
    for verify in ((False, True) if fmt == "NESTED44" else (True,)):
        fn = nq.verify_gemm if verify else nq.draft_gemv
        for pl, x in zip(layers, xs):
            full = fn(pl, x).cpu()
            for m in range(9):
                one = fn(pl, x[m:m + 1].contiguous()).cpu()
                assert torch.equal(one[0], full[m])
            assert torch.equal(fn(pl, x[:5].contiguous()).cpu(), full[:5])
        ys = [torch.empty((9, pl.n_out), dtype=torch.float32, device="cuda") for pl in layers]
        nq.LinearBatch(verify, layers, xs, ys)()
        for pl, x, y in zip(layers, xs, ys):
            assert torch.equal(y.cpu(), fn(pl, x).cpu())


def test_rejected_arguments(nq):
    pl, _ = oracle_packed(nq, synth.weights(4500, 64, 256), nq.FMT_NESTED44, 128)
    x = bf16_dev(synth.activations_bf16(4501, 2, 256))
    with pytest.raises(nq.NQError) as e:
        nq.verify_gemm(pl.as_int4(), x)             # INT4 has no refinement plane
    assert e.value.status == nq.NQ_ERR_ARG
    fp16, _ = oracle_packed(nq, synth.weights(4502, 64, 256), nq.FMT_FP16, 0)
    with pytest.raises(nq.NQError):
        nq.draft_gemv(fp16, x)                      # FP16 is a verify tier only
    y = torch.empty(2 * 64 + 1, dtype=torch.float32, device="cuda")[1:].view(2, 64)
    with pytest.raises(nq.NQError) as e:
        nq.draft_gemv(pl, x, y)
    assert e.value.status == nq.NQ_ERR_ALIGN


@pytest.mark.parametrize("g", [64, 128])
def test_every_code_pair_and_scale_class_exact(nq, g):
    """Byte-uniform planes (every (q4, r) pair, q8 down to -136) under zero,
    subnormal, small, large and negative group scales: identity activations
    return each dequantised weight q8 s / 16 (verify) or q4 s (draft) exactly."""
    from gpu_helpers import to_dev_u8
    n, k = 160, 384
    base, resid, scales = synth.random_planes(4400 + g, n, k, g)
    pl = nq.PackedLinear(n, k, g, nq.FMT_NESTED44, to_dev_u8(base), to_dev_u8(resid), to_dev_u8(scales))
    one = synth.f32_to_bf16_bits(np.float32([1.0]))[0]
    x = np.zeros((k, k), np.uint16)
    x[np.arange(k), np.arange(k)] = one
    for verify in (False, True):
        for m0 in range(0, k, 16):
            xs = x[m0:m0 + 16]
            y = (nq.verify_gemm if verify else nq.draft_gemv)(pl, bf16_dev(xs))
            ref = O.linear(O.FMT_NESTED44, n, k, g, base, resid, scales, xs, verify)
            assert np.array_equal(y.cpu().numpy().astype(np.float64), ref), (verify, m0)


@pytest.mark.parametrize("fmt", ["NESTED44", "FP8E4M3_ROW", "FP16"])
def test_wide_batch_matches_oracle_and_single_calls(nq, fmt):
    """A batch with enough rows for the widest (256-row) units: every output
    equals the oracle and, bit for bit, the layer's own single-layer call
    (4-warp units), at M = 5 and M = 9."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    f = getattr(nq, "FMT_" + fmt)
    g = 128 if fmt == "NESTED44" else 0
    shapes = []
    while sum(n for n, _ in shapes) < 2 * sms * 256 + 4096:
        i = len(shapes)
        shapes.append((4096 - 40 * (i % 3), (256, 384, 512)[i % 3]))
    layers, packs = [], []
    for i, (n, k) in enumerate(shapes):
        pl, planes = oracle_packed(nq, synth.weights(4600 + i, n, k), f, g)
        layers.append(pl)
        packs.append(planes)
    passes = (False, True) if fmt == "NESTED44" else (True,)
    for M in (5, 9):
        xs_h = [synth.activations_bf16(4700 + i + M, M, k) for i, (_, k) in enumerate(shapes)]
        xs = [bf16_dev(x) for x in xs_h]
        for verify in passes:
            ys = [torch.empty((M, n), dtype=torch.float32, device="cuda") for n, _ in shapes]
            nq.LinearBatch(verify, layers, xs, ys)()
            fn = nq.verify_gemm if verify else nq.draft_gemv
            for i in (0, 1, 2, len(shapes) - 1):
                n, k = shapes[i]
                base, resid, scales = packs[i]
                ref = O.linear(oracle_fmt(nq, f), n, k, g, base, resid, scales, xs_h[i], verify)
                assert normwise_err(ys[i].cpu().numpy(), ref) <= TOL, (fmt, M, verify, i)
            for i in range(len(shapes)):
                assert torch.equal(ys[i].cpu(), fn(layers[i], xs[i]).cpu()), (fmt, M, verify, i)
