"""Range of the activations the linears accept (bf16 in, fp16 inside).

The kernels round each bf16 activation to fp16 before multiplying (the 4-bit
codes, E4M3 and fp16 weights are exact in fp16; the tensor cores take one
16-bit type for both operands).  That is exact for 2^-14 <= |x| <= 65504;
the nibble kernels stage odd-indexed inputs as x/16 (their refinement nibble
carries a factor 16), which keeps every x with |x| >= 2^-10 exact.  Larger
magnitudes set NQ_DEV_ACT_RANGE; smaller ones lose low bits to fp16
subnormals.  These tests pin both ends against the fp64 oracle, row by row
(each row's error relative to that row's largest output).
"""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_helpers import TOL, bf16_dev, normwise_err, oracle_fmt, oracle_packed
from quantized_self_speculative_gb300 import synth

pytestmark = pytest.mark.gpu

FORMATS = [("NESTED44", False, 128), ("NESTED44", True, 64), ("INT4", False, 128),
           ("FP8E4M3_ROW", True, 0), ("FP16", True, 0)]


def scaled_rows(seed, scales, k):
    """Row m ~ N(0, 1) * scales[m], rounded to bf16 (bits)."""
    z = synth.rng(seed).standard_normal((len(scales), k), dtype=np.float32)
    x = z * np.asarray(scales, np.float32)[:, None]
    return synth.f32_to_bf16_bits(x)


def run(nq, fmt_name, verify, g, x, n=192, k=1536, seed=7000, tensor_cores=False):
    fmt = getattr(nq, "FMT_" + fmt_name)
    w = synth.weights(seed, n, k)
    pl, (base, resid, scales) = oracle_packed(nq, w, fmt, g)
    nq.device_status()   # clear
    if tensor_cores:
        y = torch.empty((x.shape[0], n), dtype=torch.float32, device="cuda")
        nq.LinearBatch(verify, [pl], [bf16_dev(x)], [y], tensor_cores=True)()
    else:
        y = (nq.verify_gemm if verify else nq.draft_gemv)(pl, bf16_dev(x))
    status = nq.device_status()
    ref = O.linear(oracle_fmt(nq, fmt), n, k, g, base, resid, scales, x, verify)
    return y.cpu().numpy(), ref, status


@pytest.mark.parametrize("fmt_name,verify,g", FORMATS)
def test_every_decade_of_the_exact_range(nq, fmt_name, verify, g):
    """Rows scaled from 2^-10 up to 1.5e4 (largest |x| about 6e4): each row
    within the 2e-3 normwise bound of its own outputs; no range flag."""
    row_scales = [2.0 ** -10 * 4, 2.0 ** -8, 1e-2, 0.3, 1.0, 30.0, 1e3, 1.5e4]
    x = scaled_rows(7100, row_scales, 1536)
    assert np.abs(synth.bf16_bits_to_f32(x)).max() <= 65504
    y, ref, status = run(nq, fmt_name, verify, g, x)
    assert status & nq.NQ_DEV_ACT_RANGE == 0
    for m in range(len(row_scales)):
        assert normwise_err(y[m:m + 1], ref[m:m + 1]) <= TOL, (m, row_scales[m])


@pytest.mark.parametrize("fmt_name,verify,g", FORMATS)
def test_tiny_activations_degrade_gracefully(nq, fmt_name, verify, g):
    """Rows whose every |x| lies between 2^-20 and 2^-10 meet fp16 subnormals
    (spacing 2^-24, or 2^-20 for the nibble kernels' x/16): the error is that
    rounding's, a few percent at most, and nothing is flushed to zero."""
    z = synth.rng(7200).uniform(-20, -10, size=(4, 1536))
    sign = np.where(synth.rng(7201).random((4, 1536)) < 0.5, -1.0, 1.0)
    x = synth.f32_to_bf16_bits((sign * 2.0 ** z).astype(np.float32))
    y, ref, status = run(nq, fmt_name, verify, g, x)
    assert status & nq.NQ_DEV_ACT_RANGE == 0
    for m in range(4):
        assert np.abs(ref[m]).max() > 0
        assert normwise_err(y[m:m + 1], ref[m:m + 1]) <= 0.05, m


@pytest.mark.parametrize("fmt_name,verify,g", FORMATS)
def test_beyond_fp16_sets_the_range_flag(nq, fmt_name, verify, g):
    """One row holds an activation of 1e5: NQ_DEV_ACT_RANGE is set and the
    other rows (batch invariance: rows do not interact) stay exact."""
    x = scaled_rows(7300, [1.0, 1.0, 1.0], 1536)
    big = synth.f32_to_bf16_bits(np.float32([1e5]))[0]
    x[1, 77] = big
    y, ref, status = run(nq, fmt_name, verify, g, x)
    assert status & nq.NQ_DEV_ACT_RANGE
    for m in (0, 2):
        assert normwise_err(y[m:m + 1], ref[m:m + 1]) <= TOL


@pytest.mark.parametrize("verify", [False, True])
def test_tensor_core_path_range(nq, verify):
    """The tensor-core linears (M >= 16 with a workspace) stage the same fp16
    activations: decades within range pass, 1e5 sets the flag."""
    row_scales = [2.0 ** -10 * 4, 1e-2, 1.0, 1e3, 1.5e4] * 4
    x = scaled_rows(7400, row_scales, 1536)
    y, ref, status = run(nq, "NESTED44", verify, 128, x, n=256, tensor_cores=True)
    assert status & nq.NQ_DEV_ACT_RANGE == 0
    for m in range(len(row_scales)):
        assert normwise_err(y[m:m + 1], ref[m:m + 1]) <= TOL, (m, row_scales[m])
    x[3, 5] = synth.f32_to_bf16_bits(np.float32([-1e5]))[0]
    _, _, status = run(nq, "NESTED44", verify, 128, x, n=256, tensor_cores=True)
    assert status & nq.NQ_DEV_ACT_RANGE
