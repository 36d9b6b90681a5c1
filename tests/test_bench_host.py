"""Host-side accounting of bench.py (no GPU): the algorithmic bytes behind
the roofline figures and the JSON line's whole-job value."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from quantized_self_speculative_gb300 import synth  # noqa: E402


def _pass_bytes(fn, M):
    layer, lm, n_layers = synth.llama2_7b_linears()
    shapes = [(n, k) for _ in range(n_layers) for _, n, k in layer] + [(lm[1], lm[2])]
    assert len(shapes) == 225
    return sum(fn(n, k, M) for n, k in shapes)


def test_draft_and_verify_pass_bytes_of_the_round():
    # base plane 0.5 B / weight, both planes 1 B / weight, fp16 scales per 128
    # inputs, bf16 activations in, fp32 outputs out: the figures the bench
    # divides by the CUDA-event time
    assert _pass_bytes(bench.draft_bytes, 1) == 3_414_627_328
    assert _pass_bytes(bench.verify_bytes, 5) == 6_749_578_240
    weights = _pass_bytes(lambda n, k, M: n * k, 1)
    assert _pass_bytes(bench.verify_bytes, 5) - 2 * (_pass_bytes(bench.draft_bytes, 1)) < 0.01 * weights


def test_acceptance_bytes_read_every_logit_once():
    B, k, V = 64, 4, 152064
    assert bench.accept_bytes(B, k, V, False) >= 4 * B * (k + 1) * V
    assert bench.accept_bytes(B, k, V, True) >= 4 * B * (2 * k + 1) * V
    assert bench.accept_bytes(B, k, V, True) - 4 * B * (2 * k + 1) * V < 4096 * B


def test_measured_traffic_constant_is_close_to_the_algorithmic_bytes():
    # the algorithmic bytes count the activations and outputs, which may stay
    # in L2: DRAM traffic can fall a little below them, never far
    ratio = bench.DRAFT_PASS_DRAM_BYTES / _pass_bytes(bench.draft_bytes, 1)
    assert 0.99 <= ratio < 1.05
