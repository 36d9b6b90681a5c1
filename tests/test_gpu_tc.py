"""Tensor-memory (tcgen05) path of the nested-nibble linears, M >= 16
(nq_draft_gemv_batch_ws / nq_verify_gemm_batch_ws) vs the fp64-accumulated
oracle.

Tolerance: normwise max relative error <= 2e-3, as for every linear.  The
path rounds each decoded weight once to fp16 (q8 * s/16 for verify, q4 * s
for the draft), so two sharper checks pin the decoding itself: one-hot
activations return exactly those fp16 weights, and the full product agrees
with an fp64 sum over the fp16-rounded weights to within 1e-5 (fp32
accumulation).
"""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_helpers import TOL, bf16_dev, normwise_err, oracle_fmt, oracle_packed
from quantized_self_speculative_gb300 import synth

pytestmark = pytest.mark.gpu


def _nibbles(a: np.ndarray, n: int, k: int) -> np.ndarray:
    """Signed 4-bit codes [n][k] from a packed plane (element 2j in the low nibble of byte j)."""
    b = np.asarray(a, dtype=np.uint8).reshape(n, k // 2)
    lo = (b & 0xF).astype(np.int16)
    hi = (b >> 4).astype(np.int16)
    codes = np.empty((n, k), dtype=np.int16)
    codes[:, 0::2], codes[:, 1::2] = lo, hi
    return np.where(codes >= 8, codes - 16, codes)


def fp16_weights(base, resid, scales, n, k, g, verify):
    """Decoded weights rounded once to fp16, as the tensor-core path feeds them."""
    s = np.asarray(scales).view(np.float16).reshape(n, k // g).astype(np.float64)
    q4 = _nibbles(base, n, k).astype(np.float64)
    srow = np.repeat(s, g, axis=1)
    if verify:
        q8 = 16 * q4 + _nibbles(resid, n, k).astype(np.float64)
        return (q8 * srow / 16).astype(np.float16)
    return (q4 * srow).astype(np.float16)


def run_tc(nq, layers, xs, M, verify):
    ys = [torch.empty((M, L.n_out), dtype=torch.float32, device="cuda") for L in layers]
    b = nq.LinearBatch(verify, layers, [bf16_dev(x) for x in xs], ys, tensor_cores=True)
    assert b.ws.numel() >= nq.linear_workspace_bytes(verify, layers, M) > 0
    torch.cuda.synchronize()
    nq.device_status()                 # clear the sticky word
    b()
    torch.cuda.synchronize()
    assert nq.device_status() == 0
    return [y.cpu().numpy() for y in ys]


CASES = [  # (fmt, verify, n, k, group, M)
    ("NESTED44", True, 128, 128, 128, 16),     # one tile, one k-block
    ("NESTED44", True, 200, 384, 128, 16),     # ragged tile, 3 k-blocks
    ("NESTED44", True, 300, 512, 64, 40),      # group 64, N padded to 48
    ("NESTED44", True, 257, 256, 128, 144),    # the batched-verify width
    ("NESTED44", True, 130, 1024, 64, 256),    # widest single chunk
    ("NESTED44", True, 129, 256, 128, 300),    # two M chunks (256 + 44)
    ("NESTED44", False, 200, 384, 128, 16),    # draft: base plane only
    ("NESTED44", False, 333, 640, 64, 33),
    ("INT4", False, 140, 512, 128, 144),
    # 256-input k-blocks (padded M <= 64 and k % 256 == 0)
    ("NESTED44", True, 1000, 1024, 128, 16),
    ("NESTED44", False, 1000, 1024, 128, 16),
    ("NESTED44", True, 130, 768, 64, 64),
    ("NESTED44", False, 257, 512, 64, 20),
    ("INT4", False, 300, 1536, 128, 48),
]


@pytest.mark.parametrize("fmt,verify,n,k,g,M", CASES)
def test_tc_matches_oracle(nq, fmt, verify, n, k, g, M):
    f = getattr(nq, "FMT_" + fmt)
    seed = 7000 + n + k + M + (1 if verify else 0)
    w = synth.weights(seed, n, k)
    pl, (base, resid, scales) = oracle_packed(nq, w, f, g)
    x = synth.activations_bf16(seed + 1, M, k)
    (y,) = run_tc(nq, [pl], [x], M, verify)
    ref = O.linear(oracle_fmt(nq, f), n, k, g, base, resid, scales, x, verify)
    err = normwise_err(y, ref)
    assert err <= TOL, (fmt, verify, n, k, g, M, err)
    # the same product over the fp16-rounded weights, to fp32 accumulation error
    w16 = fp16_weights(base, resid, scales, n, k, g, verify).astype(np.float64)
    xf = synth.bf16_bits_to_f32(x).astype(np.float16).astype(np.float64)
    ref16 = xf @ w16.T
    assert normwise_err(y, ref16) <= 1e-5, normwise_err(y, ref16)


def test_tc_one_hot_returns_fp16_weights(nq):
    n, k, g, M = 150, 256, 64, 16
    w = synth.weights(7100, n, k)
    for verify in (False, True):
        pl, (base, resid, scales) = oracle_packed(nq, w, nq.FMT_NESTED44, g)
        cols = np.arange(M) * (k // M) + 3
        x = np.zeros((M, k), dtype=np.uint16)
        x[np.arange(M), cols] = 0x3F80   # bf16 1.0
        (y,) = run_tc(nq, [pl], [x], M, verify)
        w16 = fp16_weights(base, resid, scales, n, k, g, verify).astype(np.float32)
        np.testing.assert_array_equal(y, w16[:, cols].T)


def test_tc_large_scales_take_the_exact_slow_path(nq):
    """Groups with s > 0.0625 (|w| up to ~0.5 and beyond) decode through the
    1024-biased path; mixed with small groups in the same warp."""
    n, k, g, M = 256, 512, 128, 32
    w = synth.weights(7200, n, k)
    w[::3] *= 40.0                     # every third row: s ~ 0.3
    w[5, :128] *= 500.0                # one group with s ~ 4
    for verify in (False, True):
        pl, (base, resid, scales) = oracle_packed(nq, w, nq.FMT_NESTED44, g)
        x = synth.activations_bf16(7201, M, k)
        (y,) = run_tc(nq, [pl], [x], M, verify)
        ref = O.linear(O.FMT_NESTED44, n, k, g, base, resid, scales, x, verify)
        assert normwise_err(y, ref) <= TOL
        w16 = fp16_weights(base, resid, scales, n, k, g, verify).astype(np.float64)
        ref16 = synth.bf16_bits_to_f32(x).astype(np.float16).astype(np.float64) @ w16.T
        assert normwise_err(y, ref16) <= 1e-5


def test_tc_batch_of_layers_matches_single_calls(nq):
    """Several linears of different shapes in one persistent launch: each
    output equals the oracle, and the batch equals per-layer launches bit for
    bit (tile order never changes a tile's arithmetic)."""
    shapes = [(384, 256), (130, 640), (1000, 128), (257, 384)]
    M, g = 24, 128
    layers, packs, xs = [], [], []
    for i, (n, k) in enumerate(shapes):
        pl, planes = oracle_packed(nq, synth.weights(7300 + i, n, k), nq.FMT_NESTED44, g)
        layers.append(pl)
        packs.append(planes)
        xs.append(synth.activations_bf16(7400 + i, M, k))
    for verify in (False, True):
        ys = run_tc(nq, layers, xs, M, verify)
        for (n, k), (base, resid, scales), x, y in zip(shapes, packs, xs, ys):
            ref = O.linear(O.FMT_NESTED44, n, k, g, base, resid, scales, x, verify)
            assert normwise_err(y, ref) <= TOL
        singles = [run_tc(nq, [L], [x], M, verify)[0] for L, x in zip(layers, xs)]
        for a, b in zip(ys, singles):
            np.testing.assert_array_equal(a, b)


def test_tc_small_m_falls_back(nq):
    """M < 16 needs no workspace and runs the streaming kernel through the
    *_ws entry point, bit-identical to the plain call."""
    n, k, g, M = 200, 512, 128, 9
    pl, _ = oracle_packed(nq, synth.weights(7500, n, k), nq.FMT_NESTED44, g)
    assert nq.linear_workspace_bytes(True, [pl], M) == 0
    x = bf16_dev(synth.activations_bf16(7501, M, k))
    ys = [torch.empty((M, n), dtype=torch.float32, device="cuda")]
    nq.LinearBatch(True, [pl], [x], ys, tensor_cores=True)()
    y_plain = nq.verify_gemm(pl, x)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ys[0].cpu().numpy(), y_plain.cpu().numpy())


def _upload_planes(nq, base, resid, scales, n, k, g):
    from gpu_helpers import to_dev_u8
    return nq.PackedLinear(n, k, g, nq.FMT_NESTED44, to_dev_u8(base), to_dev_u8(resid), to_dev_u8(scales))


@pytest.mark.parametrize("g", [64, 128])
@pytest.mark.parametrize("rows_per_call", [256, 64])   # 128-input k-blocks; 256-input k-blocks (padded M <= 64)
def test_tc_every_code_pair_and_scale_class(nq, g, rows_per_call):
    """Byte-uniform planes (all 256 (q4, r) pairs, q4 = -8 with r < 0 included:
    q8 = 16 q4 + r reaches -136) under zero, subnormal, fast, slow and negative
    group scales; identity activations read back every decoded weight, which
    must be fp16(q8 s / 16) (verify) or fp16(q4 s) (draft), rounded once."""
    n, k = 192, 512
    base, resid, scales = synth.random_planes(7600 + g, n, k, g)
    pl = _upload_planes(nq, base, resid, scales, n, k, g)
    one = synth.f32_to_bf16_bits(np.float32([1.0]))[0]
    for verify in (False, True):
        w16 = fp16_weights(base, resid, scales, n, k, g, verify).astype(np.float32)
        for c0 in range(0, k, rows_per_call):
            x = np.zeros((rows_per_call, k), np.uint16)
            x[np.arange(rows_per_call), c0 + np.arange(rows_per_call)] = one
            (y,) = run_tc(nq, [pl], [x], rows_per_call, verify)
            np.testing.assert_array_equal(y, w16[:, c0:c0 + rows_per_call].T)
            ref = O.linear(O.FMT_NESTED44, n, k, g, base, resid, scales, x, verify)
            assert normwise_err(y, ref) <= 2.0 ** -11


def test_tc_repeated_launches_are_bit_identical(nq):
    """Warp-specialised stages hand data over through mbarriers; a missed
    hand-off would show up as run-to-run differences.  Twelve launches of a
    multi-layer batch at the batched-verify width give one result."""
    shapes = [(1024, 1024), (300, 2048), (640, 512)]
    M, g = 144, 128
    layers = [oracle_packed(nq, synth.weights(7700 + i, n, k), nq.FMT_NESTED44, g)[0]
              for i, (n, k) in enumerate(shapes)]
    xs = [bf16_dev(synth.activations_bf16(7710 + i, M, k)) for i, (_, k) in enumerate(shapes)]
    for verify in (False, True):
        ys = [torch.empty((M, n), dtype=torch.float32, device="cuda") for n, _ in shapes]
        b = nq.LinearBatch(verify, layers, xs, ys, tensor_cores=True)
        first = None
        for _ in range(12):
            for y in ys:
                y.fill_(float("nan"))
            b()
            got = [y.cpu() for y in ys]
            if first is None:
                first = got
            else:
                for a, c in zip(first, got):
                    assert torch.equal(a, c)


def test_bounded_wait_gives_up_and_the_context_stays_usable(nq):
    """Failure path of the bounded mbarrier waits, without a GPU fault: a wait
    that nothing completes gives up after its limit and reports
    NQ_DEV_TIMEOUT; later launches run clean."""
    import time
    torch.cuda.synchronize()
    nq.device_status()
    t0 = time.perf_counter()
    nq.selftest_bounded_wait(20000)          # 20 ms
    st = nq.device_status()
    dt = time.perf_counter() - t0
    assert st & nq.NQ_DEV_TIMEOUT, st
    assert 0.02 <= dt < 10.0, dt
    # the context is usable: a tensor-core pass afterwards is correct and clean
    n, k, g, M = 200, 512, 128, 32
    pl, (base, resid, scales) = oracle_packed(nq, synth.weights(7800, n, k), nq.FMT_NESTED44, g)
    x = synth.activations_bf16(7801, M, k)
    (y,) = run_tc(nq, [pl], [x], M, True)
    ref = O.linear(O.FMT_NESTED44, n, k, g, base, resid, scales, x, True)
    assert normwise_err(y, ref) <= TOL


def test_tc_full_width_batch_is_repeatable(nq):
    """The batched-verify workload itself (8 LLaMA-3-8B-shaped layers, M = 144,
    2688 tiles): 30 launches give one bit pattern.  A missing proxy fence
    between the decoders' shared-memory reads and the TMA refill of a weight
    stage showed up here as a differing tile in about one pass in ten."""
    layer, _, _ = synth.llama3_8b_linears()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(77)
    layers = []
    for _ in range(8):
        for _, n, k in layer:
            w = torch.randn((n, k), generator=gen, device="cuda").mul_(0.02)
            layers.append(nq.pack_weights(w, nq.FMT_NESTED44, 128))
            del w
    M = 144
    xs = [torch.randn((M, L.k_in), generator=gen, device="cuda").to(torch.bfloat16) for L in layers]
    ys = [torch.empty((M, L.n_out), dtype=torch.float32, device="cuda") for L in layers]
    b = nq.LinearBatch(True, layers, xs, ys, tensor_cores=True)
    b()
    torch.cuda.synchronize()
    first = [y.clone() for y in ys]
    for _ in range(30):
        b()
        torch.cuda.synchronize()
        for y, y0 in zip(ys, first):
            assert torch.equal(y, y0)
    assert nq.device_status() == 0
