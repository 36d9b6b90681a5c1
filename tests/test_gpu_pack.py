"""GPU pack (K1) vs the CPU oracle: bit-exact bytes and scales."""
import numpy as np
import pytest
import torch

import oracle as O
from quantized_self_speculative_gb300 import synth

pytestmark = pytest.mark.gpu


def special_rows(w):
    w = w.copy()
    w[0] = 0.0                                   # zero row -> s = 0 -> all codes 0
    w[1] = 0.013                                 # constant row
    w[2, ::3] = -w[2, ::3] * 50                  # large outliers in some groups
    w[3] = np.float32(1e-7) * np.sign(w[3])      # tiny values: the fp16 scale underflows to 0
    w[4] = np.float32(1e-6) * np.sign(w[4])      # the fp16 scale is subnormal
    return w


@pytest.mark.parametrize("n,k,g", [(1024, 1024, 128), (200, 640, 64), (77, 768, 128), (5, 64, 64)])
def test_nested_pack_bit_exact(nq, n, k, g):
    w = special_rows(synth.weights(500 + n, n, k))
    for fmt in (nq.FMT_NESTED44, nq.FMT_INT4):
        pl = nq.pack_weights(torch.from_numpy(w).cuda(), fmt, g)
        torch.cuda.synchronize()
        base, resid, scales = O.pack_nested(w, g, with_resid=fmt == nq.FMT_NESTED44)
        assert np.array_equal(pl.base.cpu().numpy(), base.reshape(-1))
        assert np.array_equal(pl.scales.cpu().numpy().view(np.uint16), scales.reshape(-1))
        if fmt == nq.FMT_NESTED44:
            assert np.array_equal(pl.resid.cpu().numpy(), resid.reshape(-1))
        else:
            assert pl.resid is None


@pytest.mark.parametrize("n,k", [(300, 512), (64, 3584)])
def test_fp8_and_fp16_pack_bit_exact(nq, n, k):
    w = special_rows(synth.weights(600 + n, n, k))
    wd = torch.from_numpy(w).cuda()
    p8 = nq.pack_weights(wd, nq.FMT_FP8E4M3_ROW, 0)
    p16 = nq.pack_weights(wd, nq.FMT_FP16, 0)
    torch.cuda.synchronize()
    codes, scale = O.pack_fp8(w)
    assert np.array_equal(p8.base.cpu().numpy(), codes.reshape(-1))
    assert np.array_equal(p8.scales.cpu().numpy().view(np.float32), scale)
    assert np.array_equal(p16.base.cpu().numpy().view(np.uint16), O.pack_fp16(w).reshape(-1))


def test_e4m3_encoder_dense_sweep_matches_oracle(nq):
    # every fp32 bit pattern with a 13-bit stride over the E4M3 range, both signs
    u = np.arange(0, 0x43E00000 + 1, 8191, dtype=np.uint32)
    vals = u.view(np.float32)
    vals = np.concatenate([vals, -vals])
    w = np.zeros(((vals.size + 1023) // 1024, 1024), np.float32)
    w.reshape(-1)[:vals.size] = vals
    w[:, 0] = 448.0                              # row scale exactly 1 -> codes encode the values themselves
    p8 = nq.pack_weights(torch.from_numpy(w).cuda(), nq.FMT_FP8E4M3_ROW, 0)
    torch.cuda.synchronize()
    codes, scale = O.pack_fp8(w)
    assert np.all(scale == 1.0)
    assert np.array_equal(p8.base.cpu().numpy(), codes.reshape(-1))
