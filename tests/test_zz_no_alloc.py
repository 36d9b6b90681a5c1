"""Allocation-free greedy acceptance (spec_accept_greedy_noalloc).

Some callers cannot allocate device memory where they decide tokens -- their
device memory belongs to another component (a serving runtime with a fixed
budget), or an allocation must not fail or block inside the decode loop.  The
entry point keeps its scratch in a fixed array inside the library; these
tests call it through the C ABI and check that two calls in a row give
exactly the token ids and counts of spec_accept_greedy and of the CPU oracle
(integer outputs: the tolerance is zero).  Collected last on purpose.
"""
import ctypes as C

import math

import numpy as np
import pytest
import torch

import oracle as O
from quantized_self_speculative_gb300 import synth

pytestmark = pytest.mark.gpu


def noalloc(nq):
    f = nq.lib().spec_accept_greedy_noalloc
    f.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p]
    f.restype = C.c_int
    return f


def inputs(B, k, V, seed):
    tl = synth.target_logits(seed, B, k, V, 2.0)
    dl = synth.draft_logits_from(tl, seed + 1, 0.5)
    d = synth.draft_tokens_greedy(dl)
    return d, tl


def scratch_need(B, k, V):
    """Bytes of the fixed scratch a call uses: the row tickets, then one
    (value, index) partial per row, position and 16384-entry chunk."""
    return 256 * math.ceil(4 * B / 256) + B * (k + 1) * math.ceil(V / 16384) * 8


def call_twice(nq, B, k, V, make):
    f = noalloc(nq)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        d, tl = make(9500 + 10 * call + B)
        ref_out, ref_cnt = nq.accept_greedy(d, tl)
        out = torch.full((B, k + 1), -7, dtype=torch.int32, device="cuda")
        cnt = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        st = f(d.data_ptr(), tl.data_ptr(), B, k, V, out.data_ptr(), cnt.data_ptr(), stream)
        assert st == nq.NQ_OK, nq.status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(cnt.cpu(), ref_cnt.cpu())
        assert torch.equal(out.cpu(), ref_out.cpu())
        yield d, tl, out, cnt


@pytest.mark.parametrize("B,k,V", [(64, 8, 152064), (5, 4, 4099), (256, 4, 4096)])
def test_noalloc_matches_workspace_call_and_oracle_twice(nq, B, k, V):
    def make(seed):
        d, tl = inputs(B, k, V, seed)
        return torch.from_numpy(d).cuda(), torch.from_numpy(tl).cuda()
    for d, tl, out, cnt in call_twice(nq, B, k, V, make):
        orc_out, orc_cnt = O.accept_greedy(d.cpu().numpy(), tl.cpu().numpy())
        assert np.array_equal(cnt.cpu().numpy(), orc_cnt)
        assert np.array_equal(out.cpu().numpy(), orc_out)


def test_noalloc_at_the_scratch_limit(nq):
    """The largest batch whose partials fit the 1 MiB scratch at k = 8,
    V = 163840 (1,048,448 bytes; counting 4096-entry chunks instead of the
    16384-entry chunks the kernel writes would ask for four times that).  The
    8.5 GB of logits are drawn on the GPU; the reference is spec_accept_greedy."""
    B, k, V = 1448, 8, 163840
    assert scratch_need(B, k, V) <= 1 << 20 < scratch_need(B + 1, k, V)

    def make(seed):
        g = torch.Generator(device="cuda")
        g.manual_seed(seed)
        tl = torch.randn((B, k + 1, V), generator=g, device="cuda").mul_(2.0)
        d = (tl[:, :k] + 0.5 * torch.randn((B, k, V), generator=g, device="cuda")).argmax(-1).to(torch.int32)
        return d.contiguous(), tl
    for _ in call_twice(nq, B, k, V, make):
        pass
    torch.cuda.empty_cache()


def test_noalloc_rejects_sizes_beyond_its_scratch(nq):
    f = noalloc(nq)
    A = 0x10000   # never dereferenced: the call is rejected on the host
    assert f(A, A, 2000, 16, 524288, A, A, None) == nq.NQ_ERR_WORKSPACE
    assert scratch_need(1449, 8, 163840) > 1 << 20          # just beyond the scratch
    assert f(A, A, 1449, 8, 163840, A, A, None) == nq.NQ_ERR_WORKSPACE
    assert f(A, A, 4, 0, 100, A, A, None) == nq.NQ_ERR_ARG
