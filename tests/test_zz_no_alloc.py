"""Allocation-free greedy acceptance (spec_accept_greedy_noalloc).

Some callers cannot allocate device memory where they decide tokens -- their
device memory belongs to another component (a serving runtime with a fixed
budget), or an allocation must not fail or block inside the decode loop.  The
entry point keeps its scratch in a fixed array inside the library; these
tests call it through the C ABI and check that two calls in a row give
exactly the token ids and counts of spec_accept_greedy (integer outputs:
the tolerance is zero).  Collected last on purpose.
"""
import ctypes as C

import numpy as np
import pytest
import torch

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
    return torch.from_numpy(d).cuda(), torch.from_numpy(tl).cuda()


@pytest.mark.parametrize("B,k,V", [(64, 8, 152064), (5, 4, 4099), (256, 4, 4096)])
def test_noalloc_matches_workspace_call_twice(nq, B, k, V):
    f = noalloc(nq)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        d, tl = inputs(B, k, V, 9500 + 10 * call + B)
        ref_out, ref_cnt = nq.accept_greedy(d, tl)
        out = torch.full((B, k + 1), -7, dtype=torch.int32, device="cuda")
        cnt = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        st = f(d.data_ptr(), tl.data_ptr(), B, k, V, out.data_ptr(), cnt.data_ptr(), stream)
        assert st == nq.NQ_OK, nq.status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(cnt.cpu(), ref_cnt.cpu())
        assert torch.equal(out.cpu(), ref_out.cpu())


def test_noalloc_rejects_sizes_beyond_its_scratch(nq):
    f = noalloc(nq)
    A = 0x10000   # never dereferenced: the call is rejected on the host
    assert f(A, A, 2000, 16, 524288, A, A, None) == nq.NQ_ERR_WORKSPACE
    assert f(A, A, 4, 0, 100, A, A, None) == nq.NQ_ERR_ARG
