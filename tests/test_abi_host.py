"""The C-ABI library builds, loads and exports every symbol that include/nq.h
declares; host-side sizes and argument validation work without a GPU (every
call here is rejected before any CUDA call, and no pointer is dereferenced)."""
import ctypes as C
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "nq.h")


@pytest.fixture(scope="module")
def L():
    from quantized_self_speculative_gb300 import build, nq
    build.build()
    return nq.lib()


def declared_functions():
    src = open(HEADER).read()
    return re.findall(r"NQ_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    assert {"nq_pack_weights", "nq_draft_gemv", "nq_verify_gemm", "spec_accept_greedy",
            "spec_accept_sample"} <= names
    assert len(names) >= 11


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_packed_bytes(L):
    from quantized_self_speculative_gb300 import nq
    assert nq.packed_bytes(4096, 4096, 128, nq.FMT_NESTED44) == (4096 * 2048, 4096 * 2048, 4096 * 32 * 2)
    assert nq.packed_bytes(1024, 1024, 64, nq.FMT_INT4) == (1024 * 512, 0, 1024 * 16 * 2)
    assert nq.packed_bytes(512, 3584, 0, nq.FMT_FP8E4M3_ROW) == (512 * 3584, 0, 512 * 4)
    assert nq.packed_bytes(512, 3584, 0, nq.FMT_FP16) == (512 * 3584 * 2, 0, 0)
    for args, st in [((64, 96, 64, nq.FMT_NESTED44), nq.NQ_ERR_SHAPE),     # k % 64
                     ((64, 192, 128, nq.FMT_NESTED44), nq.NQ_ERR_SHAPE),   # k % group
                     ((64, 256, 96, nq.FMT_INT4), nq.NQ_ERR_SHAPE),        # group not 64/128
                     ((0, 256, 64, nq.FMT_INT4), nq.NQ_ERR_SHAPE),
                     ((64, 256, 64, 7), nq.NQ_ERR_ARG)]:
        with pytest.raises(nq.NQError) as e:
            nq.packed_bytes(*args)
        assert e.value.status == st


def test_workspace_bytes(L):
    from quantized_self_speculative_gb300 import nq
    # sections, each starting on a 256-byte boundary: two ticket arrays,
    # (2k+1) partials per row of max(4096-entry chunks, 2048-entry segment
    # pairs), a 32-B decision record per row, one maximum and one sum per
    # 1024-entry segment (16 per 16384-entry block) per vector per row, one sum per
    # segment per row, 64 leaf sums per segment per row; for the draft
    # features one u per partial
    a = lambda n: (n + 255) // 256 * 256

    def expect(B, k, V):
        C, NSP, NV = -(-V // 4096), 16 * -(-V // 16384), 2 * k + 1
        P = max(C, NSP // 2)
        return (a(4 * B) * 2 + a(B * NV * P * 8) + a(32 * B) + 2 * a(B * NV * NSP * 4)
                + a(4 * B * NSP) + a(256 * B * NSP) + 4 * B * NV * P)

    assert nq.workspace_bytes(64, 8, 152064) == expect(64, 8, 152064) == 5102080
    assert nq.workspace_bytes(1, 4, 4096) == expect(1, 4, 4096) == 7712
    assert nq.workspace_bytes(3, 16, 4099) == expect(3, 16, 4099)
    # k = 0 sizes the draft argmax's workspace (no drafts, one position per row)
    assert nq.workspace_bytes(5, 0, 32000) == expect(5, 0, 32000) > 0
    for bad in [(0, 4, 10), (1, -1, 10), (1, 17, 10), (1, 4, 0), (1, 4, 524289), (65536, 1, 1)]:
        assert nq.workspace_bytes(*bad) == 0


def test_linear_workspace_bytes(L):
    """Workspace of the tensor-core linears: fp16 activations of each layer
    (N padded to a multiple of 16, at most 256 rows per launch), 1024-byte
    regions, the largest launch of 64 layers; 0 where the path is not taken."""
    from quantized_self_speculative_gb300 import nq
    A = 0x10000
    a1k = lambda n: (n + 1023) // 1024 * 1024

    def layers(shapes, fmt=nq.FMT_NESTED44, g=128):
        return (nq.nq_weights * len(shapes))(*[nq.nq_weights(n, k, g, fmt, A, A, A) for n, k in shapes])

    one = layers([(4096, 4096)])
    assert L.nq_linear_workspace_bytes(1, one, 144, 1) == a1k(2 * 144 * 4096)
    assert L.nq_linear_workspace_bytes(1, one, 16, 0) == a1k(2 * 16 * 4096)
    assert L.nq_linear_workspace_bytes(1, one, 17, 1) == a1k(2 * 32 * 4096)
    assert L.nq_linear_workspace_bytes(1, one, 1000, 1) == a1k(2 * 256 * 4096)
    assert L.nq_linear_workspace_bytes(1, one, 15, 1) == 0                  # streaming kernel
    mix = layers([(1024, 4096), (4096, 14336), (333, 384)])
    assert L.nq_linear_workspace_bytes(3, mix, 40, 1) == sum(a1k(2 * 48 * k) for k in (4096, 14336, 384))
    many = layers([(512, 4096)] * 200)
    assert L.nq_linear_workspace_bytes(200, many, 64, 1) == 64 * a1k(2 * 64 * 4096)
    assert L.nq_linear_workspace_bytes(1, layers([(256, 192)], g=64), 64, 1) == 0   # k % 128 != 0
    assert L.nq_linear_workspace_bytes(1, layers([(256, 512)], fmt=nq.FMT_INT4), 64, 0) == a1k(2 * 64 * 512)
    assert L.nq_linear_workspace_bytes(1, layers([(256, 512)], fmt=nq.FMT_INT4), 64, 1) == 0   # invalid pair
    assert L.nq_linear_workspace_bytes(1, layers([(256, 512)], fmt=nq.FMT_FP16, g=0), 64, 1) == 0
    # a missing or short workspace is rejected before any launch
    ptrs = (C.c_void_p * 1)(A)
    need = L.nq_linear_workspace_bytes(1, one, 144, 1)
    assert L.nq_verify_gemm_batch_ws(1, one, ptrs, 144, ptrs, None, need, None) == nq.NQ_ERR_WORKSPACE
    assert L.nq_verify_gemm_batch_ws(1, one, ptrs, 144, ptrs, A, need - 16, None) == nq.NQ_ERR_WORKSPACE
    assert L.nq_verify_gemm_batch_ws(1, one, ptrs, 144, ptrs, A + 8, need, None) == nq.NQ_ERR_ALIGN
    assert L.nq_draft_gemv_batch_ws(1, one, ptrs, 0, ptrs, A, need, None) == nq.NQ_ERR_ARG


def test_status_strings(L):
    from quantized_self_speculative_gb300 import nq
    assert nq.status_string(0) == "NQ_OK"
    assert "WORKSPACE" in nq.status_string(nq.NQ_ERR_WORKSPACE)
    assert nq.status_string(99) == "unknown nq_status"


def test_host_validation_rejects_before_launch(L):
    from quantized_self_speculative_gb300 import nq
    A = 0x10000            # fake, 16-byte aligned device addresses: never dereferenced
    W = nq.nq_weights(256, 512, 128, nq.FMT_NESTED44, A, A + 0x100000, A + 0x200000)
    assert L.nq_draft_gemv(None, A, 1, A, None) == nq.NQ_ERR_ARG
    assert L.nq_draft_gemv(C.byref(W), A, 0, A, None) == nq.NQ_ERR_ARG           # M = 0
    assert L.nq_draft_gemv(C.byref(W), A + 2, 1, A, None) == nq.NQ_ERR_ALIGN      # x misaligned
    bad = nq.nq_weights(256, 512, 128, nq.FMT_NESTED44, A + 8, A, A)
    assert L.nq_verify_gemm(C.byref(bad), A, 1, A, None) == nq.NQ_ERR_ALIGN
    i4 = nq.nq_weights(256, 512, 128, nq.FMT_INT4, A, None, A)
    assert L.nq_verify_gemm(C.byref(i4), A, 1, A, None) == nq.NQ_ERR_ARG        # INT4 is draft-only
    f16 = nq.nq_weights(256, 512, 0, nq.FMT_FP16, A, None, None)
    assert L.nq_draft_gemv(C.byref(f16), A, 1, A, None) == nq.NQ_ERR_ARG        # FP16 is verify-only
    g96 = nq.nq_weights(256, 576, 96, nq.FMT_NESTED44, A, A, A)
    assert L.nq_draft_gemv(C.byref(g96), A, 1, A, None) == nq.NQ_ERR_SHAPE
    nores = nq.nq_weights(256, 512, 128, nq.FMT_NESTED44, A, None, A)
    assert L.nq_verify_gemm(C.byref(nores), A, 1, A, None) == nq.NQ_ERR_ARG
    # batch: layers of different kernel families in one call are rejected
    ws = (nq.nq_weights * 2)(W, nq.nq_weights(256, 512, 64, nq.FMT_NESTED44, A, A, A))
    ptrs = (C.c_void_p * 2)(A, A)
    assert L.nq_draft_gemv_batch(2, ws, ptrs, 1, ptrs, None) == nq.NQ_ERR_ARG
    assert L.nq_draft_gemv_batch(0, ws, ptrs, 1, ptrs, None) == nq.NQ_ERR_ARG
    # acceptance
    need = nq.workspace_bytes(4, 4, 5000)
    assert L.spec_accept_greedy(A, A, 4, 0, 5000, A, A, A, need, None) == nq.NQ_ERR_ARG        # k = 0
    assert L.spec_accept_greedy(A, A, 4, 4, 5000, A, A, A + 4, need, None) == nq.NQ_ERR_ALIGN  # ws
    assert L.spec_accept_greedy(A, A, 4, 4, 5000, A, A, A, need - 1, None) == nq.NQ_ERR_WORKSPACE
    assert L.spec_accept_greedy(A, A, 4, 4, 5000, A, A, None, need, None) == nq.NQ_ERR_ARG
    assert L.spec_accept_sample(A, A, A, 4, 4, 5000, 0.0, A, 0, A, A, A, need, None) == nq.NQ_ERR_ARG
    assert L.spec_accept_sample(A, A, A, 4, 4, 5000, float("nan"), A, 0, A, A, A, need, None) == nq.NQ_ERR_ARG
    assert L.spec_accept_sample(A, A + 4, A, 4, 4, 5000, 1.0, A, 0, A, A, A, need, None) == nq.NQ_ERR_ALIGN
    assert L.nq_pack_weights(None, C.byref(W), None) == nq.NQ_ERR_ARG
    assert L.nq_pack_weights(A + 4, C.byref(W), None) == nq.NQ_ERR_ALIGN
    assert L.nq_get_device_status(None, None) == nq.NQ_ERR_ARG
    L.nq_selftest_bounded_wait.argtypes = [C.c_uint32, C.c_void_p]
    assert L.nq_selftest_bounded_wait(0, None) == nq.NQ_ERR_ARG
    assert L.nq_selftest_bounded_wait(1000001, None) == nq.NQ_ERR_ARG


def test_product_and_oracle_share_nothing():
    """The CUDA path never imports / links the oracle, and vice versa."""
    pkg = os.path.join(ROOT, "quantized_self_speculative_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b|nq_oracle|libnq_oracle", src, re.M), f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c", ".h")):
            src = open(os.path.join(ROOT, "oracle", f)).read()
            assert not re.search(r"^\s*(import|from)\s+quantized_self_speculative_gb300|nq_internal|libnq\.so|nq\.h",
                                 src, re.M), f


def test_round_kv_and_int8_entry_points_validate_on_the_host(L):
    """Sizes of the nested KV cache and the attention workspace, and argument
    checks of the round bookkeeping, KV and int8-activation entry points: every
    call here is rejected before any CUDA call."""
    from quantized_self_speculative_gb300 import nq
    A = 0x10000
    pb, sb = C.c_size_t(), C.c_size_t()
    assert L.nq_kv_cache_bytes(2, 4, 128, 64, 1000, C.byref(pb), C.byref(sb)) == nq.NQ_OK
    assert pb.value == 2 * 4 * 1000 * 64 and sb.value == 2 * 4 * 1000 * 2 * 2      # planes of d/2, two scales a row
    assert L.nq_kv_cache_bytes(1, 1, 96, 64, 10, None, None) == nq.NQ_ERR_SHAPE      # head_dim 64 or 128
    assert L.nq_kv_cache_bytes(1, 1, 64, 128, 10, None, None) == nq.NQ_ERR_SHAPE     # group > head_dim
    assert L.nq_kv_cache_bytes(0, 1, 64, 64, 10, None, None) == nq.NQ_ERR_ARG
    # one (output, max, sum) record per (sequence, query row, query head, 256-row split)
    assert L.nq_attn_workspace_bytes(2, 5, 8, 128, 1000) == 2 * 5 * 8 * 4 * 130 * 4
    assert L.nq_attn_workspace_bytes(1, 1, 1, 96, 10) == 0
    cache = nq.nq_kv_cache(1, 2, 128, 128, 512, 0, A, A, A, A, A, A)
    need = L.nq_attn_workspace_bytes(1, 5, 4, 128, 512)
    assert L.nq_attn_decode(C.byref(cache), A, 5, 4, A, 3, 0.1, A, A, need, None) == nq.NQ_ERR_ARG      # planes
    assert L.nq_attn_decode(C.byref(cache), A, 5, 3, A, 2, 0.1, A, A, need, None) == nq.NQ_ERR_ARG      # heads ratio
    assert L.nq_attn_decode(C.byref(cache), A + 4, 5, 4, A, 2, 0.1, A, A, need, None) == nq.NQ_ERR_ALIGN
    assert L.nq_attn_decode(C.byref(cache), A, 5, 4, A, 2, 0.1, A, A, need - 4, None) == nq.NQ_ERR_WORKSPACE
    assert L.nq_attn_decode(C.byref(cache), A, 5, 4, A, 2, 0.0, A, A, need, None) == nq.NQ_ERR_ARG      # scale
    assert L.nq_kv_append(C.byref(cache), A, A, 0, A, None) == nq.NQ_ERR_ARG                           # n_new
    assert L.nq_kv_append(C.byref(cache), A + 4, A, 1, A, None) == nq.NQ_ERR_ALIGN
    odd = nq.nq_kv_cache(1, 2, 128, 128, 512, 0, A + 8, A, A, A, A, A)
    assert L.nq_kv_append(C.byref(odd), A, A, 1, A, None) == nq.NQ_ERR_ALIGN
    # int8 activations
    assert L.nq_quantize_act_int8(A, 0, 64, A, A, None) == nq.NQ_ERR_ARG
    assert L.nq_quantize_act_int8(A + 2, 1, 64, A, A, None) == nq.NQ_ERR_ALIGN
    W = nq.nq_weights(256, 512, 128, nq.FMT_NESTED44, A, A, A)
    ptrs = (C.c_void_p * 1)(A)
    assert L.nq_linear_a8_batch(0, C.byref(W), ptrs, ptrs, 1, 1, ptrs, None) == nq.NQ_ERR_ARG
    f8 = nq.nq_weights(256, 512, 0, nq.FMT_FP8E4M3_ROW, A, None, A)
    assert L.nq_linear_a8_batch(1, C.byref(f8), ptrs, ptrs, 1, 1, ptrs, None) == nq.NQ_ERR_ARG        # nested planes only
    i4 = nq.nq_weights(256, 512, 128, nq.FMT_INT4, A, None, A)
    assert L.nq_linear_a8_batch(1, C.byref(i4), ptrs, ptrs, 1, 1, ptrs, None) == nq.NQ_ERR_ARG        # INT4 verify
    bad = (C.c_void_p * 1)(A + 4)
    assert L.nq_linear_a8_batch(1, C.byref(W), bad, ptrs, 1, 1, ptrs, None) == nq.NQ_ERR_ALIGN
    # round bookkeeping
    assert L.nq_embed_rows(A, 100, 12, A, 1, 1, A, None) == nq.NQ_ERR_ARG                              # d % 8
    assert L.nq_embed_rows(A + 2, 100, 16, A, 1, 1, A, None) == nq.NQ_ERR_ALIGN
    assert L.spec_round_commit(A, A, 0, 4, A, A, 10, A, None) == nq.NQ_ERR_ARG
    assert L.spec_round_commit(A, A, 2, 4, A + 2, A, 10, A, None) == nq.NQ_ERR_ALIGN
