"""CPU oracle for the quantized self-speculative hot path -- TEST INFRASTRUCTURE.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline / reference leg
of `bench.py` may import this package.  The product path
(`quantized_self_speculative_gb300`) never does, and this package never
imports the product.  The arithmetic lives in `nq_oracle.c` (plain C, no SIMD,
no BLAS, `-ffp-contract=off`); this module only marshals numpy arrays.

Every routine cites the passage it follows in `nq_oracle.c`.  All functions
are pinned by `-m "not gpu"` tests (tests/test_oracle_*.py); none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nq_oracle.c")
_HDR = os.path.join(_HERE, "nq_oracle.h")
_LIB = os.path.join(_HERE, "libnq_oracle.so")
_lock = threading.Lock()
_lib = None

FMT_NESTED44, FMT_INT4, FMT_FP8, FMT_FP16 = 0, 1, 2, 3
LEAF = 16

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-Wall", "-shared", "-fPIC"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (seconds).  Returns the library path."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Weights(C.Structure):
    _fields_ = [("n", C.c_int32), ("k", C.c_int32), ("group", C.c_int32), ("format", C.c_int32),
                ("base", C.c_void_p), ("resid", C.c_void_p), ("scales", C.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = C.CDLL(build())
            L = _lib
            vp, i32, u64, f32 = C.c_void_p, C.c_int, C.c_uint64, C.c_float
            L.orc_pack_nested.argtypes = [vp, i32, i32, i32, vp, vp, vp]
            L.orc_pack_fp8.argtypes = [vp, i32, i32, vp, vp]
            L.orc_pack_fp16.argtypes = [vp, i32, i32, vp]
            L.orc_linear.argtypes = [C.POINTER(_Weights), i32, vp, i32, vp, i32, vp]
            L.orc_accept_greedy.argtypes = [vp, vp, i32, i32, i32, vp, vp]
            L.orc_accept_sample.argtypes = [vp, vp, vp, i32, i32, i32, f32, vp, u64, vp, vp]
            L.orc_accept_sample_f64.argtypes = [vp, vp, vp, i32, i32, i32, f32, vp, u64, vp, vp, vp]
            L.orc_philox4x32_10.argtypes = [vp, vp, vp]
            L.orc_uniform.argtypes = [u64, C.c_uint32, C.c_uint32, u64]
            L.orc_uniform.restype = f32
            L.orc_uniform_n.argtypes = [vp, vp, vp, vp, vp, i32]
            L.orc_exp2c.argtypes = [f32]
            L.orc_exp2c.restype = f32
            L.orc_exp2_coef.argtypes = [i32]
            L.orc_exp2_coef.restype = f32
            L.orc_temper_coef.argtypes = [f32]
            L.orc_temper_coef.restype = f32
            L.orc_exp2c_n.argtypes = [vp, vp, i32]
            L.orc_softmax_canonical.argtypes = [vp, i32, f32, vp]
            L.orc_tree_sample.argtypes = [vp, i32, f32]
            L.orc_softmax_stats.argtypes = [vp, i32, f32, vp, vp, vp, vp]
            L.orc_draft_argmax.argtypes = [vp, i32, i32, vp]
            L.orc_sample_p.argtypes = [vp, i32, f32, f32]
            L.orc_draft_features.argtypes = [vp, vp, i32, i32, i32, f32, vp]
            L.orc_quantize_act_int8.argtypes = [vp, i32, i32, vp, vp]
            L.orc_linear_a8.argtypes = [C.POINTER(_Weights), i32, vp, vp, i32, vp]
            L.orc_attn_decode.argtypes = [vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, i32, f32, vp]
            L.orc_round_commit.argtypes = [vp, vp, i32, i32, vp, vp, i32, vp]
            L.orc_f32_to_f16_n.argtypes = [vp, vp, i32]
            L.orc_f16_to_f32_n.argtypes = [vp, vp, i32]
            L.orc_f32_to_e4m3_n.argtypes = [vp, vp, i32]
            L.orc_e4m3_to_f32_n.argtypes = [vp, vp, i32]
            L.orc_nibble_value.argtypes = [C.c_uint]
            L.orc_quantise_weight.argtypes = [f32, f32, C.POINTER(C.c_int), C.POINTER(C.c_int)]
        return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(C.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its input (rc={rc})")


# ---------------------------------------------------------------- formats
def f32_to_f16_bits(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.empty(x.size, np.uint16)
    lib().orc_f32_to_f16_n(_p(x), _p(out), x.size)
    return out


def f16_bits_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16).ravel()
    out = np.empty(h.size, np.float32)
    lib().orc_f16_to_f32_n(_p(h), _p(out), h.size)
    return out


def f32_to_e4m3(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.empty(x.size, np.uint8)
    lib().orc_f32_to_e4m3_n(_p(x), _p(out), x.size)
    return out


def e4m3_to_f32(c) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.uint8).ravel()
    out = np.empty(c.size, np.float32)
    lib().orc_e4m3_to_f32_n(_p(c), _p(out), c.size)
    return out


def nibble_value(nib: int) -> int:
    return lib().orc_nibble_value(nib)


def quantise_weight(w: float, s: float):
    q4, r = C.c_int(), C.c_int()
    lib().orc_quantise_weight(w, s, C.byref(q4), C.byref(r))
    return q4.value, r.value


# ---------------------------------------------------------------- C1 pack
def pack_nested(w: np.ndarray, group: int, with_resid: bool = True):
    """W fp32 [n][k] -> (base u8 [n][k/2], resid u8 [n][k/2] | None, scales fp16-bits [n][k/g])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    base = np.zeros((n, k // 2), np.uint8)
    resid = np.zeros((n, k // 2), np.uint8) if with_resid else None
    scales = np.zeros((n, k // group), np.uint16)
    rc = lib().orc_pack_nested(_p(w), n, k, group, _p(base), _p(resid) if with_resid else None, _p(scales))
    _check(rc, "pack_nested")
    return base, resid, scales


def pack_fp8(w: np.ndarray):
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    codes = np.zeros((n, k), np.uint8)
    scale = np.zeros(n, np.float32)
    _check(lib().orc_pack_fp8(_p(w), n, k, _p(codes), _p(scale)), "pack_fp8")
    return codes, scale


def pack_fp16(w: np.ndarray):
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    out = np.zeros((n, k), np.uint16)
    _check(lib().orc_pack_fp16(_p(w), n, k, _p(out)), "pack_fp16")
    return out


# ---------------------------------------------------------------- C2 linear
def linear(fmt: int, n: int, k: int, group: int, base, resid, scales, x_bf16: np.ndarray,
           use_resid: bool, rows=None) -> np.ndarray:
    """fp64 y [M][len(rows) or n] of the dequantised linear (draft: base only;
    verify: both planes)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M = x.shape[0]
    assert x.shape[1] == k
    base = np.ascontiguousarray(base)
    resid = None if resid is None else np.ascontiguousarray(resid)
    scales = None if scales is None else np.ascontiguousarray(scales)
    W = _Weights(n, k, group, fmt, base.ctypes.data,
                 None if resid is None else resid.ctypes.data,
                 None if scales is None else scales.ctypes.data)
    if rows is None:
        y = np.zeros((M, n), np.float64)
        rc = lib().orc_linear(C.byref(W), int(use_resid), _p(x), M, None, 0, _p(y))
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int32)
        y = np.zeros((M, rows.size), np.float64)
        rc = lib().orc_linear(C.byref(W), int(use_resid), _p(x), M, _p(rows), rows.size, _p(y))
    _check(rc, "linear")
    return y


# ---------------------------------------------------------------- C3 greedy
def accept_greedy(draft: np.ndarray, tgt_logits: np.ndarray):
    draft = np.ascontiguousarray(draft, dtype=np.int32)
    tl = np.ascontiguousarray(tgt_logits, dtype=np.float32)
    B, k = draft.shape
    V = tl.shape[-1]
    assert tl.shape == (B, k + 1, V)
    out = np.zeros((B, k + 1), np.int32)
    cnt = np.zeros(B, np.int32)
    _check(lib().orc_accept_greedy(_p(draft), _p(tl), B, k, V, _p(out), _p(cnt)), "accept_greedy")
    return out, cnt


# ---------------------------------------------------------------- C4 sampled
def _sample_args(draft, draft_logits, tgt_logits, seeds):
    draft = np.ascontiguousarray(draft, dtype=np.int32)
    dl = np.ascontiguousarray(draft_logits, dtype=np.float32)
    tl = np.ascontiguousarray(tgt_logits, dtype=np.float32)
    seeds = np.ascontiguousarray(seeds, dtype=np.uint64)
    B, k = draft.shape
    V = tl.shape[-1]
    assert dl.shape == (B, k, V) and tl.shape == (B, k + 1, V) and seeds.shape == (B,)
    return draft, dl, tl, seeds, B, k, V


def accept_sample(draft, draft_logits, tgt_logits, temperature: float, seeds, round_: int):
    draft, dl, tl, seeds, B, k, V = _sample_args(draft, draft_logits, tgt_logits, seeds)
    out = np.zeros((B, k + 1), np.int32)
    cnt = np.zeros(B, np.int32)
    rc = lib().orc_accept_sample(_p(draft), _p(dl), _p(tl), B, k, V, float(temperature), _p(seeds),
                                 int(round_), _p(out), _p(cnt))
    _check(rc, "accept_sample")
    return out, cnt


def accept_sample_f64(draft, draft_logits, tgt_logits, temperature: float, seeds, round_: int):
    draft, dl, tl, seeds, B, k, V = _sample_args(draft, draft_logits, tgt_logits, seeds)
    out = np.zeros((B, k + 1), np.int32)
    cnt = np.zeros(B, np.int32)
    margin = np.zeros(B, np.float64)
    lib().orc_accept_sample_f64(_p(draft), _p(dl), _p(tl), B, k, V, float(temperature), _p(seeds),
                                int(round_), _p(out), _p(cnt), _p(margin))
    return out, cnt, margin


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    kk = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, np.uint32)
    lib().orc_philox4x32_10(_p(c), _p(kk), _p(out))
    return out


def uniform(seed: int, j: int, purpose: int, round_: int) -> float:
    return lib().orc_uniform(seed, j, purpose, round_)


def uniforms(seed, j, purpose, round_) -> np.ndarray:
    seed, j, purpose, round_ = np.broadcast_arrays(np.asarray(seed, np.uint64), np.asarray(j, np.uint32),
                                                   np.asarray(purpose, np.uint32), np.asarray(round_, np.uint64))
    seed, j, purpose, round_ = (np.ascontiguousarray(a.ravel()) for a in (seed, j, purpose, round_))
    out = np.zeros(seed.size, np.float32)
    lib().orc_uniform_n(_p(seed), _p(j), _p(purpose), _p(round_), _p(out), seed.size)
    return out


def exp2c(t) -> np.ndarray:
    t = np.ascontiguousarray(t, dtype=np.float32).ravel()
    out = np.empty(t.size, np.float32)
    lib().orc_exp2c_n(_p(t), _p(out), t.size)
    return out


def exp2_coef(i: int) -> float:
    return lib().orc_exp2_coef(i)


def temper_coef(T: float) -> float:
    return lib().orc_temper_coef(T)


def softmax_canonical(logits, temperature: float = 1.0) -> np.ndarray:
    l = np.ascontiguousarray(logits, dtype=np.float32).ravel()
    p = np.zeros(l.size, np.float32)
    _check(lib().orc_softmax_canonical(_p(l), l.size, float(temperature), _p(p)), "softmax_canonical")
    return p


def tree_sample(w, u: float) -> int:
    w = np.ascontiguousarray(w, dtype=np.float32).ravel()
    return lib().orc_tree_sample(_p(w), w.size, float(u))


def softmax_stats(logits, temperature: float = 1.0):
    """Intermediate values of the canonical recipe for one logits vector:
    per 1024-entry segment (mz, s) and the root (M, S) of the (max, sum) tree."""
    l = np.ascontiguousarray(logits, dtype=np.float32)
    V = l.shape[0]
    ns = -(-V // 1024)
    mz, s = np.empty(ns, np.float32), np.empty(ns, np.float32)
    M, S = C.c_float(), C.c_float()
    if lib().orc_softmax_stats(l.ctypes.data, V, float(temperature), mz.ctypes.data, s.ctypes.data,
                               C.byref(M), C.byref(S)) < 0:
        raise ValueError("non-finite logits")
    return mz, s, np.float32(M.value), np.float32(S.value)


# ------------------------------------------------------------------ round bookkeeping
# "How Speculative Decoding Speeds Up Inference", "Drafting and checking
# tokens"; BitNest Fig. 4 (the rejected suffix's cache entries are dropped).

def draft_argmax(logits):
    """The draft's greedy choice per row of logits [M][V] (lowest index on ties)."""
    l = np.ascontiguousarray(logits, dtype=np.float32)
    M, V = l.shape
    tok = np.empty(M, np.int32)
    if lib().orc_draft_argmax(l.ctypes.data, M, V, tok.ctypes.data) < 0:
        raise ValueError("non-finite logits")
    return tok


def round_commit(out_tok, out_cnt, seq, seq_len, x0):
    """Append the emitted tokens; returns (seq, seq_len, x0, rc) updated copies
    (rc 1: a sequence ran out of room, -1: a count outside 1..k+1)."""
    out_tok = np.ascontiguousarray(out_tok, dtype=np.int32)
    out_cnt = np.ascontiguousarray(out_cnt, dtype=np.int32)
    B, k1 = out_tok.shape
    seq = np.array(seq, dtype=np.int32, copy=True)
    seq_len = np.array(seq_len, dtype=np.int32, copy=True)
    x0 = np.array(x0, dtype=np.int32, copy=True)
    rc = lib().orc_round_commit(out_tok.ctypes.data, out_cnt.ctypes.data, B, k1 - 1, seq.ctypes.data,
                                seq_len.ctypes.data, seq.shape[1], x0.ctypes.data)
    return seq, seq_len, x0, rc


def embed_rows(table, ids):
    """Rows of table [V][d] (bf16 bits) for the token ids; a plain gather."""
    return np.ascontiguousarray(np.asarray(table)[np.asarray(ids, dtype=np.int64)])


def embed_round(table, x0, draft):
    """The verify pass's rows per sequence: x0[b], then draft[b][0..k-1]."""
    ids = np.concatenate([np.asarray(x0, np.int64)[:, None], np.asarray(draft, np.int64)], axis=1)
    return embed_rows(table, ids.reshape(-1))


def sample_p(logits, temperature: float, u: float) -> int:
    """A draw from the canonical p of one logits vector with uniform u (the
    bonus draw's two-level rule: segment weights, then the segment's leaves)."""
    l = np.ascontiguousarray(logits, dtype=np.float32)
    r = lib().orc_sample_p(l.ctypes.data, l.shape[0], float(temperature), float(u))
    if r < 0:
        raise ValueError("non-finite logits")
    return r


def draft_features(draft, draft_logits, temperature: float = 1.0):
    """SpecKV's per-step draft features for each row: (mean entropy, mean
    confidence, max entropy, min confidence) over the k drafted positions,
    entropy in nats of softmax(draft_logits / T), confidence = the drafted
    token's draft probability.  fp64 [B][4]."""
    d = np.ascontiguousarray(draft, dtype=np.int32)
    dl = np.ascontiguousarray(draft_logits, dtype=np.float32)
    B, k, V = dl.shape
    out = np.empty((B, 4), np.float64)
    if lib().orc_draft_features(d.ctypes.data, dl.ctypes.data, B, k, V, float(temperature), out.ctypes.data) < 0:
        raise ValueError("invalid draft tokens, logits or temperature")
    return out


# ------------------------------------------------------------------ nested KV cache
# BitNest Fig. 4: the draft reads the low-bit base view of the cache, the
# verification pass the full view.  Rows are quantised like NESTED44 weight
# rows (pack_nested over head_dim, groups of G).

def kv_rows_pack(rows, group: int):
    """Quantise K or V rows fp32 [..., d] like NESTED44 weight rows: returns
    (base, resid, scales) with the leading shape kept."""
    r = np.ascontiguousarray(rows, dtype=np.float32)
    lead, d = r.shape[:-1], r.shape[-1]
    base, resid, scales = pack_nested(r.reshape(-1, d), group)
    return (base.reshape(*lead, d // 2), resid.reshape(*lead, d // 2), scales.reshape(*lead, d // group))


def attn_decode(q, cache, lens, planes: int, scale: float):
    """fp64 attention of q [B][M][Hq][d] over the cache dict {k_base, k_resid,
    k_scales, v_base, v_resid, v_scales} ([B][Hkv][L][...] arrays, scales as
    fp16 bits) with lengths lens [B]; returns fp32 [B][M][Hq][d]."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    B, M, Hq, d = q.shape
    kb = np.ascontiguousarray(cache["k_base"], dtype=np.uint8)
    Hkv, L = kb.shape[1], kb.shape[2]
    G = d // cache["k_scales"].shape[-1]
    arrs = [np.ascontiguousarray(cache[n]) for n in ("k_resid", "k_scales", "v_base", "v_resid", "v_scales")]
    arrs[1] = arrs[1].view(np.uint16)
    arrs[4] = arrs[4].view(np.uint16)
    ln = np.ascontiguousarray(lens, dtype=np.int32)
    out = np.empty_like(q)
    if lib().orc_attn_decode(q.ctypes.data, B, M, Hq, Hkv, d, G, L, kb.ctypes.data, arrs[0].ctypes.data,
                             arrs[1].ctypes.data, arrs[2].ctypes.data, arrs[3].ctypes.data, arrs[4].ctypes.data,
                             ln.ctypes.data, int(planes), float(scale), out.ctypes.data) < 0:
        raise ValueError("bad attention arguments")
    return out


# ------------------------------------------------------------------ W8A8 (int8 activations)
# BitNest Table 1 "W4A8 -> W8A8" and Table 12: the draft multiplies 4-bit base
# codes, the target the 8-bit codes, both against int8 activations.

def quantize_act_int8(x_bf16):
    """bf16 bits [M][K] -> (int8 codes [M][K], fp32 row scales [M]):
    s = fp32(absmax / 127), code = clamp(rint(x / s), -127, 127)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, K = x.shape
    xq = np.empty((M, K), np.int8)
    sx = np.empty(M, np.float32)
    if lib().orc_quantize_act_int8(x.ctypes.data, M, K, xq.ctypes.data, sx.ctypes.data) < 0:
        raise ValueError("non-finite activation")
    return xq, sx


def linear_a8(fmt: int, n: int, k: int, group: int, base, resid, scales, xq, sx, verify: bool):
    """W8A8 / W4A8 linear: exact integer group dots, fp64 scaling -> fp64 [M][n]."""
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    sx = np.ascontiguousarray(sx, dtype=np.float32)
    M = xq.shape[0]
    base = np.ascontiguousarray(base)
    resid = None if resid is None else np.ascontiguousarray(resid)
    scales = np.ascontiguousarray(scales)
    W = _Weights(n, k, group, fmt, _p(base), _p(resid) if resid is not None else None, _p(scales))
    y = np.empty((M, n), np.float64)
    if lib().orc_linear_a8(C.byref(W), int(verify), xq.ctypes.data, sx.ctypes.data, M, y.ctypes.data) < 0:
        raise ValueError("bad format for an int8-activation linear")
    return y
