"""Thin ctypes binding of libnq.so (include/nq.h).  Argument marshalling only:
every step of the hot path runs in the library's CUDA kernels.  PyTorch
provides device memory and the current stream.

The library must have been built (``quantized_self_speculative_gb300.build``);
there is no fallback: a missing library raises immediately.
"""
from __future__ import annotations

import ctypes as C
import os
import threading
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnq.so")

NQ_OK, NQ_ERR_ARG, NQ_ERR_SHAPE, NQ_ERR_ALIGN, NQ_ERR_CUDA = 0, 1, 2, 3, 4
NQ_ERR_NONFINITE, NQ_ERR_TIMEOUT, NQ_ERR_WORKSPACE, NQ_ERR_TOKEN = 5, 6, 7, 8
NQ_DEV_NONFINITE, NQ_DEV_BAD_TOKEN, NQ_DEV_TIMEOUT, NQ_DEV_ACT_RANGE, NQ_DEV_SEQ_FULL = 0x1, 0x2, 0x4, 0x8, 0x10
FMT_NESTED44, FMT_INT4, FMT_FP8E4M3_ROW, FMT_FP16 = 0, 1, 2, 3

_lock = threading.Lock()
_lib = None


class NQError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


class nq_weights(C.Structure):
    _fields_ = [("n_out", C.c_int32), ("k_in", C.c_int32), ("group", C.c_int32), ("format", C.c_int32),
                ("base", C.c_void_p), ("resid", C.c_void_p), ("scales", C.c_void_p)]


class nq_kv_cache(C.Structure):
    _fields_ = [("batch", C.c_int32), ("heads_kv", C.c_int32), ("head_dim", C.c_int32), ("group", C.c_int32),
                ("max_len", C.c_int32), ("pad", C.c_int32),
                ("k_base", C.c_void_p), ("k_resid", C.c_void_p), ("k_scales", C.c_void_p),
                ("v_base", C.c_void_p), ("v_resid", C.c_void_p), ("v_scales", C.c_void_p)]


def lib():
    """Load libnq.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libnq.so is missing at {LIB_PATH}; build it with "
                                   "`python -m quantized_self_speculative_gb300.build` (needs nvcc)")
            L = C.CDLL(LIB_PATH)
            vp, i32, sz, u64, f32 = C.c_void_p, C.c_int, C.c_size_t, C.c_uint64, C.c_float
            W = C.POINTER(nq_weights)
            L.nq_packed_bytes.argtypes = [i32, i32, i32, i32, C.POINTER(sz), C.POINTER(sz), C.POINTER(sz)]
            L.nq_pack_weights.argtypes = [vp, W, vp]
            for name in ("nq_draft_gemv", "nq_verify_gemm"):
                getattr(L, name).argtypes = [W, vp, i32, vp, vp]
            for name in ("nq_draft_gemv_batch", "nq_verify_gemm_batch"):
                getattr(L, name).argtypes = [i32, W, C.POINTER(vp), i32, C.POINTER(vp), vp]
            for name in ("nq_draft_gemv_batch_ws", "nq_verify_gemm_batch_ws"):
                getattr(L, name).argtypes = [i32, W, C.POINTER(vp), i32, C.POINTER(vp), vp, sz, vp]
                getattr(L, name).restype = i32
            L.nq_linear_workspace_bytes.argtypes = [i32, W, i32, i32]
            L.nq_linear_workspace_bytes.restype = sz
            L.spec_accept_workspace_bytes.argtypes = [i32, i32, i32]
            L.spec_accept_workspace_bytes.restype = sz
            L.spec_accept_greedy.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, sz, vp]
            L.spec_accept_sample.argtypes = [vp, vp, vp, i32, i32, i32, f32, vp, u64, vp, vp, vp, sz, vp]
            L.nq_status_string.argtypes = [i32]
            L.nq_status_string.restype = C.c_char_p
            L.nq_get_device_status.argtypes = [vp, C.POINTER(C.c_uint32)]
            L.spec_draft_argmax.argtypes = [vp, i32, i32, vp, i32, vp, sz, vp]
            L.nq_quantize_act_int8.argtypes = [vp, i32, i32, vp, vp, vp]
            L.nq_linear_a8_batch.argtypes = [i32, W, C.POINTER(vp), C.POINTER(vp), i32, i32, C.POINTER(vp), vp]
            for name in ("nq_quantize_act_int8", "nq_linear_a8_batch"):
                getattr(L, name).restype = i32
            KV = C.POINTER(nq_kv_cache)
            L.nq_kv_cache_bytes.argtypes = [i32, i32, i32, i32, i32, C.POINTER(sz), C.POINTER(sz)]
            L.nq_kv_append.argtypes = [KV, vp, vp, i32, vp, vp]
            L.nq_attn_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
            L.nq_attn_workspace_bytes.restype = sz
            L.nq_attn_decode.argtypes = [KV, vp, i32, i32, vp, i32, f32, vp, vp, sz, vp]
            for name in ("nq_kv_cache_bytes", "nq_kv_append", "nq_attn_decode"):
                getattr(L, name).restype = i32
            L.spec_accept_sample_features.argtypes = [vp, vp, vp, i32, i32, i32, f32, vp, u64, vp, vp, vp, vp, sz, vp]
            L.spec_accept_sample_features.restype = i32
            L.nq_embed_rows.argtypes = [vp, i32, i32, vp, i32, i32, vp, vp]
            L.nq_embed_round.argtypes = [vp, i32, i32, vp, vp, i32, i32, vp, vp]
            L.spec_round_commit.argtypes = [vp, vp, i32, i32, vp, vp, i32, vp, vp]
            for name in ("spec_draft_argmax", "nq_embed_rows", "nq_embed_round", "spec_round_commit"):
                getattr(L, name).restype = i32
            L.nq_selftest_bounded_wait.argtypes = [C.c_uint32, vp]
            L.nq_selftest_bounded_wait.restype = i32
            for name in ("nq_packed_bytes", "nq_pack_weights", "nq_draft_gemv", "nq_verify_gemm",
                         "nq_draft_gemv_batch", "nq_verify_gemm_batch", "spec_accept_greedy",
                         "spec_accept_sample", "nq_get_device_status"):
                getattr(L, name).restype = i32
            _lib = L
        return _lib


def status_string(status: int) -> str:
    return lib().nq_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != NQ_OK:
        raise NQError(status, what)


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dev(t: torch.Tensor, dtype, what: str) -> int:
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{what} must be a contiguous CUDA tensor of {dtype}")
    return t.data_ptr()


# ---------------------------------------------------------------- weights
def packed_bytes(n_out: int, k_in: int, group: int, fmt: int):
    b, r, s = C.c_size_t(), C.c_size_t(), C.c_size_t()
    _check(lib().nq_packed_bytes(n_out, k_in, group, fmt, C.byref(b), C.byref(r), C.byref(s)), "nq_packed_bytes")
    return b.value, r.value, s.value


@dataclass
class PackedLinear:
    """A packed linear layer W [n_out][k_in]; buffers are uint8 device tensors."""
    n_out: int
    k_in: int
    group: int
    fmt: int
    base: torch.Tensor
    resid: Optional[torch.Tensor]
    scales: Optional[torch.Tensor]

    def struct(self) -> nq_weights:
        return nq_weights(self.n_out, self.k_in, self.group, self.fmt, self.base.data_ptr(),
                          None if self.resid is None else self.resid.data_ptr(),
                          None if self.scales is None else self.scales.data_ptr())

    def as_int4(self) -> "PackedLinear":
        """The INT4 view of a NESTED44 layer (same base plane and scales)."""
        return PackedLinear(self.n_out, self.k_in, self.group, FMT_INT4, self.base, None, self.scales)

    @property
    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.base, self.resid, self.scales) if t is not None)


def alloc_packed(n_out: int, k_in: int, group: int, fmt: int, device=None) -> PackedLinear:
    device = device or torch.device("cuda")
    b, r, s = packed_bytes(n_out, k_in, group, fmt)
    mk = lambda n: torch.empty(n, dtype=torch.uint8, device=device) if n else None
    return PackedLinear(n_out, k_in, group, fmt, mk(b), mk(r), mk(s))


def pack_weights(w: torch.Tensor, fmt: int = FMT_NESTED44, group: int = 128, stream=None) -> PackedLinear:
    n, k = w.shape
    out = alloc_packed(n, k, group, fmt, w.device)
    st = out.struct()
    _check(lib().nq_pack_weights(_dev(w, torch.float32, "w"), C.byref(st), _stream(stream)), "nq_pack_weights")
    return out


def pack_from_host(base, resid, scales, n_out, k_in, group, fmt, device=None) -> PackedLinear:
    """Upload already-packed planes (numpy arrays) to the device."""
    device = device or torch.device("cuda")
    t = lambda a: None if a is None else torch.from_numpy(a.reshape(-1).view("uint8").copy()).to(device)
    return PackedLinear(n_out, k_in, group, fmt, t(base), t(resid), t(scales))


# ---------------------------------------------------------------- linears
def _linear(fn: str, w: PackedLinear, x: torch.Tensor, y: Optional[torch.Tensor], stream) -> torch.Tensor:
    M = x.shape[0]
    if x.shape[-1] != w.k_in:
        raise ValueError("x must be [M][k_in]")
    if y is None:
        y = torch.empty((M, w.n_out), dtype=torch.float32, device=x.device)
    st = w.struct()
    xp = _dev(x, torch.bfloat16, "x") if x.dtype == torch.bfloat16 else _dev(x, torch.int16, "x")
    _check(getattr(lib(), fn)(C.byref(st), xp, M, _dev(y, torch.float32, "y"), _stream(stream)), fn)
    return y


def draft_gemv(w: PackedLinear, x: torch.Tensor, y=None, stream=None) -> torch.Tensor:
    """Draft pass: base plane only.  x: bf16 [M][k_in] -> y fp32 [M][n_out]."""
    return _linear("nq_draft_gemv", w, x, y, stream)


def verify_gemm(w: PackedLinear, x: torch.Tensor, y=None, stream=None) -> torch.Tensor:
    """Verify pass: both planes (8-bit target), or the FP8 / FP16 tiers."""
    return _linear("nq_verify_gemm", w, x, y, stream)


def linear_workspace_bytes(verify: bool, layers: Sequence[PackedLinear], M: int) -> int:
    """Workspace of nq_{draft_gemv,verify_gemm}_batch_ws (0: the tensor-core
    path is not taken for these layers and M)."""
    w = (nq_weights * len(layers))(*[L.struct() for L in layers])
    return lib().nq_linear_workspace_bytes(len(layers), w, M, int(verify))


class LinearBatch:
    """Prebuilt argument arrays for nq_{draft_gemv,verify_gemm}_batch: one
    persistent launch over many independent linears at the same M.  With
    tensor_cores=True the *_batch_ws entry point is used with a workspace
    allocated here (the tensor-memory kernel for M >= 16)."""

    def __init__(self, verify: bool, layers: Sequence[PackedLinear], xs: Sequence[torch.Tensor],
                 ys: Sequence[torch.Tensor], tensor_cores: bool = False):
        n = len(layers)
        assert n == len(xs) == len(ys) and n > 0
        self.fn = "nq_verify_gemm_batch" if verify else "nq_draft_gemv_batch"
        self.M = xs[0].shape[0]
        for L, x, y in zip(layers, xs, ys):
            assert x.shape == (self.M, L.k_in) and y.shape == (self.M, L.n_out)
            _dev(x, torch.bfloat16, "x")
            _dev(y, torch.float32, "y")
        self.count = n
        self.w = (nq_weights * n)(*[L.struct() for L in layers])
        self.x = (C.c_void_p * n)(*[x.data_ptr() for x in xs])
        self.y = (C.c_void_p * n)(*[y.data_ptr() for y in ys])
        self.ws = None
        if tensor_cores:
            self.fn += "_ws"
            nb = lib().nq_linear_workspace_bytes(n, self.w, self.M, int(verify))
            self.ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=xs[0].device)
        self._keep = (list(layers), list(xs), list(ys))

    def __call__(self, stream=None):
        if self.ws is None:
            _check(getattr(lib(), self.fn)(self.count, self.w, self.x, self.M, self.y, _stream(stream)), self.fn)
        else:
            _check(getattr(lib(), self.fn)(self.count, self.w, self.x, self.M, self.y, self.ws.data_ptr(),
                                           self.ws.numel(), _stream(stream)), self.fn)


# ---------------------------------------------------------------- acceptance
def workspace_bytes(B: int, k: int, V: int) -> int:
    return lib().spec_accept_workspace_bytes(B, k, V)


def accept_workspace(B: int, k: int, V: int, device=None) -> torch.Tensor:
    """Zero-filled workspace (the calls leave it ready for reuse)."""
    n = workspace_bytes(B, k, V)
    if n == 0:
        raise NQError(NQ_ERR_ARG, "spec_accept_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device or torch.device("cuda"))


def accept_greedy(draft: torch.Tensor, tgt_logits: torch.Tensor, ws: Optional[torch.Tensor] = None,
                  out_tok=None, out_cnt=None, stream=None):
    B, k = draft.shape
    V = tgt_logits.shape[-1]
    if tgt_logits.shape != (B, k + 1, V):
        raise ValueError("tgt_logits must be [B][k+1][V]")
    ws = ws if ws is not None else accept_workspace(B, k, V, draft.device)
    out_tok = out_tok if out_tok is not None else torch.empty((B, k + 1), dtype=torch.int32, device=draft.device)
    out_cnt = out_cnt if out_cnt is not None else torch.empty(B, dtype=torch.int32, device=draft.device)
    _check(lib().spec_accept_greedy(_dev(draft, torch.int32, "draft"), _dev(tgt_logits, torch.float32, "tgt_logits"),
                                    B, k, V, _dev(out_tok, torch.int32, "out_tok"), _dev(out_cnt, torch.int32, "out_cnt"),
                                    _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)), "spec_accept_greedy")
    return out_tok, out_cnt


def accept_sample(draft: torch.Tensor, draft_logits: torch.Tensor, tgt_logits: torch.Tensor, temperature: float,
                  seeds: torch.Tensor, round_: int, ws: Optional[torch.Tensor] = None, out_tok=None, out_cnt=None,
                  stream=None):
    B, k = draft.shape
    V = tgt_logits.shape[-1]
    if tgt_logits.shape != (B, k + 1, V) or draft_logits.shape != (B, k, V):
        raise ValueError("draft_logits must be [B][k][V] and tgt_logits [B][k+1][V]")
    ws = ws if ws is not None else accept_workspace(B, k, V, draft.device)
    out_tok = out_tok if out_tok is not None else torch.empty((B, k + 1), dtype=torch.int32, device=draft.device)
    out_cnt = out_cnt if out_cnt is not None else torch.empty(B, dtype=torch.int32, device=draft.device)
    seeds_p = _dev(seeds, torch.int64, "seeds") if seeds.dtype == torch.int64 else _dev(seeds, torch.uint64, "seeds")
    _check(lib().spec_accept_sample(_dev(draft, torch.int32, "draft"), _dev(draft_logits, torch.float32, "draft_logits"),
                                    _dev(tgt_logits, torch.float32, "tgt_logits"), B, k, V, float(temperature),
                                    seeds_p, int(round_) & (2**64 - 1), _dev(out_tok, torch.int32, "out_tok"),
                                    _dev(out_cnt, torch.int32, "out_cnt"), _dev(ws, torch.uint8, "ws"), ws.numel(),
                                    _stream(stream)), "spec_accept_sample")
    return out_tok, out_cnt


# ---------------------------------------------------------------- round bookkeeping
def draft_argmax(logits: torch.Tensor, tok: torch.Tensor, tok_stride: int = 1, ws: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    """tok[m * tok_stride] = argmax of logits row m (fp32 [M][V]); tok is an
    int32 tensor viewed flat (it may be a strided slice's base)."""
    M, V = logits.shape
    ws = ws if ws is not None else accept_workspace(M, 0, V, logits.device)
    _check(lib().spec_draft_argmax(_dev(logits, torch.float32, "logits"), M, V, tok.data_ptr(), int(tok_stride),
                                   _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)), "spec_draft_argmax")
    return tok


def embed_rows(table: torch.Tensor, ids: torch.Tensor, M: int, ids_stride: int = 1, out=None, stream=None):
    """out[m] = table[ids[m * ids_stride]] (table bf16 [V][d]); ids int32."""
    V, d = table.shape
    out = out if out is not None else torch.empty((M, d), dtype=torch.bfloat16, device=table.device)
    _check(lib().nq_embed_rows(_dev(table, torch.bfloat16, "table"), V, d, ids.data_ptr(), int(ids_stride), M,
                               _dev(out, torch.bfloat16, "out"), _stream(stream)), "nq_embed_rows")
    return out


def embed_round(table: torch.Tensor, x0: torch.Tensor, draft: Optional[torch.Tensor], B: int, k: int, out=None,
                stream=None):
    """The verify rows of a round: out[b][0] = table[x0[b]], out[b][j] = table[draft[b][j-1]]."""
    V, d = table.shape
    out = out if out is not None else torch.empty((B * (k + 1), d), dtype=torch.bfloat16, device=table.device)
    _check(lib().nq_embed_round(_dev(table, torch.bfloat16, "table"), V, d, x0.data_ptr(),
                                None if draft is None else draft.data_ptr(), B, k, _dev(out, torch.bfloat16, "out"),
                                _stream(stream)), "nq_embed_round")
    return out


def round_commit(out_tok: torch.Tensor, out_cnt: torch.Tensor, seq: torch.Tensor, seq_len: torch.Tensor,
                 x0: torch.Tensor, stream=None) -> None:
    """Append the emitted tokens to seq [B][max_len] (int32), advance seq_len,
    set x0 to each row's last emitted token (all in place, on the device)."""
    B, k1 = out_tok.shape
    _check(lib().spec_round_commit(_dev(out_tok, torch.int32, "out_tok"), _dev(out_cnt, torch.int32, "out_cnt"), B,
                                   k1 - 1, _dev(seq, torch.int32, "seq"), _dev(seq_len, torch.int32, "seq_len"),
                                   seq.shape[1], _dev(x0, torch.int32, "x0"), _stream(stream)), "spec_round_commit")


def accept_sample_features(draft: torch.Tensor, draft_logits: torch.Tensor, tgt_logits: torch.Tensor,
                           temperature: float, seeds: torch.Tensor, round_: int, ws: Optional[torch.Tensor] = None,
                           out_tok=None, out_cnt=None, features=None, stream=None):
    """spec_accept_sample plus SpecKV's step features per row: (mean entropy,
    mean confidence, max entropy, min confidence) of the k drafted positions."""
    B, k = draft.shape
    V = tgt_logits.shape[-1]
    ws = ws if ws is not None else accept_workspace(B, k, V, draft.device)
    out_tok = out_tok if out_tok is not None else torch.empty((B, k + 1), dtype=torch.int32, device=draft.device)
    out_cnt = out_cnt if out_cnt is not None else torch.empty(B, dtype=torch.int32, device=draft.device)
    features = features if features is not None else torch.empty((B, 4), dtype=torch.float32, device=draft.device)
    seeds_p = _dev(seeds, torch.int64, "seeds") if seeds.dtype == torch.int64 else _dev(seeds, torch.uint64, "seeds")
    _check(lib().spec_accept_sample_features(
        _dev(draft, torch.int32, "draft"), _dev(draft_logits, torch.float32, "draft_logits"),
        _dev(tgt_logits, torch.float32, "tgt_logits"), B, k, V, float(temperature), seeds_p, int(round_) & (2**64 - 1),
        _dev(out_tok, torch.int32, "out_tok"), _dev(out_cnt, torch.int32, "out_cnt"),
        _dev(features, torch.float32, "features"), _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)),
        "spec_accept_sample_features")
    return out_tok, out_cnt, features


# ---------------------------------------------------------------- int8 activations (W4A8 -> W8A8)
def quantize_act_int8(x: torch.Tensor, xq=None, sx=None, stream=None):
    """bf16 [M][K] -> (int8 codes [M][K], fp32 row scales [M])."""
    M, K = x.shape
    xq = xq if xq is not None else torch.empty((M, K), dtype=torch.int8, device=x.device)
    sx = sx if sx is not None else torch.empty(M, dtype=torch.float32, device=x.device)
    _check(lib().nq_quantize_act_int8(_dev(x, torch.bfloat16, "x"), M, K, _dev(xq, torch.int8, "xq"),
                                      _dev(sx, torch.float32, "sx"), _stream(stream)), "nq_quantize_act_int8")
    return xq, sx


class LinearA8Batch:
    """Prebuilt argument arrays for nq_linear_a8_batch (one launch over many
    linears at the same M, int8 activation codes and row scales)."""

    def __init__(self, verify: bool, layers: Sequence[PackedLinear], xqs, sxs, ys):
        n = len(layers)
        self.verify, self.count, self.M = int(verify), n, xqs[0].shape[0]
        self.w = (nq_weights * n)(*[L.struct() for L in layers])
        self.xq = (C.c_void_p * n)(*[t.data_ptr() for t in xqs])
        self.sx = (C.c_void_p * n)(*[t.data_ptr() for t in sxs])
        self.y = (C.c_void_p * n)(*[t.data_ptr() for t in ys])
        self._keep = (list(layers), list(xqs), list(sxs), list(ys))

    def __call__(self, stream=None):
        _check(lib().nq_linear_a8_batch(self.count, self.w, self.xq, self.sx, self.M, self.verify, self.y,
                                        _stream(stream)), "nq_linear_a8_batch")


def linear_a8(w: PackedLinear, xq: torch.Tensor, sx: torch.Tensor, verify: bool, y=None, stream=None):
    """One int8-activation linear: y fp32 [M][n_out]."""
    M = xq.shape[0]
    y = y if y is not None else torch.empty((M, w.n_out), dtype=torch.float32, device=xq.device)
    LinearA8Batch(verify, [w], [xq], [sx], [y])(stream)
    return y


# ---------------------------------------------------------------- nested KV cache
class KVCache:
    """One layer's nested KV cache (device buffers allocated here, uint8;
    BitNest Fig. 4): planes [batch][heads_kv][max_len][head_dim/2], fp16
    scales [batch][heads_kv][max_len][head_dim/group], for K and for V."""

    def __init__(self, batch: int, heads_kv: int, head_dim: int, group: int, max_len: int, device=None):
        device = device or torch.device("cuda")
        pb, sb = C.c_size_t(), C.c_size_t()
        _check(lib().nq_kv_cache_bytes(batch, heads_kv, head_dim, group, max_len, C.byref(pb), C.byref(sb)),
               "nq_kv_cache_bytes")
        self.batch, self.heads_kv, self.head_dim, self.group, self.max_len = batch, heads_kv, head_dim, group, max_len
        mk = lambda n: torch.zeros(n, dtype=torch.uint8, device=device)
        self.k_base, self.k_resid, self.k_scales = mk(pb.value), mk(pb.value), mk(sb.value)
        self.v_base, self.v_resid, self.v_scales = mk(pb.value), mk(pb.value), mk(sb.value)
        self.plane_bytes, self.scale_bytes = pb.value, sb.value

    def struct(self) -> nq_kv_cache:
        return nq_kv_cache(self.batch, self.heads_kv, self.head_dim, self.group, self.max_len, 0,
                           self.k_base.data_ptr(), self.k_resid.data_ptr(), self.k_scales.data_ptr(),
                           self.v_base.data_ptr(), self.v_resid.data_ptr(), self.v_scales.data_ptr())

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor, pos: torch.Tensor, stream=None) -> None:
        """Quantise k_new, v_new fp32 [batch][heads_kv][n][head_dim] into rows pos[b] .."""
        n = k_new.shape[2]
        st = self.struct()
        _check(lib().nq_kv_append(C.byref(st), _dev(k_new, torch.float32, "k_new"), _dev(v_new, torch.float32, "v_new"),
                                  n, _dev(pos, torch.int32, "pos"), _stream(stream)), "nq_kv_append")

    def attention(self, q: torch.Tensor, lens: torch.Tensor, planes: int, scale: float, out=None, ws=None,
                  stream=None) -> torch.Tensor:
        """softmax(scale q K^T) V over the 4-bit (planes=1) or 8-bit (planes=2)
        view; q fp32 [batch][M][heads_q][head_dim]."""
        B, M, Hq, d = q.shape
        out = out if out is not None else torch.empty_like(q)
        need = lib().nq_attn_workspace_bytes(B, M, Hq, d, self.max_len)
        ws = ws if ws is not None else torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
        st = self.struct()
        _check(lib().nq_attn_decode(C.byref(st), _dev(q, torch.float32, "q"), M, Hq, _dev(lens, torch.int32, "lens"),
                                    int(planes), float(scale), _dev(out, torch.float32, "out"),
                                    _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)), "nq_attn_decode")
        return out

    def host_dict(self):
        """The cache buffers as numpy arrays shaped for the oracle."""
        sh = (self.batch, self.heads_kv, self.max_len)
        p = lambda t: t.cpu().numpy().reshape(*sh, self.head_dim // 2)
        sc = lambda t: t.cpu().numpy().view("uint16").reshape(*sh, self.head_dim // self.group)
        return dict(k_base=p(self.k_base), k_resid=p(self.k_resid), k_scales=sc(self.k_scales),
                    v_base=p(self.v_base), v_resid=p(self.v_resid), v_scales=sc(self.v_scales))


def selftest_bounded_wait(limit_us: int, stream=None) -> None:
    """Run the bounded-wait diagnostic (a wait that nothing completes gives up
    after limit_us and sets NQ_DEV_TIMEOUT); read the bit with device_status()."""
    _check(lib().nq_selftest_bounded_wait(int(limit_us), _stream(stream)), "nq_selftest_bounded_wait")


def device_status(stream=None) -> int:
    """Read and clear the sticky device status word (NQ_DEV_* bits)."""
    v = C.c_uint32()
    _check(lib().nq_get_device_status(_stream(stream), C.byref(v)), "nq_get_device_status")
    return v.value
