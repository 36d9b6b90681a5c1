"""Helpers shared by the GPU parity tests (no method arithmetic here)."""
import numpy as np
import torch

import oracle as O

TOL = 2e-3   # normwise max relative error vs the fp64-accumulated oracle (bf16 activations)


def normwise_err(y_gpu: np.ndarray, y_ref: np.ndarray) -> float:
    denom = np.abs(y_ref).max()
    return float(np.abs(y_gpu.astype(np.float64) - y_ref).max() / (denom if denom > 0 else 1.0))


def to_dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a).reshape(-1).view(np.uint8).copy()).cuda()


def oracle_packed(nq, w: np.ndarray, fmt: int, group: int):
    """Pack on the CPU with the oracle; upload the planes; return (PackedLinear, host planes)."""
    n, k = w.shape
    if fmt in (nq.FMT_NESTED44, nq.FMT_INT4):
        base, resid, scales = O.pack_nested(w, group, with_resid=fmt == nq.FMT_NESTED44)
    elif fmt == nq.FMT_FP8E4M3_ROW:
        base, scales = O.pack_fp8(w)
        resid = None
    else:
        base, resid, scales = O.pack_fp16(w), None, None
    pl = nq.PackedLinear(n, k, group, fmt, to_dev_u8(base), None if resid is None else to_dev_u8(resid),
                         None if scales is None else to_dev_u8(scales))
    return pl, (base, resid, scales)


def oracle_fmt(nq, fmt):
    return {nq.FMT_NESTED44: O.FMT_NESTED44, nq.FMT_INT4: O.FMT_INT4,
            nq.FMT_FP8E4M3_ROW: O.FMT_FP8, nq.FMT_FP16: O.FMT_FP16}[fmt]


def bf16_dev(x_bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(x_bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
