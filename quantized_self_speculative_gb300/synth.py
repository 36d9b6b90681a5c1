"""Seeded synthetic inputs for the hot path (numpy PCG64).

This module draws inputs only: weights, activations, logits and draft tokens
with the shapes and distributions of the workloads the kernels are measured
on.  It holds none of the method's arithmetic (no quantisation, no dequantised
matmul, no acceptance rule), so the CUDA path and the CPU oracle can both be
fed from it without sharing any of their computation.
"""
from __future__ import annotations

import numpy as np


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bfloat16 (nearest, ties to even); returns the uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def weights(seed: int, n_out: int, k_in: int, std: float = 0.02) -> np.ndarray:
    """W fp32 [n_out][k_in] ~ N(0, std^2)."""
    return (rng(seed).standard_normal((n_out, k_in), dtype=np.float32) * np.float32(std)).astype(np.float32)


def random_planes(seed: int, n_out: int, k_in: int, group: int):
    """Packed nibble planes drawn byte-uniform (every 4-bit code pair, including
    base -8 with a negative refinement, which quantising tiny weights also
    produces) and fp16 group-scale bits from a mix of classes: zero, subnormal,
    normal up to 0.0625, normal above it (up to 8), and negatives of the normal
    classes.  Returns (base uint8 [n][k/2], resid uint8 [n][k/2],
    scales uint16 [n][k/group])."""
    g = rng(seed)
    base = g.integers(0, 256, size=(n_out, k_in // 2), dtype=np.uint8)
    resid = g.integers(0, 256, size=(n_out, k_in // 2), dtype=np.uint8)
    shape = (n_out, k_in // group)
    cls = g.integers(0, 6, size=shape)
    bits = np.where(cls == 0, 0,
           np.where(cls == 1, g.integers(1, 0x0400, size=shape),
           np.where(cls == 2, g.integers(0x0400, 0x2C00, size=shape),
           np.where(cls == 3, g.integers(0x2C00, 0x4800, size=shape),
           np.where(cls == 4, 0x8000 | g.integers(0x0400, 0x2C00, size=shape),
                    0x8000 | g.integers(0x2C00, 0x4800, size=shape))))))
    return base, resid, bits.astype(np.uint16)


def activations_bf16(seed: int, m: int, k_in: int, std: float = 1.0) -> np.ndarray:
    """x bf16 bits [m][k_in], values ~ N(0, std^2) rounded to bfloat16."""
    return f32_to_bf16_bits(rng(seed).standard_normal((m, k_in), dtype=np.float32) * np.float32(std))


def target_logits(seed: int, B: int, k: int, V: int, std: float) -> np.ndarray:
    """Target logits fp32 [B][k+1][V] ~ N(0, std^2)."""
    return (rng(seed).standard_normal((B, k + 1, V), dtype=np.float32) * np.float32(std)).astype(np.float32)


def draft_logits_from(tgt: np.ndarray, seed: int, noise_std: float) -> np.ndarray:
    """Draft logits fp32 [B][k][V] = target logits at positions 0..k-1 plus N(0, noise_std^2)."""
    B, k1, V = tgt.shape
    noise = rng(seed).standard_normal((B, k1 - 1, V), dtype=np.float32) * np.float32(noise_std)
    return (tgt[:, :-1, :] + noise).astype(np.float32)


def draft_tokens_greedy(draft_logits: np.ndarray) -> np.ndarray:
    """The draft model's own greedy choices: argmax over the vocabulary [B][k]."""
    return np.argmax(draft_logits, axis=-1).astype(np.int32)


def draft_tokens_sampled(draft_logits: np.ndarray, seed: int, temperature: float = 1.0) -> np.ndarray:
    """The draft model's sampled tokens d_j ~ softmax(draft_logits_j / T) [B][k],
    drawn with numpy in fp64 (this is the draft model's behaviour, upstream of
    the acceptance step)."""
    g = rng(seed)
    z = draft_logits.astype(np.float64) / temperature
    z -= z.max(axis=-1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=-1, keepdims=True)
    cdf = np.cumsum(p, axis=-1)
    u = g.random(p.shape[:-1])[..., None] * cdf[..., -1:]
    tok = (cdf <= u).sum(axis=-1)
    return np.minimum(tok, p.shape[-1] - 1).astype(np.int32)


def seeds_for(run: int, B: int) -> np.ndarray:
    """Per-row Philox seeds: 1000 * run + b."""
    return (np.uint64(1000 * run) + np.arange(B, dtype=np.uint64)).astype(np.uint64)


# Linear-layer shapes of the synthetic models (n_out, k_in), per layer, plus lm_head.
def llama2_7b_linears():
    h, f = 4096, 11008
    layer = [("q", h, h), ("k", h, h), ("v", h, h), ("o", h, h), ("gate", f, h), ("up", f, h), ("down", h, f)]
    return layer, ("lm_head", 32000, h), 32


def llama3_8b_linears():
    h, f = 4096, 14336
    layer = [("q", h, h), ("k", 1024, h), ("v", 1024, h), ("o", h, h), ("gate", f, h), ("up", f, h), ("down", h, f)]
    return layer, ("lm_head", 128256, h), 32


def qwen25_7b_linears():
    h, f = 3584, 18944
    layer = [("q", h, h), ("k", 512, h), ("v", 512, h), ("o", h, h), ("gate", f, h), ("up", f, h), ("down", h, f)]
    return layer, ("lm_head", 152064, h), 28
