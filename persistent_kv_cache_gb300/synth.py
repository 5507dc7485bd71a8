"""Seeded synthetic inputs for the KV-cache workloads.

This module only draws numbers: it holds none of the cache or attention
arithmetic, and both the CUDA path's tests/benchmark and the CPU oracle take
their inputs from it.  Every tensor comes from ``torch.Generator`` seeded with
``(seed, stream)``, so a given call always returns the same bytes on one
machine.

The rotary cos/sin caches are inputs of the attention operator (the
onnxruntime GroupQueryAttention op takes them as ``cos_cache``/``sin_cache``
tensors, indexed by absolute position); ``rope_cache`` builds the usual table
for base ``theta`` in float64 and rounds it to float32.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

_MASK63 = (1 << 63) - 1


def _gen(seed: int, stream: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(((seed * 1_000_003) ^ (stream * 0x9E3779B1)) & _MASK63)
    return g


def normal(shape, seed: int, stream: int, dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """N(0, 1) drawn in float32, rounded to ``dtype`` (round-to-nearest-even)."""
    t = torch.randn(tuple(shape), generator=_gen(seed, stream, device), dtype=torch.float32,
                    device=device)
    return t.to(dtype)


def randint(low: int, high: int, shape, seed: int, stream: int, dtype=torch.int64,
            device="cpu") -> torch.Tensor:
    """Uniform integers in [low, high)."""
    return torch.randint(low, high, tuple(shape), generator=_gen(seed, stream, device),
                         dtype=torch.int64, device=device).to(dtype)


def rope_cache(max_pos: int, head_dim: int, theta: float = 10000.0):
    """(cos, sin) float32 tables of shape [max_pos, head_dim / 2]: angle
    pos * theta^(-2i / head_dim), computed in float64."""
    half = head_dim // 2
    inv = theta ** (-(2.0 * np.arange(half, dtype=np.float64)) / head_dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return (torch.from_numpy(np.cos(ang).astype(np.float32)),
            torch.from_numpy(np.sin(ang).astype(np.float32)))


def bits(t: torch.Tensor) -> np.ndarray:
    """CPU tensor -> numpy array the oracle accepts (16-bit floats as uint16 bits)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float16:
        return t.numpy()
    return t.numpy()


def from_bits(a: np.ndarray, dtype) -> torch.Tensor:
    """Inverse of :func:`bits`."""
    if dtype == torch.bfloat16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a))


# --------------------------------------------------------------------------
# workload descriptions (shapes and distributions of the five workloads)
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class ScatterWorkload:
    """Circular TensorScatter into one cache of shape (B, H, max_seq, D)."""
    name: str
    batch: int
    heads: int
    max_seq: int
    head_dim: int
    new_tokens: tuple
    steps_per_len: int
    dtype: torch.dtype = torch.bfloat16


@dataclass(frozen=True)
class DecodeWorkload:
    """Append S new tokens, then GQA attention over the cache."""
    name: str
    batch: int
    q_heads: int
    kv_heads: int
    head_dim: int
    capacity: int
    window: int            # <= 0: no local window
    windowed: bool         # windowed (sliding) cache vs contiguous cache
    total_lo: int          # absolute total length range after the step (inclusive)
    total_hi: int
    new_tokens: tuple = (1,)
    steps: int = 1
    rope: bool = True
    dtype: torch.dtype = torch.bfloat16
    theta: float = 10000.0
    extra: dict = field(default_factory=dict)


TINY = DecodeWorkload("tiny-f32-scatter-then-decode", batch=2, q_heads=4, kv_heads=2,
                      head_dim=8, capacity=16, window=0, windowed=False, total_lo=1,
                      total_hi=16, rope=False, dtype=torch.float32)
SCATTER = ScatterWorkload("scatter-circular-bf16-16x8x4096x128", batch=16, heads=8,
                          max_seq=4096, head_dim=128, new_tokens=(1, 16, 64),
                          steps_per_len=100)
CONTIG_DECODE = DecodeWorkload("contiguous-decode-bf16-b32-h32kv8-d128-c8192", batch=32,
                               q_heads=32, kv_heads=8, head_dim=128, capacity=8192, window=0,
                               windowed=False, total_lo=512, total_hi=8192)
WINDOW_DECODE = DecodeWorkload("window-decode-bf16-b64-h64kv8-d64-w128", batch=64, q_heads=64,
                               kv_heads=8, head_dim=64, capacity=128, window=128, windowed=True,
                               total_lo=1, total_hi=32768, steps=256)
# the drifting layout at the capacity the sliding-window PR's CPU commit finds
# best for decode latency (C = W + 16, so a block of 17 rows is reclaimed
# every 17 one-token steps)
WINDOW_DECODE_DRIFT = DecodeWorkload("window-decode-drift-bf16-b64-h64kv8-d64-c144-w128",
                                     batch=64, q_heads=64, kv_heads=8, head_dim=64,
                                     capacity=144, window=128, windowed=True, total_lo=1,
                                     total_hi=32768, steps=256, extra={"policy": 2})
# the same window held in a ring of C = W slots (token p in slot p mod C)
WINDOW_DECODE_RING = DecodeWorkload("window-decode-ring-bf16-b64-h64kv8-d64-c128-w128",
                                    batch=64, q_heads=64, kv_heads=8, head_dim=64,
                                    capacity=128, window=128, windowed=True, total_lo=1,
                                    total_hi=32768, steps=256, extra={"policy": 3})
WINDOW_PREFILL = DecodeWorkload("window-prefill-bf16-b8-h16kv8-d256-w4096", batch=8,
                                q_heads=16, kv_heads=8, head_dim=256, capacity=4096,
                                window=4096, windowed=True, total_lo=0, total_hi=20000,
                                new_tokens=(64, 512, 2048))
# one-token decode on the windowed-prefill workload's heads (16 / 8, head_dim
# 256) held as a ring of C = W = 4096 slots, past lengths as the prefill's
WINDOW_DECODE_256 = DecodeWorkload("window-decode-ring-bf16-b8-h16kv8-d256-c4096-w4096",
                                   batch=8, q_heads=16, kv_heads=8, head_dim=256,
                                   capacity=4096, window=4096, windowed=True, total_lo=1,
                                   total_hi=20000, extra={"policy": 3})
