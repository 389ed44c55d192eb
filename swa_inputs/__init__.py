"""Seeded synthetic inputs for SWA(w, s) prefill and decode.

This module is shared by the CUDA path's tests and benchmark and by the fp64
oracle's tests. It holds no attention arithmetic: it only draws random tensors
with the shapes and value distributions of the workloads the pages describe
(Llama-3.1-8B / Mistral-7B head geometry: Hq=32, Hkv=8, d=128; windows 64..2048;
4 or 100 sinks; contexts up to 256K) and casts them to bf16.

Two generators:

* ``prefill_inputs`` draws q, k, v for a whole prompt from
  ``torch.Generator('cpu').manual_seed(seed)`` as fp32 N(0,1), in the order
  q, k, v, then rounds to bf16 (round-to-nearest-even). Optionally the keys of
  the first ``sink_rows`` positions are multiplied by ``sink_scale`` (a power of
  two, so exact in bf16) so that the sink tokens draw heavy attention mass.

* ``keyed_rows`` is a counter-based generator: the row for (seed, stream, b,
  head, position) is a pure function of those integers (splitmix64 hash ->
  two uniforms -> Box-Muller), so a decode test at position 262143 can draw
  exactly the keys/values of any earlier position without storing the whole
  history.
"""
from __future__ import annotations

import numpy as np
import torch

__all__ = [
    "prefill_inputs",
    "keyed_rows",
    "decode_query",
    "bf16_bits",
    "to_bf16",
]


def to_bf16(x: np.ndarray | torch.Tensor) -> torch.Tensor:
    """Round an fp32 array to a bf16 torch tensor (round-to-nearest-even)."""
    if isinstance(x, np.ndarray):
        x = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return x.to(torch.float32).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw 16-bit patterns of a bf16 tensor as a contiguous uint16 array."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def prefill_inputs(B: int, L: int, Hq: int, Hkv: int, d: int, seed: int,
                   sink_rows: int = 0, sink_scale: float = 4.0):
    """q [B,L,Hq,d], k [B,L,Hkv,d], v [B,L,Hkv,d] as bf16 CPU tensors."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    q = torch.randn(B, L, Hq, d, generator=g, dtype=torch.float32)
    k = torch.randn(B, L, Hkv, d, generator=g, dtype=torch.float32)
    v = torch.randn(B, L, Hkv, d, generator=g, dtype=torch.float32)
    if sink_rows > 0:
        k[:, :sink_rows] *= float(sink_scale)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)


def _splitmix64(x: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser (Steele, Lea, Flood 2014) on uint64 arrays."""
    with np.errstate(over="ignore"):
        z = (x + np.uint64(0x9E3779B97F4A7C15)) & _M64
        z = ((z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)) & _M64
        z = ((z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)) & _M64
        return z ^ (z >> np.uint64(31))


def keyed_rows(seed: int, stream: int, b: int, head: int, positions, d: int,
               scale: float = 1.0) -> torch.Tensor:
    """bf16 rows [len(positions), d] of N(0, scale^2) values keyed by position.

    ``stream`` separates independent tensors (e.g. 0 = keys, 1 = values,
    2 = queries). Each element is a pure function of
    (seed, stream, b, head, position, element index).
    """
    pos = np.asarray(positions, dtype=np.uint64).reshape(-1, 1)
    half = (d + 1) // 2
    idx = np.arange(half, dtype=np.uint64).reshape(1, -1)
    with np.errstate(over="ignore"):
        base = _splitmix64(np.uint64(seed) * np.uint64(0x100000001B3)
                           ^ np.uint64(stream) * np.uint64(0x9E3779B1)
                           ^ np.uint64(b) << np.uint64(20)
                           ^ np.uint64(head) << np.uint64(44))
        h = _splitmix64(base ^ (pos << np.uint64(16)) ^ idx)
    u1 = ((h >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)
    h2 = _splitmix64(h)
    u2 = (h2 >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    r = np.sqrt(-2.0 * np.log(u1))
    z0 = r * np.cos(2.0 * np.pi * u2)
    z1 = r * np.sin(2.0 * np.pi * u2)
    z = np.empty((pos.shape[0], 2 * half), dtype=np.float64)
    z[:, 0::2] = z0
    z[:, 1::2] = z1
    return to_bf16((z[:, :d] * scale).astype(np.float32))


def decode_query(B: int, Hq: int, d: int, seed: int) -> torch.Tensor:
    """One decode step's queries q [B, Hq, d] as bf16, N(0,1) from ``seed``."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    return torch.randn(B, Hq, d, generator=g, dtype=torch.float32).to(torch.bfloat16)
