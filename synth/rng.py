"""Counter-based SplitMix64 streams, numpy and torch flavours (bit-identical)."""

from __future__ import annotations

import hashlib

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
_C1 = 0xBF58476D1CE4E5B9
_C2 = 0x94D049BB133111EB
_MASK = (1 << 64) - 1


def _signed(v: int) -> int:
    v &= _MASK
    return v - (1 << 64) if v >= (1 << 63) else v


def stream_key(seed: int, *tags) -> int:
    """A 64-bit stream key from a seed and any tags (ints or strings)."""
    h = hashlib.sha256(repr((int(seed),) + tuple(tags)).encode()).digest()
    return int.from_bytes(h[:8], "little")


def mix64_np(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= np.uint64(_C1)
        z ^= z >> np.uint64(27)
        z *= np.uint64(_C2)
        z ^= z >> np.uint64(31)
    return z


def u64_stream_np(key: int, start: int, count: int) -> np.ndarray:
    """Values start .. start+count-1 of stream `key` as uint64."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = idx * np.uint64(GOLDEN) + np.uint64(key & _MASK)
    return mix64_np(z)


def _lsr(z, s: int):
    # logical shift right on int64 tensors
    return (z >> s) & ((1 << (64 - s)) - 1)


def u64_stream_torch(key: int, start: int, count: int, device="cpu"):
    """Same values as u64_stream_np, as an int64 torch tensor (two's complement)."""
    import torch

    idx = torch.arange(start + 1, start + count + 1, dtype=torch.int64, device=device)
    z = idx * _signed(GOLDEN) + _signed(key)
    z = (z ^ _lsr(z, 30)) * _signed(_C1)
    z = (z ^ _lsr(z, 27)) * _signed(_C2)
    z = z ^ _lsr(z, 31)
    return z


def u64_stream_torch_keys(keys, count: int, device="cpu"):
    """Rows of streams: out[r, i] = value i of stream keys[r] (int64 tensor)."""
    import torch

    k = torch.tensor([_signed(int(v)) for v in keys], dtype=torch.int64, device=device)[:, None]
    idx = torch.arange(1, count + 1, dtype=torch.int64, device=device)[None, :]
    z = idx * _signed(GOLDEN) + k
    z = (z ^ _lsr(z, 30)) * _signed(_C1)
    z = (z ^ _lsr(z, 27)) * _signed(_C2)
    return z ^ _lsr(z, 31)


def uniform01_np(key: int, start: int, count: int) -> np.ndarray:
    """Doubles in [0, 1) with 53 random bits."""
    return (u64_stream_np(key, start, count) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
