"""Seeded, counter-based synthetic inputs for the CSA2 attention step.

This module is the only code shared by the CPU oracle's tests and the CUDA
path's tests and benchmark.  It does none of the method's arithmetic: it
only turns (stream, element index) pairs into values with the distributions
the workloads call for, so that any slice of any tensor can be regenerated
independently, on the host (numpy) or on the device (torch integer ops).

Every value comes from a 32-bit integer hash followed by a table lookup or an
exact integer-to-float conversion.  No floating-point arithmetic runs on the
device, so the host and device generators agree bit for bit.

Distributions
-------------
* ``normal``:  the bf16 value nearest to the Gaussian quantile
  ``Phi^-1((k + 0.5) / 65536)`` for a 16-bit hash value ``k`` (optionally
  times a constant, applied in float64 before the one rounding to bf16 or
  fp32).  This is inverse-CDF sampling of N(0, sigma^2) at 16-bit resolution.
* ``uniform``: ``((h >> 9) + 0.5) * 2**-23`` in (0, 1), exact in fp32.
"""
from __future__ import annotations

import functools

import numpy as np

MASK32 = 0xFFFFFFFF
_M = 0x045D9F3B          # multiplier < 2**27: products of 32-bit values stay < 2**59
_GOLD = 0x9E3779B9


# --------------------------------------------------------------------------
# integer hash (host: numpy uint32, whose multiply wraps modulo 2**32 -- the
# same value as the masked 64-bit product of the device twin)
# --------------------------------------------------------------------------
_M32 = np.uint32(_M)
_S16 = np.uint32(16)


def _mix_np(x: np.ndarray, t: np.ndarray) -> np.ndarray:
    """In-place 32-bit mix of x (t: scratch of the same shape)."""
    for _ in range(2):
        np.right_shift(x, _S16, out=t)
        np.bitwise_xor(x, t, out=x)
        np.multiply(x, _M32, out=x)
    np.right_shift(x, _S16, out=t)
    np.bitwise_xor(x, t, out=x)
    return x


def _mix_int(x: int) -> int:
    x = (((x >> 16) ^ x) * _M) & MASK32
    x = (((x >> 16) ^ x) * _M) & MASK32
    return (x >> 16) ^ x


def stream_id(*parts: int) -> int:
    """Fold integers (seed, tensor id, sequence, layer, ...) into a 32-bit stream key."""
    h = 0x12345678
    for p in parts:
        h = _mix_int((h ^ (int(p) & MASK32)) & MASK32)
        h = _mix_int((h + _GOLD) & MASK32)
    return h


def _keys(stream: int, hi: int):
    k1 = _mix_int((stream ^ ((hi * _GOLD) & MASK32)) & MASK32)
    k2 = _mix_int((k1 + 0x7F4A7C15) & MASK32)
    return k1, k2


def _generate(stream: int, start: int, count: int, out: np.ndarray, fn) -> np.ndarray:
    """out[i] = fn(hash of element start + i), computed in cache-sized chunks."""
    chunk = 1 << 18
    x = np.empty(min(chunk, max(count, 1)), dtype=np.uint32)
    t = np.empty_like(x)
    i = start
    pos = 0
    while pos < count:                      # never cross a change of the high 32 index bits
        hi = i >> 32
        lo = i & MASK32
        n = min(count - pos, (1 << 32) - lo, chunk)
        k1, k2 = _keys(stream, hi)
        xv, tv = x[:n], t[:n]
        xv[:] = np.arange(lo, lo + n, dtype=np.uint64)
        np.bitwise_xor(xv, np.uint32(k1), out=xv)
        _mix_np(xv, tv)
        np.bitwise_xor(xv, np.uint32(k2), out=xv)
        _mix_np(xv, tv)
        out[pos:pos + n] = fn(xv)
        pos += n
        i += n
    return out


def hash_np(stream: int, start: int, count: int) -> np.ndarray:
    """32-bit hashes of element indices [start, start+count) of a stream (uint32 array)."""
    return _generate(stream, start, count, np.empty(count, np.uint32), lambda h: h)


def hash_torch(stream: int, start: int, count: int, device):
    """Device twin of :func:`hash_np` using int64 torch ops (identical values)."""
    import torch
    out = torch.empty(count, dtype=torch.int64, device=device)
    i = start
    pos = 0
    while pos < count:
        hi = i >> 32
        lo = i & MASK32
        n = min(count - pos, (1 << 32) - lo)
        k1, k2 = _keys(stream, hi)
        x = torch.arange(lo, lo + n, dtype=torch.int64, device=device)
        for k in (k1, k2):
            x = x ^ k
            x = (((x >> 16) ^ x) * _M) & MASK32
            x = (((x >> 16) ^ x) * _M) & MASK32
            x = (x >> 16) ^ x
        out[pos:pos + n] = x
        pos += n
        i += n
    return out


# --------------------------------------------------------------------------
# value tables
# --------------------------------------------------------------------------
def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even) and return the 16-bit patterns."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


@functools.lru_cache(maxsize=None)
def _quantiles() -> np.ndarray:
    from scipy.special import ndtri
    k = np.arange(65536, dtype=np.float64)
    return ndtri((k + 0.5) / 65536.0)


@functools.lru_cache(maxsize=None)
def normal_table_bf16(sigma: float = 1.0) -> np.ndarray:
    """uint16 bf16 patterns of sigma * Phi^-1((k+0.5)/65536), k = 0..65535."""
    v = (_quantiles() * float(sigma)).astype(np.float32)   # float64 -> float32 (RNE)
    return _f32_to_bf16_bits(v)                             # float32 -> bf16 (RNE)


@functools.lru_cache(maxsize=None)
def normal_table_f32(sigma: float = 1.0) -> np.ndarray:
    return (_quantiles() * float(sigma)).astype(np.float32)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# samplers
# --------------------------------------------------------------------------
def _lookup(table: np.ndarray):
    return lambda h: table.take((h >> _S16).astype(np.intp))


def normal_bf16(stream: int, start: int, count: int, sigma: float = 1.0) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0, sigma^2) samples."""
    return _generate(stream, start, count, np.empty(count, np.uint16), _lookup(normal_table_bf16(sigma)))


def normal_f32(stream: int, start: int, count: int, sigma: float = 1.0) -> np.ndarray:
    return _generate(stream, start, count, np.empty(count, np.float32), _lookup(normal_table_f32(sigma)))


def uniform_f32(stream: int, start: int, count: int) -> np.ndarray:
    h = hash_np(stream, start, count)
    return (((h >> np.uint32(9)).astype(np.float64) + 0.5) * 2.0 ** -23).astype(np.float32)


def normal_bf16_torch(stream: int, start: int, count: int, device, sigma: float = 1.0):
    """Device twin of :func:`normal_bf16`: returns a torch.bfloat16 tensor."""
    import torch
    tab = torch.from_numpy(normal_table_bf16(sigma).astype(np.int16)).to(device)
    h = hash_torch(stream, start, count, device)
    return tab[h >> 16].view(torch.bfloat16)


def normal_f32_torch(stream: int, start: int, count: int, device, sigma: float = 1.0):
    import torch
    tab = torch.from_numpy(normal_table_f32(sigma)).to(device)
    h = hash_torch(stream, start, count, device)
    return tab[h >> 16]


def uniform_f32_torch(stream: int, start: int, count: int, device):
    import torch
    h = hash_torch(stream, start, count, device)
    # (h >> 9) < 2**23, so the float conversion and the two steps below are exact
    return ((h >> 9).to(torch.float32) + 0.5) * (2.0 ** -23)
