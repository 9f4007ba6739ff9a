"""Seeded counter-based synthetic inputs, identical on the host and on the device.

Every element of every synthetic tensor is a pure function of (seed, tensor name,
flat element index), so any slice of any tensor can be drawn without drawing the rest
(the oracle draws just the sequences it checks) and the host (torch CPU) and the
device (torch CUDA) produce bit-identical values:

* hash: the SplitMix64 finalizer (Steele, Lea & Flood, "Fast splittable pseudorandom
  number generators", OOPSLA 2014) applied to ``key + index * golden``, all in
  wrapping 64-bit integer arithmetic;
* "normal" values: centred sum of the four 16-bit lanes of the hash (Irwin-Hall, n=4),
  an exact integer, scaled to unit variance by one fp32 multiply, then one fp32
  multiply by the std and one fp32 add of the mean, then round-to-nearest-even to
  the storage dtype; every step is an exactly specified IEEE operation, so the
  result does not depend on the device;
* uniforms in [0, 1): the top 24 bits of the hash times 2^-24 (exact in fp32);
* integers in [lo, hi]: lo + (hash >> 1) mod (hi - lo + 1).

This module holds none of the drafter's arithmetic; it is shared by the oracle side
and the CUDA side only as an input source.
"""
from __future__ import annotations

import math
import zlib

import torch

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
IH4_STD = math.sqrt(4.0 * (65536.0 ** 2 - 1.0) / 12.0)
IH4_MEAN = 2 * 65535
CHUNK = 1 << 20


def _s64(c: int) -> int:
    c &= MASK64
    return c - (1 << 64) if c >= (1 << 63) else c


def mix64_int(z: int) -> int:
    """SplitMix64 finalizer on a Python int (exact reference)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def _srl(z: torch.Tensor, s: int) -> torch.Tensor:
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix64_(z: torch.Tensor) -> torch.Tensor:
    """SplitMix64 finalizer, in place on an int64 tensor (wrapping arithmetic)."""
    t = torch.empty_like(z)
    for s, m in ((30, _s64(MIX1)), (27, _s64(MIX2)), (31, None)):
        torch.bitwise_right_shift(z, s, out=t)
        t.bitwise_and_((1 << (64 - s)) - 1)
        z.bitwise_xor_(t)
        if m is not None:
            z.mul_(m)
    return z


def stream_key(seed: int, name: str) -> int:
    return mix64_int((seed * GOLDEN + zlib.crc32(name.encode())) & MASK64)


def hash_at(seed: int, name: str, idx: torch.Tensor) -> torch.Tensor:
    """64-bit hash (as int64) of flat indices ``idx`` (int64 tensor)."""
    key = _s64(stream_key(seed, name))
    return _mix64_(idx * _s64(GOLDEN) + key)


def _normal_from_hash(h, std, mean, dtype):
    s = h.bitwise_and(0xFFFF)
    t = torch.empty_like(h)
    for sh in (16, 32, 48):
        torch.bitwise_right_shift(h, sh, out=t)
        t.bitwise_and_(0xFFFF)
        s.add_(t)
    s.sub_(IH4_MEAN)
    v = s.to(torch.float32)
    scale = torch.tensor(std / IH4_STD, dtype=torch.float32, device=h.device)
    z = v * scale
    if mean != 0.0:
        z = z + torch.tensor(mean, dtype=torch.float32, device=h.device)
    return z.to(dtype)


def normal_flat(seed, name, start, stop, std=1.0, mean=0.0, dtype=torch.float32,
                device="cpu") -> torch.Tensor:
    """Elements [start, stop) of the flat stream ``name``, 1-D."""
    n = stop - start
    out = torch.empty(n, dtype=dtype, device=device)
    chunk = CHUNK if torch.device(device).type == "cpu" else CHUNK << 6
    for c0 in range(0, n, chunk):
        c1 = min(n, c0 + chunk)
        idx = torch.arange(start + c0, start + c1, dtype=torch.int64, device=device)
        out[c0:c1] = _normal_from_hash(hash_at(seed, name, idx), std, mean, dtype)
    return out


def normal(seed, name, shape, std=1.0, mean=0.0, dtype=torch.float32, device="cpu",
           rows=None) -> torch.Tensor:
    """Tensor of logical shape ``shape``; ``rows=(r0, r1)`` draws only those leading
    rows (flat indices follow the full logical shape)."""
    shape = tuple(shape)
    inner = math.prod(shape[1:]) if len(shape) > 1 else 1
    r0, r1 = rows if rows is not None else (0, shape[0])
    flat = normal_flat(seed, name, r0 * inner, r1 * inner, std, mean, dtype, device)
    return flat.view((r1 - r0,) + shape[1:])


def uniform(seed, name, shape, device="cpu") -> torch.Tensor:
    n = math.prod(shape)
    idx = torch.arange(n, dtype=torch.int64, device=device)
    h = hash_at(seed, name, idx)
    u = _srl(h, 40).to(torch.float32) * (2.0 ** -24)
    return u.view(tuple(shape))


def integers(seed, name, shape, lo, hi, device="cpu") -> torch.Tensor:
    n = math.prod(shape)
    idx = torch.arange(n, dtype=torch.int64, device=device)
    h = hash_at(seed, name, idx)
    return (lo + _srl(h, 1) % (hi - lo + 1)).view(tuple(shape))


def permutation(seed, name, n) -> torch.Tensor:
    """A seeded permutation of range(n) (host): stable argsort of hash values."""
    h = hash_at(seed, name, torch.arange(n, dtype=torch.int64))
    return torch.argsort(_srl(h, 1), stable=True)
