"""Counter-based, device-independent generator of bf16 input bits.

Every draw is SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014): output ``n`` of a stream with state ``k`` is ``fmix(k + (n+1)*GAMMA)`` with the
published finaliser constants.  Only integer operations and one correctly rounded fp32 multiply
are used, so a tensor drawn on the CPU and one drawn on the GPU are bit-identical, and any single
element can be regenerated on the host on demand (used to check sampled outputs of full-size runs).

* ``uniform_int_bf16_bits``: integers uniform on ``[lo, hi]`` (one draw per element).
* ``normal_bf16_bits``: a N(0, sigma) stand-in.  Twelve 16-bit uniforms (three draws, four fields
  each) are summed (Irwin-Hall, n = 12), centred, scaled by ``fp32(sigma / 65536)`` in fp32 and
  rounded to bf16 with round-to-nearest-even.  No transcendental function is involved, so no
  libm/CUDA-math difference can change a bit.

The results are ``torch.int16`` tensors holding bf16 bit patterns (``.view(torch.bfloat16)``).
"""
from __future__ import annotations

from typing import List, Optional

import torch

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
SHARD_STREAM = 0xA11  # stream tag of the all-gather input shards
_CHUNK = 1 << 23


def _s64(x: int) -> int:
    """Python int -> the int64 value with the same low 64 bits."""
    x &= MASK64
    return x - (1 << 64) if x >= (1 << 63) else x


def fmix_int(z: int) -> int:
    """SplitMix64 finaliser on a Python int (reference form, used for keys and in tests)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def splitmix_int(key: int, n: int) -> int:
    """Output ``n`` (0-based) of the SplitMix64 sequence whose state starts at ``key``."""
    return fmix_int((key + (n + 1) * GAMMA) & MASK64)


def stream_key(seed: int, rank: int, stream: int) -> int:
    """State of the stream for (seed, rank, stream), as an unsigned 64-bit Python int."""
    k = fmix_int((seed + 1) * GAMMA)
    k = fmix_int(k ^ (((rank + 1) * GAMMA) & MASK64))
    return fmix_int(k ^ (((stream + 1) * GAMMA) & MASK64))


def _lsr(z: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 lanes holding unsigned 64-bit values."""
    return (z >> k) & ((1 << (64 - k)) - 1)


def _fmix(z: torch.Tensor) -> torch.Tensor:
    # int64 multiplication wraps modulo 2**64, i.e. it is the unsigned product's low 64 bits
    z = (z ^ _lsr(z, 30)) * _s64(MIX1)
    z = (z ^ _lsr(z, 27)) * _s64(MIX2)
    return z ^ _lsr(z, 31)


def _draw(key: int, n: torch.Tensor) -> torch.Tensor:
    """Outputs ``n`` (int64 tensor of 0-based positions) of the stream with state ``key``."""
    return _fmix((n + 1) * _s64(GAMMA) + _s64(key))


def _f32_to_bf16_bits(x: torch.Tensor) -> torch.Tensor:
    """fp32 -> bf16 bit pattern, round to nearest even (finite inputs only)."""
    b = x.view(torch.int32).to(torch.int64) & 0xFFFFFFFF
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    b = b - ((b >> 15) & 1) * 65536
    return b.to(torch.int16)


def _fill(numel: int, start: int, idx, device, fn) -> torch.Tensor:
    """Elements ``start .. start+numel-1`` of a stream, or the elements at positions ``idx``."""
    if idx is not None:
        idx = torch.as_tensor(idx, dtype=torch.int64).to(device)
        return fn(idx.reshape(-1)).reshape(idx.shape)
    out = torch.empty(numel, dtype=torch.int16, device=device)
    step = _CHUNK * (4 if out.is_cuda else 1)
    for a in range(0, numel, step):
        b = min(numel, a + step)
        i = torch.arange(start + a, start + b, dtype=torch.int64, device=out.device)
        out[a:b] = fn(i)
    return out


def uniform_int_bf16_bits(seed: int, rank: int, stream: int, numel: int, lo: int = -8, hi: int = 8,
                          device="cpu", start: int = 0, idx=None) -> torch.Tensor:
    """Integers uniform on ``[lo, hi]`` (inclusive), as bf16 bits; elements ``start .. start+numel-1``
    (or the positions in ``idx``)."""
    key = stream_key(seed, rank, stream)
    span = hi - lo + 1

    def fn(i):
        v = (_lsr(_draw(key, i), 32) % span + lo).to(torch.float32)
        return _f32_to_bf16_bits(v)

    return _fill(numel, start, idx, device, fn)


def normal_bf16_bits(seed: int, rank: int, stream: int, numel: int, sigma: float,
                     device="cpu", start: int = 0, idx=None) -> torch.Tensor:
    """N(0, sigma) stand-in (Irwin-Hall of twelve 16-bit uniforms) as bf16 bits."""
    key = stream_key(seed, rank, stream)
    scale = float(torch.tensor(sigma / 65536.0, dtype=torch.float32))

    def fn(i):
        k = torch.zeros_like(i)
        for j in range(3):
            h = _draw(key, 3 * i + j)
            k += (h & 0xFFFF) + (_lsr(h, 16) & 0xFFFF) + (_lsr(h, 32) & 0xFFFF) + _lsr(h, 48)
        z = (k - 393210).to(torch.float32)  # 12 * 65535 / 2 = 393210; |z| < 2**19, exact
        return _f32_to_bf16_bits(z * scale)

    return _fill(numel, start, idx, device, fn)


def grad_bits(g, r: int, p: int, device="cpu", start: int = 0, numel: Optional[int] = None,
              idx=None) -> torch.Tensor:
    """Gradient of parameter ``p`` on rank ``r`` of group ``g`` (flat, row-major), as bf16 bits
    (the whole tensor, a range from ``start``, or the positions ``idx``)."""
    n = g.numel(p) - start if numel is None else numel
    if g.grad_kind == "int":
        return uniform_int_bf16_bits(g.grad_seed_of(r), r, p, n, -8, 8, device=device, start=start, idx=idx)
    return normal_bf16_bits(g.grad_seed_of(r), r, p, n, g.grad_sigma, device=device, start=start, idx=idx)


def group_grads(g, device="cpu") -> List[List[torch.Tensor]]:
    """``grads[r][p]`` for the whole group, each a flat int16 tensor of bf16 bits."""
    return [[grad_bits(g, r, p, device) for p in range(g.P)] for r in range(g.R)]


def shard_bits(g, r: int, numel: int, device="cpu", start: int = 0, idx=None) -> torch.Tensor:
    """Packed all-gather input shard of rank ``r`` (``numel`` elements), N(0, shard_sigma) bits.

    Every element is drawn, padding positions included; a caller that wants a recognisable junk
    pattern in the padding overwrites those positions itself."""
    return normal_bf16_bits(g.shard_seed_of(r), r, SHARD_STREAM, numel, g.shard_sigma,
                            device=device, start=start, idx=idx)
