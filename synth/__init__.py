"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle runs.

This module holds no attention arithmetic.  It turns (seed, stream, shape) into
N(0, 1) samples with a counter-based generator, so that any element can be
produced independently of the others, on the CPU or on a CUDA device, with the
same integer stream on x86_64 and aarch64:

* counter generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014).  Output n of a stream is
  ``mix(key + (n + 1) * GAMMA)`` where ``mix`` is the SplitMix64 finaliser and
  ``key = mix(seed * GAMMA ^ stream)``.
* uniforms: the top 53 bits of an output, times 2**-53, in [0, 1).
* normals: Box-Muller on consecutive pairs: for pair p,
  ``r = sqrt(-2 ln(1 - u[2p]))``, ``theta = 2 pi u[2p+1]``,
  element 2p is ``r cos(theta)`` and element 2p+1 is ``r sin(theta)``.
  Computed in float64, rounded to float32 (round to nearest even), then to the
  requested storage dtype (bfloat16 uses round to nearest even as well).

Streams used by the attention workloads: q = 0, k = 1, v = 2; extra tensors
(row bounds, perturbations) take streams 3 and above.

The 64-bit arithmetic runs in torch int64, whose multiplication wraps modulo
2**64 on both CPU and CUDA; right shifts are made logical by masking.
"""
from __future__ import annotations

import math

import torch

_M64 = 1 << 64
GAMMA = 0x9E3779B97F4A7C15
_C1 = 0xBF58476D1CE4E5B9
_C2 = 0x94D049BB133111EB

STREAM_Q = 0
STREAM_K = 1
STREAM_V = 2
STREAM_AUX = 3
STREAM_DO = 5  # upstream gradient dO of the backward (4 is the paged pool's block shuffle)


def _s64(x: int) -> int:
    """Python int (taken modulo 2**64) -> the int64 with the same bits."""
    x %= _M64
    return x - _M64 if x >= (1 << 63) else x


def _mix_int(z: int) -> int:
    """SplitMix64 finaliser on a Python int (reference for the tensor version)."""
    z %= _M64
    z = ((z ^ (z >> 30)) * _C1) % _M64
    z = ((z ^ (z >> 27)) * _C2) % _M64
    return z ^ (z >> 31)


def _lsr(x: torch.Tensor, n: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return torch.bitwise_and(torch.bitwise_right_shift(x, n), (1 << (64 - n)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = torch.bitwise_xor(z, _lsr(z, 30)) * _s64(_C1)
    z = torch.bitwise_xor(z, _lsr(z, 27)) * _s64(_C2)
    return torch.bitwise_xor(z, _lsr(z, 31))


def stream_key(seed: int, stream: int) -> int:
    return _mix_int(((seed * GAMMA) % _M64) ^ stream)


def raw_u64(seed: int, stream: int, start: int, count: int, device="cpu") -> torch.Tensor:
    """Outputs start .. start+count-1 of a stream, as int64 bit patterns."""
    key = stream_key(seed, stream)
    n = torch.arange(start + 1, start + count + 1, dtype=torch.int64, device=device)
    return _mix(n * _s64(GAMMA) + _s64(key))


def uniform(seed: int, stream: int, start: int, count: int, device="cpu") -> torch.Tensor:
    """float64 uniforms in [0, 1) for outputs start .. start+count-1."""
    return _lsr(raw_u64(seed, stream, start, count, device), 11).to(torch.float64) * (2.0 ** -53)


_CHUNK = 1 << 24


def normal(shape, seed: int, stream: int, dtype=torch.float32, device="cpu") -> torch.Tensor:
    """N(0, 1) samples of the given shape, element i of the flattened tensor
    being the i-th Box-Muller output of (seed, stream)."""
    numel = 1
    for s in shape:
        numel *= int(s)
    out = torch.empty(numel, dtype=dtype, device=device)
    npairs = (numel + 1) // 2
    for p0 in range(0, npairs, _CHUNK):
        p1 = min(npairs, p0 + _CHUNK)
        u = uniform(seed, stream, 2 * p0, 2 * (p1 - p0), device).view(-1, 2)
        r = torch.sqrt(-2.0 * torch.log1p(-u[:, 0]))
        th = (2.0 * math.pi) * u[:, 1]
        z = torch.stack((r * torch.cos(th), r * torch.sin(th)), dim=1).reshape(-1)
        e0, e1 = 2 * p0, min(numel, 2 * p1)
        out[e0:e1] = z[: e1 - e0].to(torch.float32).to(dtype)
    return out.view(*shape)


def randint(count: int, high: int, seed: int, stream: int, device="cpu") -> torch.Tensor:
    """count integers uniform in [0, high) (floor(u * high))."""
    u = uniform(seed, stream, 0, count, device)
    return torch.clamp((u * high).floor().to(torch.int64), max=high - 1)


def empty_rows(B: int, Sq: int, fraction: float, seed: int, stream: int = STREAM_AUX):
    """Choose round(fraction * B * Sq) distinct (b, qi) pairs, seeded.

    Returns a sorted list of flat indices b * Sq + qi.  Selection is a partial
    Fisher-Yates shuffle driven by the stream's uniforms.
    """
    total = B * Sq
    n = int(round(fraction * total))
    u = uniform(seed, stream, 0, max(n, 1)).tolist()
    perm = {}
    picked = []
    for i in range(n):
        j = i + min(total - i - 1, int(u[i] * (total - i)))
        vi, vj = perm.get(i, i), perm.get(j, j)
        perm[i], perm[j] = vj, vi
        picked.append(vj)
    return sorted(picked)


def row_kv_bounds_with_empty_rows(B: int, Sq: int, Sk: int, fraction: float, seed: int,
                                  stream: int = STREAM_AUX) -> torch.Tensor:
    """int32 [B, Sq, 2] inclusive key bounds: [0, Sk-1] for every row except
    the chosen fraction, which get the empty range [1, 0]."""
    rb = torch.empty(B, Sq, 2, dtype=torch.int32)
    rb[..., 0] = 0
    rb[..., 1] = Sk - 1
    for f in empty_rows(B, Sq, fraction, seed, stream):
        b, qi = divmod(f, Sq)
        rb[b, qi, 0] = 1
        rb[b, qi, 1] = 0
    return rb


def alibi_slopes(Hq: int) -> torch.Tensor:
    """fp32 slopes 2^(-8 (h+1) / Hq), h = 0 .. Hq-1 (the geometric ALiBi family)."""
    h = torch.arange(1, Hq + 1, dtype=torch.float64)
    return torch.exp2(-8.0 * h / Hq).to(torch.float32)
