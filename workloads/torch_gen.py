"""The generators of ``workloads.rng`` written with torch tensor ops, for any device.

Same definitions, same bits: SplitMix64 outputs (64-bit wrapping arithmetic on
int64 tensors, logical shifts by masking), 53-bit uniforms, the cosine branch of
Box-Muller in float64, float64 -> float32 -> bf16 round-to-nearest-even.  Used
to fill gigabyte-sized synthetic pools directly in device memory; tests check
that it reproduces the numpy stream bit for bit.  Holds none of the method's
arithmetic.
"""
from __future__ import annotations

import math

import torch


def _s64(x: int) -> int:
    x &= 0xFFFFFFFFFFFFFFFF
    return x - (1 << 64) if x >= (1 << 63) else x


_GAMMA = _s64(0x9E3779B97F4A7C15)
_M1 = _s64(0xBF58476D1CE4E5B9)
_M2 = _s64(0x94D049BB133111EB)
_TWO_M53 = 2.0 ** -53
_CHUNK = 1 << 25


def _lsr(z: torch.Tensor, k: int) -> torch.Tensor:
    return (z >> k) & ((1 << (64 - k)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = z ^ _lsr(z, 30)
    z = z * _M1
    z = z ^ _lsr(z, 27)
    z = z * _M2
    return z ^ _lsr(z, 31)


def splitmix64(key: int, start: int, count: int, device) -> torch.Tensor:
    j = torch.arange(start + 1, start + 1 + count, dtype=torch.int64, device=device)
    return _mix(_s64(key) + j * _GAMMA)


def uniform(key: int, start: int, count: int, device) -> torch.Tensor:
    return _lsr(splitmix64(key, start, count, device), 11).to(torch.float64) * _TWO_M53


def _normal(key: int, start: int, count: int, device) -> torch.Tensor:
    z = splitmix64(key, 2 * start, 2 * count, device)
    u1 = (_lsr(z[0::2], 11).to(torch.float64) + 1.0) * _TWO_M53
    u2 = _lsr(z[1::2], 11).to(torch.float64) * _TWO_M53
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos(2.0 * math.pi * u2)


def f64_to_bf16(x: torch.Tensor) -> torch.Tensor:
    """float64 -> bf16 tensor, via float32, both steps round-to-nearest-even (explicit bit rounding)."""
    u = x.to(torch.float32).view(torch.int32).to(torch.int64) & 0xFFFFFFFF
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) & 0xFFFF
    r = torch.where(r >= 0x8000, r - 0x10000, r)
    return r.to(torch.int16).view(torch.bfloat16)


def normal_bf16(key: int, start: int, count: int, device, spike_key: int | None = None,
                spike_prob: float = 0.0, spike_factor: float = 8.0, out: torch.Tensor | None = None) -> torch.Tensor:
    """bf16 tensor of N(0, 1) draws for indices start .. start+count-1 (same bits as rng.normal_bf16)."""
    if out is None:
        out = torch.empty(count, dtype=torch.bfloat16, device=device)
    for lo in range(0, count, _CHUNK):
        n = min(_CHUNK, count - lo)
        x = _normal(key, start + lo, n, device)
        if spike_key is not None and spike_prob > 0.0:
            hit = uniform(spike_key, start + lo, n, device) < spike_prob
            x = torch.where(hit, x * spike_factor, x)
        out[lo:lo + n] = f64_to_bf16(x)
    return out


def workload_kv(wl, layer: int, device, seqs=None, upto_offset: int = 0):
    """K, V (bf16 [n, kv_heads, head_dim]) and slot mapping (int32 [n]) of every token of ``wl``'s
    sequences at ``layer``, generated on ``device`` - the same values as ``wl.kv_tokens``."""
    import numpy as np

    chosen = range(wl.num_seqs) if seqs is None else seqs
    spans, slots = [], []
    for s in chosen:
        n = int(wl.context_lens[s]) - upto_offset
        if n <= 0 or not wl.has_pages(s):
            continue
        spans.append((s, n))
        slots.append(wl.slot_mapping(s, layer, 0, n))
    total = sum(n for _, n in spans)
    te = wl.token_elems
    k = torch.empty(total * te, dtype=torch.bfloat16, device=device)
    v = torch.empty(total * te, dtype=torch.bfloat16, device=device)
    off = 0
    # Consecutive sequences of a layer occupy consecutive stream ranges only when
    # each has max_context tokens, so generate per sequence.
    for s, n in spans:
        base = wl._token_index(layer, s, 0)
        normal_bf16(wl.keys["k"], base, n * te, device, spike_key=wl.keys["spike"], spike_prob=wl.spike_prob,
                    out=k[off * te:(off + n) * te])
        normal_bf16(wl.keys["v"], base, n * te, device, out=v[off * te:(off + n) * te])
        off += n
    slot = torch.from_numpy(np.concatenate(slots) if slots else np.zeros(0, np.int32)).to(device)
    shape = (total, wl.num_kv_heads, wl.head_dim)
    return k.view(shape), v.view(shape), slot


def workload_q(wl, layer: int, device) -> torch.Tensor:
    n = wl.num_seqs * wl.num_q_heads * wl.head_dim
    return normal_bf16(wl.keys["q"], layer * n, n, device).view(wl.num_seqs, wl.num_q_heads, wl.head_dim)


