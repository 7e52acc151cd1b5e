"""Counter-based seeded random numbers for the synthetic workloads.

Nothing here computes attention, paging or any other step of the method: it only
draws numbers.  Both the CUDA path's tests/bench and the CPU oracle take their
inputs from this module, so the two sides see the same bits.

Generators used (named published methods, written from their definitions):

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): output j of a stream keyed by ``key`` is
  ``mix(key + (j + 1) * 0x9E3779B97F4A7C15)`` with the 64-bit finaliser
  ``z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB;
  z ^= z >> 31``.  Being counter-based, any index range can be regenerated on its
  own, which lets a test rebuild only the sequences it samples.
* 53-bit uniforms: ``(z >> 11) * 2**-53`` in [0, 1); the "open at zero" variant
  ``((z >> 11) + 1) * 2**-53`` in (0, 1].
* Box-Muller (Box and Muller, 1958): ``n = sqrt(-2 ln u1) * cos(2 pi u2)`` with
  u1 from output 2i (open at zero) and u2 from output 2i+1 of the stream; only the
  cosine branch is kept so that element i depends on two counter values alone.
* BF16 rounding: float64 -> float32 (IEEE round-to-nearest-even) -> bfloat16 by
  round-to-nearest-even on the upper 16 bits.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_TWO_M53 = float(2.0 ** -53)

# Work is split into chunks of this many elements and spread over host threads
# (ctypes releases the GIL during the C calls), so gigabyte-sized pools generate
# in seconds.
_CHUNK = 1 << 22


def stream_key(seed: int, tag: str) -> int:
    """64-bit key of the stream named ``tag`` under ``seed`` (FNV-1a of the tag, mixed)."""
    h = 0xCBF29CE484222325
    for b in tag.encode():
        h ^= b
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    k = np.array([(seed * 0x9E3779B97F4A7C15 + h) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return int(_mix(k)[0])


def _mix(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * _M1
    z = z ^ (z >> np.uint64(27))
    z = z * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(key: int, start: int, count: int) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of the SplitMix64 stream keyed by ``key``."""
    j = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(np.uint64(key) + j * _GAMMA)


def uniform(key: int, start: int, count: int) -> np.ndarray:
    """53-bit uniforms in [0, 1) for indices ``start .. start+count-1``."""
    return (splitmix64(key, start, count) >> np.uint64(11)).astype(np.float64) * _TWO_M53


def _normal_chunk(key: int, start: int, count: int) -> np.ndarray:
    z = splitmix64(key, 2 * start, 2 * count)
    u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * _TWO_M53
    u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * _TWO_M53
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def normal(key: int, start: int, count: int) -> np.ndarray:
    """float64 N(0, 1) draws for indices ``start .. start+count-1`` of stream ``key``."""
    return _normal_chunk(key, start, count)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 to bfloat16 (via float32, both steps round-to-nearest-even); uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float64."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


_FAST_SRC = os.path.join(os.path.dirname(os.path.abspath(__file__)), "fastgen.c")
_FAST_LIB = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfastgen.so")
_fast = None
_fast_lock = threading.Lock()


def build_fast(force: bool = False) -> str:
    """Compile the C version of the generator (same definitions) next to its source."""
    if force or not os.path.exists(_FAST_LIB) or os.path.getmtime(_FAST_LIB) < os.path.getmtime(_FAST_SRC):
        tmp = _FAST_LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-shared",
                               "-fPIC", "-o", tmp, _FAST_SRC, "-lm"])
        os.replace(tmp, _FAST_LIB)
    return _FAST_LIB


def _fast_lib():
    global _fast
    with _fast_lock:
        if _fast is None:
            L = ctypes.CDLL(build_fast())
            L.fastgen_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64,
                                              ctypes.c_double, ctypes.c_double, ctypes.c_int, ctypes.c_void_p]
            L.fastgen_normal_bf16.restype = None
            _fast = L
    return _fast


def normal_bf16_reference(key: int, start: int, count: int, spike_key: int | None = None,
                          spike_prob: float = 0.0, spike_factor: float = 8.0) -> np.ndarray:
    """The numpy definition of ``normal_bf16`` (slow; the C version must match it bit for bit)."""
    x = _normal_chunk(key, start, count)
    if spike_key is not None and spike_prob > 0.0:
        hit = uniform(spike_key, start, count) < spike_prob
        x = np.where(hit, x * spike_factor, x)
    return f64_to_bf16_bits(x)


def normal_bf16(key: int, start: int, count: int, threads: int | None = None,
                spike_key: int | None = None, spike_prob: float = 0.0,
                spike_factor: float = 8.0) -> np.ndarray:
    """N(0, 1) draws rounded to bf16 bits, for indices ``start .. start+count-1``.

    With ``spike_key`` set, element i is multiplied by ``spike_factor`` when
    ``uniform(spike_key, i) < spike_prob`` (an independent Bernoulli per element),
    before rounding.  Runs the C version of the definitions over host threads.
    """
    out = np.empty(count, dtype=np.uint16)
    threads = threads or min(16, os.cpu_count() or 1)
    lib = _fast_lib()
    use_spike = int(spike_key is not None and spike_prob > 0.0)

    def work(lo: int) -> None:
        n = min(_CHUNK, count - lo)
        lib.fastgen_normal_bf16(key, start + lo, n, spike_key or 0, float(spike_prob), float(spike_factor),
                                use_spike, out[lo:].ctypes.data)

    starts = list(range(0, count, _CHUNK))
    if len(starts) <= 1 or threads <= 1:
        for lo in starts:
            work(lo)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, starts))
    return out


def permutation(key: int, n: int) -> np.ndarray:
    """A uniformly random permutation of 0..n-1 (stable argsort of n uniforms)."""
    return np.argsort(uniform(key, 0, n), kind="stable").astype(np.int32)


def uniform_int(key: int, start: int, count: int, lo: int, hi: int) -> np.ndarray:
    """Integers uniform in the closed range [lo, hi]."""
    u = uniform(key, start, count)
    return (lo + np.floor(u * (hi - lo + 1))).astype(np.int64)
