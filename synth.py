"""Seeded synthetic inputs for the quantized GEMV workloads.

This module is the only code that the CUDA path and the CPU oracle both use.
It holds random-number generation and plain storage conversions only -- none
of the formats' arithmetic (no quantizing, no packing, no decoding, no
rotation).

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), evaluated counter-style: element k of
stream ``seed`` is mix(seed + (k + 1) * 0x9E3779B97F4A7C15).  Normal deviates
come from the Box-Muller transform (Box and Muller, 1958) on consecutive
pairs of uniforms.  Everything is vectorised numpy, split into chunks that
run on a thread pool (numpy releases the GIL inside its ufuncs).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22
_THREADS = max(1, min(16, os.cpu_count() or 1))


def _splitmix64(seed: int, start: int, n: int) -> np.ndarray:
    k = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + k * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _chunked(fn, n: int, dtype) -> np.ndarray:
    out = np.empty(n, dtype)
    starts = list(range(0, n, _CHUNK))

    def run(s):
        e = min(n, s + _CHUNK)
        out[s:e] = fn(s, e - s)

    if len(starts) <= 1:
        for s in starts:
            run(s)
    else:
        with ThreadPoolExecutor(_THREADS) as ex:
            list(ex.map(run, starts))
    return out


def uint64(seed: int, n: int) -> np.ndarray:
    """n raw 64-bit SplitMix64 outputs of stream ``seed``."""
    return _chunked(lambda s, m: _splitmix64(seed, s, m), n, np.uint64)


def uniform(seed: int, n: int) -> np.ndarray:
    """n float64 uniforms in [0, 1) (top 53 bits of each output)."""
    return _chunked(lambda s, m: (_splitmix64(seed, s, m) >> np.uint64(11)).astype(np.float64)
                    * (1.0 / 9007199254740992.0), n, np.float64)


def normal(seed: int, n: int, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    """n float32 samples of N(mean, std^2) by Box-Muller on uniform pairs."""
    def gen(s, m):
        # element k uses uniforms 2*(k//2) and 2*(k//2)+1 of the stream
        p0 = s // 2
        npairs = (s + m + 1) // 2 - p0
        u = _splitmix64(seed, 2 * p0, 2 * npairs)
        u1 = ((u[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)
        u2 = (u[1::2] >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
        r = np.sqrt(-2.0 * np.log(u1))
        z = np.empty(2 * npairs, np.float64)
        z[0::2] = r * np.cos(2.0 * np.pi * u2)
        z[1::2] = r * np.sin(2.0 * np.pi * u2)
        off = s - 2 * p0
        return (mean + std * z[off:off + m]).astype(np.float32)
    return _chunked(gen, n, np.float32)


def log_uniform(seed: int, n: int, lo: float, hi: float) -> np.ndarray:
    """n float32 values whose logarithm is uniform on [log lo, log hi)."""
    a, b = np.log(lo), np.log(hi)
    return np.exp(a + (b - a) * uniform(seed, n)).astype(np.float32)


def bytes_excluding(seed: int, n: int, excluded=(0x7F, 0xFF)) -> np.ndarray:
    """n bytes uniform over 0..255 minus ``excluded`` (uint8)."""
    allowed = np.array([b for b in range(256) if b not in set(excluded)], np.uint8)

    def gen(s, m):
        u = _splitmix64(seed, s, m) >> np.uint64(32)
        return allowed[(u % np.uint64(len(allowed))).astype(np.int64)]
    return _chunked(gen, n, np.uint8)


def signs(seed: int, n: int) -> np.ndarray:
    """n signs in {+1, -1} (int8) from the top bit of each output."""
    return np.where((uint64(seed, n) >> np.uint64(63)) == 0, 1, -1).astype(np.int8)


def bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns the uint16 bits.

    Plain storage conversion: bfloat16 is the top half of a binary32.
    """
    u = np.ascontiguousarray(v, np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    with np.errstate(over="ignore"):
        r = (u + bias) >> np.uint32(16)
    nan = np.isnan(np.asarray(v, np.float32))
    r = np.where(nan, (u >> np.uint32(16)) | np.uint32(0x40), r)
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bits to float32 (exact)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------
# Workload recipes (shapes and distributions of the decode/prefill workloads)
# --------------------------------------------------------------------------

def seeds(tag: int):
    """(weight seed, activation seed) for workload ``tag``."""
    return 1000 + tag, 2000 + tag


SIGN_SEED = 42  # seed of the 256-entry FWHT sign vector


def fmt4_raw(O: int, I: int, S: int, tag: int):
    """f32 weights N(0, 0.02^2) [O, I] and f32 activations N(0, 1) [S, I]."""
    ws, xs = seeds(tag)
    return normal(ws, O * I, 0.02).reshape(O, I), normal(xs, S * I).reshape(S, I)


def fmt7_raw(O: int, I: int, S: int, tag: int):
    """e4m3 codes [O, I] (uniform, NaN codes excluded), f32 block scales
    log-uniform in [1e-4, 1e-2] [ceil(O/128), ceil(I/128)], bf16 activations
    N(0, 1) [S, I] (uint16 bits)."""
    ws, xs = seeds(tag)
    nbo, nbi = (O + 127) // 128, (I + 127) // 128
    codes = bytes_excluding(ws, O * I).reshape(O, I)
    scales = log_uniform(ws + 500, nbo * nbi, 1e-4, 1e-2).reshape(nbo, nbi)
    x = bf16_bits(normal(xs, S * I)).reshape(S, I)
    return codes, scales, x


def mq4_raw(O: int, I: int, S: int, tag: int):
    """Unrotated f32 weights N(0, 0.02^2) [O, I], f32 activations N(0, 1)
    [S, I] and the 256 FWHT signs; the caller rotates both with the same
    signs before encoding the weights and rounding x to bf16."""
    ws, xs = seeds(tag)
    return (normal(ws, O * I, 0.02).reshape(O, I), normal(xs, S * I).reshape(S, I),
            signs(SIGN_SEED, 256))
