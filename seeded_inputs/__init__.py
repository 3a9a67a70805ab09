"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and the bench.

This module holds no attention arithmetic: it only turns (seed, stream, index) into
numbers. Both sides of every parity check read the same arrays from here, so the CPU
oracle and the CUDA kernels see identical bits.

Generator (a published, counter-based definition, restated here):

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
  OOPSLA 2014): the n-th output of a stream with state ``s0`` is
  ``mix64(s0 + (n + 1) * 0x9E3779B97F4A7C15)`` with
  ``z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31``
  (all arithmetic mod 2**64).
* Uniforms on (0, 1]: the top 53 bits, ``((x >> 11) + 1) * 2**-53``.
* Normals: Box-Muller in double, ``r = sqrt(-2 ln u1)``, element 2i gets ``r cos(2 pi u2)`` and
  element 2i+1 gets ``r sin(2 pi u2)``, where (u1, u2) come from counters (2i, 2i+1).
* The double result is rounded to float32 (round to nearest even). For bf16/fp16 tensors
  the float32 value is rounded again to nearest even. Every stored value is therefore the
  exact value the device reads; widening it to float32 or float64 is exact.

The stream state of tensor ``stream`` under ``seed`` is ``mix64(seed * 2**16 + stream)``, so
q, k and v (streams 0, 1, 2) are independent. Arrays are produced in chunks to bound memory.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

STREAM_Q, STREAM_K, STREAM_V = 0, 1, 2


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def stream_state(seed: int, stream: int) -> np.uint64:
    s = np.array([(int(seed) * 65536 + int(stream)) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return _mix64(s)[0]


def splitmix64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of one SplitMix64 stream, as uint64."""
    s0 = stream_state(seed, stream)
    n = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = s0 + n * _GAMMA
    return _mix64(z)


def uniform01(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Doubles on (0, 1] from the top 53 bits of each SplitMix64 output."""
    x = splitmix64(seed, stream, start, count)
    return ((x >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


_HERE = os.path.dirname(os.path.abspath(__file__))
_GEN_SRC = os.path.join(_HERE, "gen.c")
_GEN_LIB = os.path.join(_HERE, "_build", "libseeded_inputs.so")
_gen_lock = threading.Lock()
_gen = None


def _gen_lib():
    """The C implementation of the same generator (gen.c), compiled with gcc on first use."""
    global _gen
    with _gen_lock:
        if _gen is None:
            os.makedirs(os.path.dirname(_GEN_LIB), exist_ok=True)
            if not os.path.exists(_GEN_LIB) or os.path.getmtime(_GEN_LIB) < os.path.getmtime(_GEN_SRC):
                tmp = _GEN_LIB + f".{os.getpid()}.tmp"
                subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                                "-o", tmp, _GEN_SRC, "-lm"], check=True)
                os.replace(tmp, _GEN_LIB)
            lib = ctypes.CDLL(_GEN_LIB)
            lib.si_normal_f32.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                                          ctypes.POINTER(ctypes.c_float), ctypes.c_int]
            lib.si_normal_f32.restype = ctypes.c_int
            _gen = lib
    return _gen


def normal_f32(seed: int, stream: int, count: int) -> np.ndarray:
    """``count`` i.i.d. N(0, 1) samples rounded to float32 (Box-Muller, both branches).

    Runs the C implementation on all host cores; :func:`normal_f32_numpy` is the same
    definition in numpy, kept as its cross-check.
    """
    out = np.empty(count, dtype=np.float32)
    if count == 0:
        return out
    try:
        threads = max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        threads = os.cpu_count() or 1
    st = _gen_lib().si_normal_f32(int(seed) & 0xFFFFFFFFFFFFFFFF, int(stream), count,
                                  out.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), threads)
    if st != 0:
        raise RuntimeError("si_normal_f32 failed")
    return out


def normal_f32_numpy(seed: int, stream: int, count: int) -> np.ndarray:
    """The generator in numpy (the definition that ``gen.c`` implements)."""
    out = np.empty(count, dtype=np.float32)
    pairs = (count + 1) // 2
    done = 0
    while done < pairs:
        m = min(_CHUNK, pairs - done)
        u = uniform01(seed, stream, 2 * done, 2 * m).reshape(m, 2)
        r = np.sqrt(-2.0 * np.log(u[:, 0]))
        th = 2.0 * np.pi * u[:, 1]
        z = np.empty((m, 2), dtype=np.float64)
        z[:, 0] = r * np.cos(th)
        z[:, 1] = r * np.sin(th)
        lo = 2 * done
        hi = min(count, lo + 2 * m)
        out[lo:hi] = z.reshape(-1)[: hi - lo].astype(np.float32)
        done += m
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); returns the uint16 bit patterns.

    Inputs are finite, so no NaN handling is needed.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to the storage type and widen them back to float32 (exact)."""
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        return bf16_bits_to_f32(f32_to_bf16_bits(x))
    if dtype == "f16":
        return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).astype(np.float32)
    raise ValueError(f"unknown dtype {dtype!r}")


def qkv(seed: int, B: int, H: int, N: int, d: int, dtype: str = "f32", qk_scale: float = 1.0):
    """q, k, v of shape [B, H, N, d] as float32 arrays holding exactly the device values.

    ``qk_scale`` multiplies the generated float32 q and k before the storage rounding; the
    stress case uses 8.0, a power of two, so the product is exact.
    """
    shape = (B, H, N, d)
    count = B * H * N * d
    out = []
    for stream in (STREAM_Q, STREAM_K, STREAM_V):
        x = normal_f32(seed, stream, count)
        if stream != STREAM_V and qk_scale != 1.0:
            x = (x * np.float32(qk_scale)).astype(np.float32)
        out.append(round_to(x, dtype).reshape(shape))
    return tuple(out)


def spike_late(N: int, d: int):
    """Deterministic single-head pattern with no RNG (q, k, v as float32 [N, d]).

    Entries are small integers on fixed moduli times a step, and key N-3 is tripled so the
    running maximum still moves on the last key tile. This follows the input recipe of the
    attention.cu page ("Deterministic inputs with no exact binary values", makeInputs).
    """
    i = np.arange(N, dtype=np.int64)[:, None]
    e = np.arange(d, dtype=np.int64)[None, :]
    q = (((i * 31 + e * 7) % 97) - 48).astype(np.float32) * np.float32(0.021)
    k = (((i * 17 + e * 11) % 89) - 44).astype(np.float32) * np.float32(0.019)
    v = (((i * 13 + e * 5) % 83) - 41).astype(np.float32) * np.float32(0.011)
    if N >= 3:
        k[N - 3] = k[N - 3] * np.float32(3.0)
    return q.astype(np.float32), k.astype(np.float32), v.astype(np.float32)


def sample_rows(seed: int, N: int, count: int) -> np.ndarray:
    """Sorted distinct query rows: ``count`` drawn without replacement, plus rows 0 and N-1.

    Selection ranks rows by a SplitMix64 key on stream 7 and keeps the smallest keys.
    """
    if N <= 0:
        return np.zeros(0, dtype=np.int64)
    if count >= N:
        return np.arange(N, dtype=np.int64)
    keys = splitmix64(seed, 7, 0, N)
    pick = np.argpartition(keys, count)[:count]
    rows = np.union1d(pick.astype(np.int64), np.array([0, N - 1], dtype=np.int64))
    return rows
