"""Seeded synthetic inputs for the sparse top-k MoE FFN layer.

This module is shared by the tests, the oracle side and the benchmark. It holds
no arithmetic of the layer itself (no router, softmax, top-k, FFN or combine):
it only turns (seed, tensor stream, draw attempt, element index) into numbers.

Generator
---------
Every element is a function of its flat row-major index ``i`` alone, so any
slice (one token row, one expert's weight matrix) can be produced on its own,
on the host with numpy or on the device with ``inputgen/fill.cu``; the two give
bit-identical values.

* Uniform bits: SplitMix64 (Steele, Lea and Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014), finaliser constants of
  Stafford's "Mix13". Element ``i`` of a stream with key ``K`` uses the three
  64-bit outputs ``mix64(K + (3*i + m + 1) * GAMMA)``, ``m = 0, 1, 2``.
* Normal deviate: the Irwin-Hall sum of twelve uniforms minus six, which has
  mean 0 and variance 1. The twelve uniforms are the 16-bit fields of the three
  outputs, ``u = (v + 1/2) / 2**16``; the sum is an integer over ``2**16`` and
  is exact in fp32 (|numerator| < 2**20).
* Scaling: one IEEE fp32 multiply by ``sigma`` (round to nearest even), then,
  for bf16 tensors, one round-to-nearest-even to bf16.

The layer's workloads (x ~ N(0,1), weights ~ N(0, 1/fan_in)) take sigma = 1 and
sigma = fp32(1/sqrt(fan_in)).
"""
from __future__ import annotations

import ctypes
import os
import math

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
MIX_M1 = 0xBF58476D1CE4E5B9
MIX_M2 = 0x94D049BB133111EB

# Tensor streams of one layer instance. A re-drawn token row keeps its stream and
# flat indices and bumps the draw attempt.
STREAM_X = 1
STREAM_WR = 2
STREAM_W1 = 3
STREAM_W2 = 4

DTYPE_F32 = 0
DTYPE_BF16 = 1


def mix64_int(z: int) -> int:
    """SplitMix64 finaliser on a Python int (mod 2**64)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX_M1) & MASK64
    z = ((z ^ (z >> 27)) * MIX_M2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int, attempt: int = 0) -> int:
    """64-bit key of one tensor stream; distinct (seed, stream, attempt) give unrelated keys."""
    if not (0 <= stream < 2**31 and 0 <= attempt < 2**32 and seed >= 0):
        raise ValueError("stream_key: out-of-range seed/stream/attempt")
    return mix64_int(mix64_int(seed + GAMMA) ^ mix64_int((stream << 32) | attempt))


def _mix64_np(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX_M1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX_M2)
    return z ^ (z >> np.uint64(31))


def sigma_for_fan_in(fan_in: int) -> np.float32:
    """fp32 standard deviation 1/sqrt(fan_in), rounded once from fp64."""
    return np.float32(1.0 / math.sqrt(fan_in))


def normal_f32(start: int, count: int, key: int, sigma) -> np.ndarray:
    """Elements ``start .. start+count-1`` of a stream, as fp32 (before any bf16 rounding)."""
    sigma = np.float32(sigma)
    out = np.empty(count, np.float32)
    chunk = 1 << 20
    with np.errstate(over="ignore"):
        for c0 in range(0, count, chunk):
            n = min(chunk, count - c0)
            i = np.arange(start + c0, start + c0 + n, dtype=np.uint64)
            acc = np.zeros(n, np.int64)
            for m in range(3):
                ctr = np.uint64(key) + (np.uint64(3) * i + np.uint64(m + 1)) * np.uint64(GAMMA)
                h = _mix64_np(ctr)
                for s in (0, 16, 32, 48):
                    acc += ((h >> np.uint64(s)) & np.uint64(0xFFFF)).astype(np.int64)
            z = (acc + 6 - 393216).astype(np.float32) * np.float32(1.0 / 65536.0)
            out[c0:c0 + n] = z * sigma
    return out


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the uint16 bit patterns. No NaNs expected."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns, as fp64."""
    return (np.asarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def draw(start: int, count: int, key: int, sigma, dtype: int) -> np.ndarray:
    """Host draw: fp32 values, or uint16 bf16 bit patterns when ``dtype == DTYPE_BF16``."""
    v = normal_f32(start, count, key, sigma)
    return f32_to_bf16_bits(v) if dtype == DTYPE_BF16 else v


def as_f64(a: np.ndarray, dtype: int) -> np.ndarray:
    """Exact fp64 value of a host draw (bf16 bits or fp32)."""
    return bf16_bits_to_f64(a) if dtype == DTYPE_BF16 else np.asarray(a, np.float64)


def skew_bias(E: int, c: float) -> np.ndarray:
    """Per-expert router bias c*log((e+1)**-1.2) (expert e has popularity rank e+1), fp32."""
    e = np.arange(E, dtype=np.float64)
    return (c * (-1.2) * np.log(e + 1.0)).astype(np.float32)


# ----------------------------------------------------------------------------- device fill

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libinputgen.so")
        if not os.path.exists(path):
            raise RuntimeError(f"inputgen: {path} not built (run __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        lib.inputgen_fill_normal.restype = ctypes.c_int
        lib.inputgen_fill_normal.argtypes = [
            ctypes.c_void_p, ctypes.c_longlong, ctypes.c_longlong, ctypes.c_ulonglong,
            ctypes.c_float, ctypes.c_int, ctypes.c_void_p]
        _LIB = lib
    return _LIB


def fill_device(tensor, start: int, key: int, sigma, dtype: int, stream_handle: int = 0) -> None:
    """Fill a contiguous CUDA tensor with elements ``start ..`` of a stream (same values as ``draw``)."""
    n = tensor.numel()
    rc = _lib().inputgen_fill_normal(ctypes.c_void_p(tensor.data_ptr()), n, start, key,
                                     float(np.float32(sigma)), dtype, ctypes.c_void_p(stream_handle))
    if rc != 0:
        raise RuntimeError(f"inputgen_fill_normal failed with CUDA error {rc}")
