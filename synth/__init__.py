"""Seeded synthetic inputs shared by the tests and the benchmark.

The generator (``synth.c``) is counter based: value i of stream ``seed`` depends
only on ``(seed, i)``. It draws numbers and nothing else; the CUDA library and
the CPU oracle both receive the bytes it writes.

Conventions used by the tests and the benchmark:
  * ``normal(seed, shape, dtype, std)``: Box-Muller normals, 0.02 means a
    standard deviation of 0.02;
  * ``uniform(seed, shape, dtype, lo, hi)``: uniform on [lo, hi);
  * partial k of a P-sum uses seed ``base + k``.
bf16 tensors are returned as numpy ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "_synth.so")
_lib = None

F32, BF16, F64 = 0, 1, 2
_NP = {F32: np.float32, BF16: np.uint16, F64: np.float64}
_NAMES = {"f32": F32, "float32": F32, "bf16": BF16, "bfloat16": BF16, "f64": F64}


def build(force: bool = False) -> str:
    """Compile the generator into a shared library next to its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp, "-lpthread", "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.synth_fill.restype = ctypes.c_int
        lib.synth_fill.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_uint64, ctypes.c_double,
                                   ctypes.c_double, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int]
        _lib = lib
    return _lib


def _code(dtype) -> int:
    if isinstance(dtype, str):
        return _NAMES[dtype]
    return int(dtype)


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def fill(kind: str, seed: int, n: int, dtype, ptr: int, a: float, b: float) -> None:
    """Write n draws to raw host memory at ``ptr`` (used for pinned buffers)."""
    k = 0 if kind == "normal" else 1
    rc = _load().synth_fill(k, _code(dtype), seed & (2**64 - 1), a, b, n, ptr, _threads())
    if rc != 0:
        raise ValueError("synth_fill rejected its arguments")


def normal(seed: int, shape, dtype="f32", std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    code = _code(dtype)
    out = np.empty(tuple(shape), dtype=_NP[code])
    fill("normal", seed, out.size, code, out.ctypes.data, mean, std)
    return out


def uniform(seed: int, shape, dtype="f32", lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    code = _code(dtype)
    out = np.empty(tuple(shape), dtype=_NP[code])
    fill("uniform", seed, out.size, code, out.ctypes.data, lo, hi)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)
