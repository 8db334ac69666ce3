"""Seeded synthetic inputs (SplitMix64 counter generator + Box-Muller).

This module draws the numbers both sides consume: the CUDA path receives
them as device tensors, the oracle as host buffers.  It contains none of the
weighted-sum or scaled-SiLU arithmetic.  The C source states the generator's
definition; ``workloads`` holds the five synthetic workloads' recipes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "inputgen.c")
_LIB = os.path.join(_HERE, "libinputgen.so")

DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}
NORMAL, UNIFORM = 0, 1


def build(force: bool = False) -> str:
    """Compile libinputgen.so next to its source (gcc, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
               _SRC, "-o", _LIB + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.ig_fill.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                              ctypes.c_double, ctypes.c_double, ctypes.c_uint64, ctypes.c_uint64,
                              ctypes.c_int64]
        L.ig_fill.restype = ctypes.c_int
        L.ig_fill_rows.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                   ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64]
        L.ig_fill_rows.restype = ctypes.c_int
        L.ig_word.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
        L.ig_word.restype = ctypes.c_uint64
        L.ig_splitmix64.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        L.ig_splitmix64.restype = ctypes.c_uint64
        L.ig_round_f16.argtypes = [ctypes.c_double]
        L.ig_round_f16.restype = ctypes.c_uint32
        L.ig_round_bf16.argtypes = [ctypes.c_double]
        L.ig_round_bf16.restype = ctypes.c_uint32
        _lib = L
    return _lib


def _torch_dtype(dt: str):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dt]


def fill_(t, dt: str, dist: int, a: float, b: float, seed: int, stream: int, first: int = 0):
    """Fill a contiguous host torch tensor (any shape) with stream elements
    first .. first + numel - 1."""
    assert t.device.type == "cpu" and t.is_contiguous()
    rc = lib().ig_fill(ctypes.c_void_p(t.data_ptr()), t.numel(), DTYPE_CODE[dt], dist,
                       float(a), float(b), seed, stream, first)
    if rc != 0:
        raise ValueError("ig_fill rejected its arguments")
    return t


def fill_rows_(t, dt: str, cols: int, dist: int, a: float, b: float, seed: int, stream: int,
               first_row: int = 0):
    """Fill a host 2-D torch tensor whose row stride may exceed `cols` with the
    rows first_row.. of a logical [*, cols] tensor."""
    assert t.device.type == "cpu" and t.dim() == 2 and t.stride(1) == 1
    rc = lib().ig_fill_rows(ctypes.c_void_p(t.data_ptr()), t.shape[0], cols, t.stride(0),
                            DTYPE_CODE[dt], dist, float(a), float(b), seed, stream, first_row)
    if rc != 0:
        raise ValueError("ig_fill_rows rejected its arguments")
    return t


def make(shape, dt: str, dist: int, a: float, b: float, seed: int, stream: int, first: int = 0,
         pin: bool = False):
    """New host tensor of `shape` filled from (seed, stream) starting at element `first`."""
    import torch
    t = torch.empty(shape, dtype=_torch_dtype(dt), pin_memory=pin)
    return fill_(t, dt, dist, a, b, seed, stream, first)


def word(seed: int, stream: int, k: int) -> int:
    return lib().ig_word(seed, stream, k)


def splitmix64(state0: int, k: int) -> int:
    return lib().ig_splitmix64(state0, k)


def round_f16_bits(v: float) -> int:
    return lib().ig_round_f16(float(v))


def round_bf16_bits(v: float) -> int:
    return lib().ig_round_bf16(float(v))


if __name__ == "__main__":
    build(force="--force" in sys.argv)
    print(_LIB)
