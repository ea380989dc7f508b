"""Seeded synthetic inputs shared by the CPU oracle and the CUDA library.

This package only draws numbers (counter-based SplitMix64 + Box-Muller, see
``synth.c``) and lays them out in the shapes of the OPT workloads; it holds none
of the generation method's arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "synth.c"
_SO = _HERE / "_synth.so"
_lib = None


def build(force: bool = False) -> Path:
    """Compile ``synth.c`` into ``_synth.so`` next to it (gcc, OpenMP)."""
    if _SO.exists() and not force and _SO.stat().st_mtime >= _SRC.stat().st_mtime:
        return _SO
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=str(_HERE))
    os.close(fd)
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, str(_SRC), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(str(_SO))
        i64, u64, f64 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_double
        vp = ctypes.c_void_p
        lib.synth_normal_f32.argtypes = [vp, i64, u64, u64, f64, f64]
        lib.synth_normal_bf16.argtypes = [vp, i64, u64, u64, f64, f64]
        lib.synth_uniform_i32.argtypes = [vp, i64, u64, u64, ctypes.c_int32, ctypes.c_int32]
        lib.synth_raw_draw.argtypes = [u64, u64, u64]
        lib.synth_raw_draw.restype = u64
        lib.synth_splitmix64_next.argtypes = [ctypes.POINTER(u64)]
        lib.synth_splitmix64_next.restype = u64
        lib.synth_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.synth_f32_to_bf16.restype = ctypes.c_uint16
        _lib = lib
    return _lib


def normal(shape, seed: int, tensor_id: int, mean: float = 0.0, std: float = 1.0,
           dtype: str = "f32") -> np.ndarray:
    """Normal variates of ``shape``; ``dtype`` "f32" (float32) or "bf16" (raw uint16 bits)."""
    lib = _load()
    n = int(np.prod(shape)) if len(shape) else 1
    if dtype == "f32":
        out = np.empty(shape, dtype=np.float32)
        lib.synth_normal_f32(out.ctypes.data, n, seed, tensor_id, mean, std)
    elif dtype == "bf16":
        out = np.empty(shape, dtype=np.uint16)
        lib.synth_normal_bf16(out.ctypes.data, n, seed, tensor_id, mean, std)
    else:
        raise ValueError(f"unknown dtype {dtype!r}")
    return out


def uniform_int(shape, seed: int, tensor_id: int, lo: int, hi: int) -> np.ndarray:
    """Integers uniform in [lo, hi) as int32."""
    if not lo < hi:
        raise ValueError("empty range")
    lib = _load()
    out = np.empty(shape, dtype=np.int32)
    lib.synth_uniform_i32(out.ctypes.data, out.size, seed, tensor_id, lo, hi)
    return out


def raw_draw(seed: int, tensor_id: int, n: int) -> int:
    return int(_load().synth_raw_draw(seed, tensor_id, n))


def splitmix64_sequence(state: int, count: int) -> list[int]:
    """Plain sequential SplitMix64 outputs from ``state`` (known-answer tests)."""
    lib = _load()
    s = ctypes.c_uint64(state)
    return [int(lib.synth_splitmix64_next(ctypes.byref(s))) for _ in range(count)]


def f32_to_bf16_bits(x: float) -> int:
    return int(_load().synth_f32_to_bf16(ctypes.c_float(x)))


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of raw bf16 bits to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
