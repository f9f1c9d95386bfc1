"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

Nothing in this package computes any part of the RVQ expert FFN: it only
draws bytes, normal samples and bf16 roundings of generated activations from
counter-based SplitMix64 streams (see ``gen.c``).  The oracle and the CUDA
path both take their inputs from here, so a parity test compares two
independent computations on bit-identical inputs.

The C source is compiled with gcc on first use (or by the top-level build).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gen.c into libsynth.so (plain gcc, -O2, no arch flags)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, u32, vp = ctypes.c_uint64, ctypes.c_int32, ctypes.c_void_p
            lib.synth_sm64_at.restype = u64
            lib.synth_sm64_at.argtypes = [u64, u64]
            lib.synth_derive.restype = u64
            lib.synth_derive.argtypes = [u64, u64]
            lib.synth_bytes.restype = None
            lib.synth_bytes.argtypes = [u64, u64, u64, vp]
            lib.synth_normal_f32.restype = None
            lib.synth_normal_f32.argtypes = [u64, u64, ctypes.c_double, vp]
            lib.synth_f32_to_bf16_array.restype = None
            lib.synth_f32_to_bf16_array.argtypes = [vp, u64, vp]
            lib.synth_permutation.restype = None
            lib.synth_permutation.argtypes = [u64, u32, vp]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ---------------------------------------------------------------- primitives

def sm64_at(seed: int, i: int) -> int:
    return int(_load().synth_sm64_at(seed & (2**64 - 1), i))


def derive(seed: int, tag: int) -> int:
    return int(_load().synth_derive(seed & (2**64 - 1), tag & (2**64 - 1)))


def bytes_into(seed: int, out: np.ndarray, first: int = 0, threads: int = 0) -> np.ndarray:
    """Fill ``out`` (uint8, contiguous) with bytes [first, first+out.size) of
    the stream; splits the range over threads for large buffers."""
    assert out.dtype == np.uint8
    flat = out.reshape(-1)
    n = flat.size
    lib = _load()
    if threads <= 0:
        threads = min(16, os.cpu_count() or 1)
    if n < (1 << 22) or threads == 1:
        lib.synth_bytes(seed, first, n, _ptr(flat))
        return out
    step = ((n + threads - 1) // threads + 7) // 8 * 8
    base = flat.ctypes.data

    def work(lo):
        hi = min(n, lo + step)
        lib.synth_bytes(seed, first + lo, hi - lo, base + lo)

    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(work, range(0, n, step)))
    return out


def random_bytes(seed: int, count: int, first: int = 0) -> np.ndarray:
    return bytes_into(seed, np.empty(count, np.uint8), first)


def normal_f32(seed: int, count: int, sigma: float = 1.0) -> np.ndarray:
    out = np.empty(count, np.float32)
    _load().synth_normal_f32(seed, count, float(sigma), _ptr(out))
    return out


def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    a = np.ascontiguousarray(a, np.float32)
    out = np.empty(a.shape, np.uint16)
    _load().synth_f32_to_bf16_array(_ptr(a), a.size, _ptr(out))
    return out


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact)."""
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def permutation(seed: int, n: int) -> np.ndarray:
    out = np.empty(n, np.int32)
    _load().synth_permutation(seed, n, _ptr(out))
    return out
