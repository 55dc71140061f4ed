"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the bench.

This module only draws numbers (counter-based SplitMix64, Box-Muller,
Student-t); it holds none of the codec's arithmetic, so both sides of a
parity test can read the same buffer without sharing any method code.

The workloads follow the five synthetic weight recipes used for this codec:
  * ``normal``      N(0, 0.02^2) BF16 matrices (the 256x1024 and 8192x8192 cases)
  * ``rows_outliers`` per-row std log-uniform in [0.005, 0.05], Gaussian entries,
                    0.1 % of entries replaced by +-10 sigma_r (the 4096x4096 sweep)
  * ``student_t5``  Student-t (nu = 5) scaled to std 0.02 (DiT/Transformer layers)
  * ``special_rows`` rows of +-0, a constant, subnormals, +-inf, NaN payloads
                    (lossless path)
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile synth.c into libsynth.so next to it (gcc, -O2, pthreads)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, i32, f64, ptr = ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.synth_u64.restype = u64
        lib.synth_u64.argtypes = [u64, u64, u64]
        lib.synth_normal_bf16.argtypes = [u64, u64, f64, f64, ptr, i32]
        lib.synth_normal_f64.argtypes = [u64, u64, ptr, i32]
        lib.synth_uniform_f64.argtypes = [u64, u64, f64, f64, ptr]
        lib.synth_student_t5_bf16.argtypes = [u64, u64, f64, ptr, i32]
        lib.synth_rows_outliers_bf16.restype = i32
        lib.synth_rows_outliers_bf16.argtypes = [u64, u64, u64, f64, f64, f64, f64, ptr, i32]
        lib.synth_special_row_bf16.argtypes = [u64, u64, i32, ptr]
        _lib = lib
    return _lib


def _threads(n_threads):
    return int(n_threads) if n_threads else (os.cpu_count() or 1)


def normal_bf16(seed: int, rows: int, cols: int, std: float = 0.02, mean: float = 0.0, n_threads=None) -> np.ndarray:
    """rows x cols BF16 bit patterns (uint16) drawn from N(mean, std^2)."""
    out = np.empty((rows, cols), dtype=np.uint16)
    _load().synth_normal_bf16(seed, out.size, mean, std, out.ctypes.data, _threads(n_threads))
    return out


def student_t5_bf16(seed: int, rows: int, cols: int, std: float = 0.02, n_threads=None) -> np.ndarray:
    """rows x cols BF16 bit patterns of a Student-t (nu = 5) scaled to std."""
    out = np.empty((rows, cols), dtype=np.uint16)
    _load().synth_student_t5_bf16(seed, out.size, std, out.ctypes.data, _threads(n_threads))
    return out


def rows_outliers_bf16(seed: int, rows: int, cols: int, sig_lo: float = 0.005, sig_hi: float = 0.05,
                       frac: float = 0.001, k_sigma: float = 10.0, n_threads=None) -> np.ndarray:
    """Per-row log-uniform std, Gaussian entries, exactly round(frac*rows*cols) +-k_sigma outliers."""
    out = np.empty((rows, cols), dtype=np.uint16)
    rc = _load().synth_rows_outliers_bf16(seed, rows, cols, sig_lo, sig_hi, frac, k_sigma, out.ctypes.data,
                                          _threads(n_threads))
    if rc != 0:
        raise MemoryError("synth_rows_outliers_bf16 failed")
    return out


SPECIAL_KINDS = {"pos_zero": 0, "neg_zero": 1, "constant": 2, "subnormal": 3, "inf": 4, "nan": 5, "max_finite": 6}


def special_row_bf16(seed: int, cols: int, kind: str) -> np.ndarray:
    row = np.empty(cols, dtype=np.uint16)
    _load().synth_special_row_bf16(seed, cols, SPECIAL_KINDS[kind], row.ctypes.data)
    return row


def with_special_rows(w: np.ndarray, seed: int, placement=None) -> np.ndarray:
    """Copy of w with whole rows replaced by the special kinds (lossless edge cases)."""
    w = w.copy()
    rows = w.shape[0]
    if placement is None:
        placement = {"pos_zero": 0, "neg_zero": 1, "constant": rows // 3, "subnormal": rows // 2 + 1,
                     "inf": rows - 7, "nan": rows - 2, "max_finite": rows - 1}
    for kind, r in placement.items():
        w[r] = special_row_bf16(seed + r, w.shape[1], kind)
    return w


def normal_f64(seed: int, n: int, n_threads=None) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().synth_normal_f64(seed, n, out.ctypes.data, _threads(n_threads))
    return out


def uniform_f64(seed: int, n: int, lo: float, hi: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().synth_uniform_f64(seed, n, lo, hi, out.ctypes.data)
    return out


def u64(seed: int, stream: int, n: int) -> int:
    return int(_load().synth_u64(seed, stream, n))


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to float32 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)
