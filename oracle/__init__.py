"""Plain CPU oracle of the EntroPack codec -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  It shares no code with the CUDA
library: its C source (``entropack_oracle.c``) is compiled separately with gcc
and follows stream format version 1 step by step.

Method: "EntroPack: Fast and Accurate Entropy-Coded Weight Compression at
Arbitrary Bitrates", Abstract (row-normalised E8 lattice quantisation, a
conditional model of lattice coordinates, sampled storage estimates, tile-wise
entropy coding, reconstruction into BF16/FP16/FP8/INT8 containers) and the
"EntroPack PyTorch Guide", "Choose a compression contract" (lossy target
bitrate vs lossless tiled ANS).

Pinned by tests/test_oracle_*.py; parity unpinned: the exact resolution index
picked by the rate search (pinned only by determinism and by its distance to
the target).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "entropack_oracle.c")
_HDR = os.path.join(_HERE, "entropack_oracle.h")
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None

CONTAINERS = {"bf16": 0, "fp16": 1, "fp8": 2, "int8": 3}
ERRORS = {0: "ok", 1: "invalid_arg", 2: "shape", 3: "nonfinite", 4: "corrupt", 5: "unsupported", 6: "nomem"}


class OracleError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"oracle {what}: {ERRORS.get(code, code)}")
        self.code = code
        self.name = ERRORS.get(code, str(code))


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no FP contraction) into liboracle.so."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < newest:
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC,
                               "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P, i64, i32, f32, f64, u16, u32 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                                            ctypes.c_double, ctypes.c_uint16, ctypes.c_uint32)
        sz = ctypes.c_size_t
        L.oracle_e8_nearest.argtypes = [P, P, P]
        L.oracle_row_rms.restype = f64
        L.oracle_row_rms.argtypes = [P, i64]
        L.oracle_delta.restype = f64
        L.oracle_delta.argtypes = [i32]
        L.oracle_rn7.restype = f64
        L.oracle_rn7.argtypes = [f64]
        L.oracle_tr7.restype = f64
        L.oracle_tr7.argtypes = [f64]
        L.oracle_normalize.argtypes = [P, P]
        L.oracle_rans_encode.restype = i32
        L.oracle_rans_encode.argtypes = [P, P, i64, P, P, P, i64, P]
        L.oracle_rans_decode.restype = i32
        L.oracle_rans_decode.argtypes = [P, i64, u32, P, i64, P, P]
        L.oracle_f32_to_bf16.restype = u16
        L.oracle_f32_to_bf16.argtypes = [f32]
        L.oracle_f32_to_f16.restype = u16
        L.oracle_f32_to_f16.argtypes = [f32]
        L.oracle_f32_to_e4m3_satfinite.restype = ctypes.c_uint8
        L.oracle_f32_to_e4m3_satfinite.argtypes = [f32]
        L.oracle_f32_to_int8.restype = ctypes.c_int8
        L.oracle_f32_to_int8.argtypes = [f32]
        L.oracle_block_symbols.restype = i32
        L.oracle_block_symbols.argtypes = [P, i32, P, P, P]
        L.oracle_estimate_bpp.restype = f64
        L.oracle_estimate_bpp.argtypes = [P, i64, i64, f32, i32]
        L.oracle_select_j.restype = i32
        L.oracle_select_j.argtypes = [P, i64, i64, f32, f32, P]
        L.oracle_encode.restype = i32
        L.oracle_encode.argtypes = [P, i64, i64, f32, i32, f32, P, P]
        L.oracle_encode_at.argtypes = [P, i64, i64, f32, i32, i32, f32, P, P]
        L.oracle_smallest_valid_j.restype = i32
        L.oracle_smallest_valid_j.argtypes = [P, i64, i64]
        L.oracle_encode_lossless.restype = i32
        L.oracle_encode_lossless.argtypes = [P, i64, i64, P, P]
        L.oracle_encode_lossless_dtype.restype = i32
        L.oracle_encode_lossless_dtype.argtypes = [P, i64, i64, i32, P, P]
        L.oracle_free.argtypes = [P]
        L.oracle_decode.restype = i32
        L.oracle_decode.argtypes = [P, sz, P, P, i64, i64]
        L.oracle_decode_symbols.restype = i32
        L.oracle_decode_symbols.argtypes = [P, sz, P, i64, i64]
        L.oracle_gemm_f64.argtypes = [P, P, P, i64, i64, i64]
        L.oracle_decode_lattice.restype = i32
        L.oracle_decode_lattice.argtypes = [P, sz, P, i64, i64]
        L.oracle_convert_f32.argtypes = [i32, i64, P, P]
        L.oracle_nf4_levels.argtypes = [P]
        L.oracle_int4_levels.argtypes = [P]
        L.oracle_q4_roundtrip.restype = f64
        L.oracle_q4_roundtrip.argtypes = [P, i64, i64, P, P, P, P]
        L.oracle_e4m3_to_f64.restype = f64
        L.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        L.oracle_fp8_row_roundtrip.restype = f64
        L.oracle_fp8_row_roundtrip.argtypes = [P, i64, i64, P, P, P]
        _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------ pieces
def e8_nearest(x):
    """Nearest E8 point to x (8 doubles): returns (a int64[8], coset) with q = a + coset/2."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    a = np.zeros(8, dtype=np.int64)
    c = ctypes.c_int(0)
    lib().oracle_e8_nearest(_p(x), _p(a), ctypes.byref(c))
    return a, c.value


def row_rms(row_bits: np.ndarray) -> float:
    row_bits = np.ascontiguousarray(row_bits, dtype=np.uint16)
    return lib().oracle_row_rms(_p(row_bits), row_bits.size)


def delta(j: int) -> float:
    return lib().oracle_delta(j)


def rn7(v: float) -> float:
    return lib().oracle_rn7(v)


def tr7(v: float) -> float:
    return lib().oracle_tr7(v)


def normalize(counts) -> np.ndarray:
    counts = np.ascontiguousarray(counts, dtype=np.uint64)
    assert counts.shape == (256,)
    f = np.zeros(256, dtype=np.uint32)
    lib().oracle_normalize(_p(counts), _p(f))
    return f


def rans_encode(syms, ctx, freq_by_ctx):
    """rANS-encode one lane. freq_by_ctx: (<=8, 256) table; returns (state, words)."""
    syms = np.ascontiguousarray(syms, dtype=np.uint8)
    ctx = np.ascontiguousarray(ctx, dtype=np.uint8)
    F = np.zeros((8, 256), dtype=np.uint32)
    F[: len(freq_by_ctx)] = freq_by_ctx
    words = np.zeros(max(16, syms.size + 8), dtype=np.uint16)
    st = ctypes.c_uint32(0)
    nw = ctypes.c_int64(0)
    rc = lib().oracle_rans_encode(_p(syms), _p(ctx), syms.size, _p(F), ctypes.byref(st), _p(words), words.size,
                                  ctypes.byref(nw))
    if rc:
        raise OracleError(rc, "rans_encode")
    return st.value, words[: nw.value].copy()


def rans_decode(words, state, ctx, freq_by_ctx):
    words = np.ascontiguousarray(words, dtype=np.uint16)
    ctx = np.ascontiguousarray(ctx, dtype=np.uint8)
    F = np.zeros((8, 256), dtype=np.uint32)
    F[: len(freq_by_ctx)] = freq_by_ctx
    out = np.zeros(ctx.size, dtype=np.uint8)
    rc = lib().oracle_rans_decode(_p(words), words.size, state, _p(ctx), ctx.size, _p(F), _p(out))
    if rc:
        raise OracleError(rc, "rans_decode")
    return out


def f32_to_bf16(v: float) -> int:
    return lib().oracle_f32_to_bf16(v)


def f32_to_f16(v: float) -> int:
    return lib().oracle_f32_to_f16(v)


def f32_to_e4m3(v: float) -> int:
    return lib().oracle_f32_to_e4m3_satfinite(v)


def f32_to_int8(v: float) -> int:
    return lib().oracle_f32_to_int8(v)


def block_symbols(a, coset):
    a = np.ascontiguousarray(a, dtype=np.int64)
    u = np.zeros(8, dtype=np.uint8)
    cx = np.zeros(8, dtype=np.uint8)
    pl = np.zeros(8, dtype=np.int32)
    n = lib().oracle_block_symbols(_p(a), coset, _p(u), _p(cx), _p(pl))
    return u, cx, pl, n


def estimate_bpp(w_bits: np.ndarray, sample_frac: float, j: int) -> float:
    w_bits = np.ascontiguousarray(w_bits, dtype=np.uint16)
    return lib().oracle_estimate_bpp(_p(w_bits), w_bits.shape[0], w_bits.shape[1], sample_frac, j)


def select_j(w_bits: np.ndarray, target_bpp: float, sample_frac: float = 0.05):
    """Returns (j, j_lo): the chosen resolution index and the smallest admissible one."""
    w_bits = np.ascontiguousarray(w_bits, dtype=np.uint16)
    jlo = ctypes.c_int(0)
    j = lib().oracle_select_j(_p(w_bits), w_bits.shape[0], w_bits.shape[1], target_bpp, sample_frac,
                              ctypes.byref(jlo))
    return j, jlo.value


# ----------------------------------------------------------------- codec
def _take_blob(ptr, size) -> bytes:
    data = ctypes.string_at(ptr, size.value)
    lib().oracle_free(ptr)
    return data


def encode(w_bits: np.ndarray, target_bpp: float = 4.0, container: str = "bf16", sample_frac: float = 0.05) -> bytes:
    """Lossy E8 encode of a BF16 matrix (uint16 bit patterns, M x K)."""
    w_bits = np.ascontiguousarray(w_bits, dtype=np.uint16)
    ptr = ctypes.c_void_p(0)
    size = ctypes.c_size_t(0)
    rc = lib().oracle_encode(_p(w_bits), w_bits.shape[0], w_bits.shape[1], target_bpp, CONTAINERS[container],
                             sample_frac, ctypes.byref(ptr), ctypes.byref(size))
    if rc:
        raise OracleError(rc, "encode")
    return _take_blob(ptr, size)


def encode_at(w_bits: np.ndarray, j: int, target_bpp: float = 4.0, container: str = "bf16",
              sample_frac: float = 0.05) -> bytes:
    """Lossy E8 encode at resolution index j (no rate search); target_bpp is only recorded."""
    w_bits = np.ascontiguousarray(w_bits, dtype=np.uint16)
    ptr = ctypes.c_void_p(0)
    size = ctypes.c_size_t(0)
    rc = lib().oracle_encode_at(_p(w_bits), w_bits.shape[0], w_bits.shape[1], target_bpp, int(j),
                                CONTAINERS[container], sample_frac, ctypes.byref(ptr), ctypes.byref(size))
    if rc:
        raise OracleError(rc, "encode_at")
    return _take_blob(ptr, size)


def smallest_valid_j(w_bits: np.ndarray) -> int:
    w_bits = np.ascontiguousarray(w_bits, dtype=np.uint16)
    return lib().oracle_smallest_valid_j(_p(w_bits), w_bits.shape[0], w_bits.shape[1])


J_MIN, J_MAX = -640, 128


def allocate_bits(layers, avg_bpp: float, sensitivities=None, sample_frac: float = 0.05) -> dict:
    """Per-layer resolution indices for a whole-model storage budget.

    Reading of the pages' per-layer allocation ("EntroPack PyTorch Guide",
    "Separate reconstruction metrics from application metrics": different
    bitrates across layers, allocation recorded; the Chinese overview page:
    give the limited space to the layers whose errors matter more), driven by
    the sampled storage estimates (Abstract).  Minimising
    sum_l alpha_l * n_l * D_l subject to sum_l n_l * R_l <= avg_bpp * sum_l n_l,
    with the high-resolution E8 error D_l ~ G * Delta_l^2 (the same for every
    row-normalised layer at one Delta), gives equal slopes:
    alpha_l * Delta_l^2 constant, i.e. j_l = t - 32 * log2(alpha_l) on the
    Delta_j = 2^(j / 64) grid.  Steps:
      1. o_l = round(32 * log2(alpha_l)); j_l(t) = clamp(t - o_l, j_min_l, J_MAX)
         with j_min_l the layer's smallest admissible index;
      2. E(t) = sum_l n_l * estimate_l(j_l(t)) bits, budget B = avg_bpp * sum_l n_l;
      3. t = the smallest shared index with E(t) <= B, by bisection between
         t_lo = min_l(j_min_l + o_l) and t_hi = max_l(J_MAX + o_l) (t_lo if it
         already fits, t_hi if nothing fits).
    Returns {"t", "j": [...], "est_bpp": [...], "offsets": [...], "budget_bits", "est_bits"}.
    """
    L = len(layers)
    alphas = [1.0] * L if sensitivities is None else [float(a) for a in sensitivities]
    if len(alphas) != L or not all(math.isfinite(a) and a > 0 for a in alphas) or not (avg_bpp > 0):
        raise ValueError("one positive finite sensitivity per layer and a positive budget are required")
    n = [int(w.shape[0]) * int(w.shape[1]) for w in layers]
    jmin = [smallest_valid_j(w) for w in layers]
    off = [int(round_half_away(32.0 * math.log2(a))) for a in alphas]
    cache = {}

    def est(l, j):
        if (l, j) not in cache:
            cache[(l, j)] = estimate_bpp(layers[l], sample_frac, j)
        return cache[(l, j)]

    def j_of(l, t):
        return min(max(t - off[l], jmin[l]), J_MAX)

    def total(t):
        e = 0.0
        for l in range(L):
            e += float(n[l]) * est(l, j_of(l, t))
        return e

    budget = float(np.float32(avg_bpp)) * float(sum(n))
    t_lo = min(jmin[l] + off[l] for l in range(L))
    t_hi = max(J_MAX + off[l] for l in range(L))
    if total(t_lo) <= budget:
        t = t_lo
    elif total(t_hi) > budget:
        t = t_hi
    else:
        lo, hi = t_lo, t_hi
        while hi - lo > 1:
            mid = lo + (hi - lo) // 2
            if total(mid) <= budget:
                hi = mid
            else:
                lo = mid
        t = hi
    js = [j_of(l, t) for l in range(L)]
    return {"t": t, "j": js, "est_bpp": [est(l, js[l]) for l in range(L)], "offsets": off,
            "budget_bits": budget, "est_bits": total(t)}


def round_half_away(x: float) -> float:
    """Round to the nearest integer, halves away from zero (C's lround)."""
    return math.copysign(math.floor(abs(x) + 0.5), x)


LOSSLESS_DTYPES = {"bf16": (0, np.uint16), "fp16": (1, np.uint16), "fp8": (2, np.uint8), "fp32": (4, np.uint32)}


def encode_lossless(w_bits: np.ndarray, dtype: str = "bf16") -> bytes:
    """Lossless tiled ANS of a matrix of element bit patterns (uint16 for BF16/FP16, uint8 for FP8, uint32 for FP32)."""
    code, npt = LOSSLESS_DTYPES[dtype]
    w_bits = np.ascontiguousarray(w_bits, dtype=npt)
    ptr = ctypes.c_void_p(0)
    size = ctypes.c_size_t(0)
    rc = lib().oracle_encode_lossless_dtype(_p(w_bits), w_bits.shape[0], w_bits.shape[1], code, ctypes.byref(ptr),
                                            ctypes.byref(size))
    if rc:
        raise OracleError(rc, "encode_lossless")
    return _take_blob(ptr, size)


def header(blob: bytes) -> dict:
    """Header fields of a stream, read with numpy (no codec arithmetic)."""
    h = np.frombuffer(blob[:128], dtype=np.uint8)
    u64 = lambda o: int(h[o:o + 8].view(np.uint64)[0])
    return {
        "mode": int(h[6]), "container": int(h[7]), "M": u64(8), "K": u64(16), "n_tiles": u64(24),
        "target_bpp": float(h[32:36].view(np.float32)[0]), "j": int(h[36:40].view(np.int32)[0]),
        "delta": float(h[40:48].view(np.float64)[0]), "n_ctx": int(h[53]),
        "tables_off": u64(56), "rowmeta_off": u64(64), "offsets_off": u64(72), "payload_off": u64(80),
        "total_bytes": u64(88), "n_sample_rows": int(h[96:100].view(np.uint32)[0]),
    }


_OUT_DTYPE = {0: np.uint16, 1: np.uint16, 2: np.uint8, 3: np.int8, 4: np.uint32}


def decode(blob: bytes, t_lo: int = 0, t_hi: int | None = None, out=None):
    """Decode tiles [t_lo, t_hi) of a blob; returns (container array M x K, row scales t_r or None)."""
    h = header(blob)
    M, K = h["M"], h["K"]
    t_hi = h["n_tiles"] if t_hi is None else t_hi
    if out is None:
        out = np.zeros((M, K), dtype=_OUT_DTYPE[h["container"]])
    rs = np.zeros(M, dtype=np.float32)
    buf = np.frombuffer(blob, dtype=np.uint8)
    rc = lib().oracle_decode(_p(buf), len(blob), _p(out), _p(rs), t_lo, t_hi)
    if rc:
        raise OracleError(rc, "decode")
    has_scale = h["mode"] == 0 and h["container"] >= 2
    return out, (rs if has_scale else None)


def decode_symbols(blob: bytes, t_lo: int = 0, t_hi: int | None = None) -> np.ndarray:
    h = header(blob)
    t_hi = h["n_tiles"] if t_hi is None else t_hi
    out = np.zeros((h["M"], h["K"]), dtype=np.uint8)
    buf = np.frombuffer(blob, dtype=np.uint8)
    rc = lib().oracle_decode_symbols(_p(buf), len(blob), _p(out), t_lo, t_hi)
    if rc:
        raise OracleError(rc, "decode_symbols")
    return out


def decode_lattice(blob: bytes) -> np.ndarray:
    """k = 2q of every coordinate (M x K int32) of a lossy blob."""
    h = header(blob)
    out = np.zeros((h["M"], h["K"]), dtype=np.int32)
    buf = np.frombuffer(blob, dtype=np.uint8)
    rc = lib().oracle_decode_lattice(_p(buf), len(blob), _p(out), 0, h["n_tiles"])
    if rc:
        raise OracleError(rc, "decode_lattice")
    return out


def convert_f32(values: np.ndarray, kind: str) -> np.ndarray:
    """Oracle conversion of fp32 values to a container (bit patterns; int8 values)."""
    values = np.ascontiguousarray(values, dtype=np.float32)
    dt = {"bf16": np.uint16, "fp16": np.uint16, "fp8": np.uint8, "int8": np.int8}[kind]
    out = np.zeros(values.shape, dtype=dt)
    lib().oracle_convert_f32(CONTAINERS[kind], values.size, _p(values), _p(out))
    return out


def decode_threaded(blob: bytes, n_threads: int | None = None):
    """Tile-parallel oracle decode (contiguous tile ranges on host threads; ctypes drops the GIL)."""
    import threading
    h = header(blob)
    n_threads = n_threads or (os.cpu_count() or 1)
    out = np.zeros((h["M"], h["K"]), dtype=_OUT_DTYPE[h["container"]])
    nt = h["n_tiles"]
    errs = []

    def work(lo, hi):
        try:
            decode(blob, lo, hi, out=out)
        except OracleError as e:
            errs.append(e)

    th = [threading.Thread(target=work, args=(nt * i // n_threads, nt * (i + 1) // n_threads))
          for i in range(n_threads)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    if errs:
        raise errs[0]
    _, rs = decode(blob, 0, 0)
    return out, rs


def gemm_f64(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y = x @ w.T in fp64 by a plain triple loop (x: T x K, w: N x K)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    y = np.zeros((x.shape[0], w.shape[0]), dtype=np.float64)
    lib().oracle_gemm_f64(_p(x), _p(w), _p(y), x.shape[0], w.shape[0], x.shape[1])
    return y


def container_to_f64(y: np.ndarray, container: str | int, row_scale=None) -> np.ndarray:
    """Widen container values to fp64 weights (times the row scale for FP8/INT8)."""
    import torch
    c = CONTAINERS[container] if isinstance(container, str) else container
    if c == 0:
        v = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    elif c == 1:
        v = y.view(np.float16).astype(np.float64)
    elif c == 2:
        v = torch.from_numpy(y.view(np.uint8).copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    else:
        v = y.astype(np.float64)
    if row_scale is not None:
        v = v * row_scale.astype(np.float64)[:, None]
    return v


def q4_levels(kind: str) -> np.ndarray:
    """The 16 fp64 levels of a 4-bit comparator codebook: "nf4" (ascending) or "int4" (k/7, then 0)."""
    cb = np.zeros(16, dtype=np.float64)
    {"nf4": lib().oracle_nf4_levels, "int4": lib().oracle_int4_levels}[kind](_p(cb))
    return cb


def q4_roundtrip(w_bits: np.ndarray, kind: str = "nf4", block: int = 64):
    """Block-absmax 4-bit comparator of a BF16 matrix.

    Returns (codes uint8 0..15, FP32 block scales, BF16 reconstruction bits, bits per weight)."""
    w_bits = np.ascontiguousarray(w_bits, dtype=np.uint16)
    n = w_bits.size
    codes = np.zeros(w_bits.shape, dtype=np.uint8)
    scales = np.zeros((n + block - 1) // block, dtype=np.float32)
    recon = np.zeros(w_bits.shape, dtype=np.uint16)
    levels = q4_levels(kind)
    bits = lib().oracle_q4_roundtrip(_p(w_bits), n, block, _p(levels), _p(codes), _p(scales), _p(recon))
    return codes, scales, recon, bits


def e4m3_to_f64(b: int) -> float:
    return lib().oracle_e4m3_to_f64(int(b))


def fp8_row_roundtrip(w_bits: np.ndarray, with_codes: bool = False):
    """Per-row-scaled FP8 E4M3 comparator: (BF16 reconstruction bits, bits per weight).

    with_codes: also return the E4M3 bytes (M x K) and the FP32 row scales."""
    w_bits = np.ascontiguousarray(w_bits, dtype=np.uint16)
    recon = np.zeros(w_bits.shape, dtype=np.uint16)
    codes = np.zeros(w_bits.shape, dtype=np.uint8)
    scales = np.zeros(w_bits.shape[0], dtype=np.float32)
    bits = lib().oracle_fp8_row_roundtrip(_p(w_bits), w_bits.shape[0], w_bits.shape[1], _p(recon), _p(codes),
                                          _p(scales))
    return (recon, bits, codes, scales) if with_codes else (recon, bits)


def rel_l2(w_hat: np.ndarray, w: np.ndarray) -> float:
    """Relative L2 weight error ||w_hat - w|| / ||w|| in fp64."""
    w = np.asarray(w, dtype=np.float64)
    return float(np.linalg.norm(np.asarray(w_hat, dtype=np.float64) - w) / np.linalg.norm(w))
