"""ctypes binding of libentropack.so (argument marshalling only).

Every step of the codec runs inside the library: the host encoder in C++,
decoding in the sm_103a kernels.  There is no Python or CPU fallback: if the
shared library is missing this module raises at import time.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libentropack.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libentropack.so not found at {LIB_PATH}; build it with "
        "`python -m dit_weight_compression_02_b300.build` (needs nvcc)")

lib = ctypes.CDLL(LIB_PATH)

P = ctypes.c_void_p
i32, i64, f32, f64, sz, u32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double, ctypes.c_size_t, ctypes.c_uint32


class EpParams(ctypes.Structure):
    _fields_ = [("mode", i32), ("target_bpp", f32), ("container", i32), ("sample_frac", f32), ("n_threads", i32)]


class EpInfo(ctypes.Structure):
    _fields_ = [("rows", i64), ("cols", i64), ("n_tiles", i64), ("mode", i32), ("container", i32),
                ("target_bpp", f32), ("j", i32), ("delta", f64), ("total_bytes", ctypes.c_uint64),
                ("n_sample_rows", u32), ("actual_bpp", f64), ("out_elem_bytes", sz), ("has_row_scale", i32)]


class EpBatchItem(ctypes.Structure):
    _fields_ = [("h_blob", P), ("d_blob", P), ("bytes", sz), ("d_out", P), ("d_row_scale_out", P)]


class EpBatchPlan(ctypes.Structure):
    _fields_ = [("n_items", i64), ("total_units", i64), ("ring", i32), ("kind", i32), ("n_ctx", i32),
                ("reserved", i32), ("d_workspace", P), ("workspace_bytes", sz), ("items_off", ctypes.c_uint64),
                ("units_off", ctypes.c_uint64), ("counters_off", ctypes.c_uint64)]


# name -> (restype, argtypes); mirrors include/entropack.h
class EpLayerRef(ctypes.Structure):
    _fields_ = [("w", P), ("rows", i64), ("cols", i64), ("sensitivity", f32)]


SIGNATURES = {
    "ep_version": (i32, []),
    "ep_status_string": (ctypes.c_char_p, [i32]),
    "ep_encode": (i32, [P, i64, i64, ctypes.POINTER(EpParams), ctypes.POINTER(P), ctypes.POINTER(sz)]),
    "ep_free": (None, [P]),
    "ep_actual_bpp": (i32, [P, sz, ctypes.POINTER(f64)]),
    "ep_query": (i32, [P, sz, ctypes.POINTER(EpInfo)]),
    "ep_decode": (i32, [P, P, sz, P, P, P, P]),
    "ep_decode_symbols": (i32, [P, P, sz, P, P, P, P, P]),
    "ep_batch_workspace_bytes": (sz, [i64]),
    "ep_batch_prepare": (i32, [ctypes.POINTER(EpBatchItem), i64, i32, P, sz, ctypes.POINTER(EpBatchPlan)]),
    "ep_batch_decode": (i32, [ctypes.POINTER(EpBatchPlan), P, P]),
    "ep_sync_status": (i32, [P, P]),
    "ep_batch_decode_static": (i32, [ctypes.POINTER(EpBatchItem), i64, i32, P, P]),
    "ep_linear_bf16": (i32, [P, P, P, P, i64, i64, i64, P, P]),
    "ep_compressed_linear": (i32, [P, P, sz, P, i64, P, P, i32, P, sz, P, P]),
    "ep_encode_at": (i32, [P, i64, i64, ctypes.POINTER(EpParams), i32, ctypes.POINTER(P), ctypes.POINTER(sz)]),
    "ep_estimate_bpp": (i32, [P, i64, i64, f32, i32, i32, ctypes.POINTER(f64), ctypes.POINTER(i32)]),
    "ep_allocate_bits": (i32, [ctypes.POINTER(EpLayerRef), i64, f32, f32, i32, P, P, ctypes.POINTER(i32)]),
    "ep_stream_open": (i32, [P, sz, ctypes.POINTER(P)]),
    "ep_stream_close": (None, [P]),
    "ep_decode_h": (i32, [P, P, P, P, P, P]),
    "ep_compressed_linear_h": (i32, [P, P, P, i64, P, P, i32, P, sz, P, P]),
    "ep_fused_tokens_per_pass": (i64, [i64]),
    "ep_q4_levels": (i32, [i32, P]),
    "ep_q4_encode": (i32, [P, i64, i64, P, P, P, i32]),
    "ep_q4_decode": (i32, [P, P, i64, i64, P, P, P]),
    "ep_fp8_row_encode": (i32, [P, i64, i64, P, P, i32]),
    "ep_fp8_row_decode": (i32, [P, P, i64, i64, P, P]),
}

for _name, (_res, _args) in SIGNATURES.items():
    _fn = getattr(lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

STATUS = {0: "EP_OK", 1: "EP_ERR_INVALID_ARG", 2: "EP_ERR_SHAPE", 3: "EP_ERR_NONFINITE", 4: "EP_ERR_CORRUPT",
          5: "EP_ERR_UNSUPPORTED", 6: "EP_ERR_NOMEM", 7: "EP_ERR_CUDA"}


class EntroPackError(RuntimeError):
    def __init__(self, code: int, what: str):
        msg = lib.ep_status_string(code).decode()
        super().__init__(f"{what}: {STATUS.get(code, code)} ({msg})")
        self.code = code
        self.status = STATUS.get(code, str(code))


def check(code: int, what: str) -> None:
    if code != 0:
        raise EntroPackError(code, what)
