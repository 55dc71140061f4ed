"""Python surface of the EntroPack B300 library (thin marshalling over the C ABI).

Names follow the pages' interface ("EntroPack PyTorch Guide", "Choose a
compression contract" and "Replace one linear layer before a whole model"):
``compress`` / ``decompress``, ``EntroPackLossyConfig`` (target bitrate),
``TileANSConfig`` (lossless), ``CompressedLinear.from_linear``, and
``target_bpp`` vs ``actual_bpp`` (which includes metadata).  Encoding runs in
the library's host encoder, decoding in its sm_103a kernels; PyTorch only
provides device memory and streams.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np
import torch

from ._lib import EpBatchItem, EpBatchPlan, EpInfo, EpParams, EntroPackError, check, lib

CONTAINERS = {"bf16": 0, "fp16": 1, "fp8": 2, "int8": 3, "fp32": 4}
CONTAINER_DTYPES = {0: torch.bfloat16, 1: torch.float16, 2: torch.float8_e4m3fn, 3: torch.int8, 4: torch.float32}
# element types of lossless streams: name -> (container code, numpy bit-pattern type)
LOSSLESS_DTYPES = {"bf16": (0, np.uint16), "fp16": (1, np.uint16), "fp8": (2, np.uint8), "fp32": (4, np.uint32)}
_TORCH_TO_LOSSLESS = {torch.bfloat16: "bf16", torch.float16: "fp16", torch.float8_e4m3fn: "fp8", torch.float32: "fp32"}
_BITS_VIEW = {torch.bfloat16: torch.int16, torch.float16: torch.int16, torch.float8_e4m3fn: torch.uint8,
              torch.float32: torch.int32}
MODE_LOSSY, MODE_LOSSLESS = 0, 1


def _ptr(x) -> ctypes.c_void_p:
    if isinstance(x, torch.Tensor):
        return ctypes.c_void_p(x.data_ptr())
    if isinstance(x, np.ndarray):
        return ctypes.c_void_p(x.ctypes.data)
    if x is None:
        return ctypes.c_void_p(0)
    return ctypes.c_void_p(int(x))


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ------------------------------------------------------------------- host side
def bf16_bits(w) -> np.ndarray:
    """BF16 bit patterns (uint16, C-contiguous, host) of a tensor or array."""
    if isinstance(w, torch.Tensor):
        if w.dtype != torch.bfloat16:
            raise TypeError("compress expects a BF16 tensor (EntroPack encodes BF16 weights)")
        return w.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(w)
    if a.dtype != np.uint16:
        raise TypeError("expected BF16 bit patterns as uint16")
    return a


def element_bits(w, dtype: str) -> np.ndarray:
    """Bit patterns (C-contiguous, host) of a tensor or array holding elements of a lossless dtype."""
    code, npt = LOSSLESS_DTYPES[dtype]
    if isinstance(w, torch.Tensor):
        if _TORCH_TO_LOSSLESS.get(w.dtype) != dtype:
            raise TypeError(f"tensor dtype {w.dtype} does not match the lossless dtype {dtype}")
        return w.detach().contiguous().cpu().view(_BITS_VIEW[w.dtype]).numpy().view(npt)
    a = np.ascontiguousarray(w)
    if a.dtype != npt:
        raise TypeError(f"expected {np.dtype(npt).name} bit patterns for {dtype}")
    return a


def encode(w_bits: np.ndarray, target_bpp: float = 4.0, container: str = "bf16", lossless: bool = False,
           sample_frac: float = 0.05, n_threads: int = 0) -> bytes:
    """ep_encode: a rows x cols matrix -> stream bytes.

    Lossy: BF16 bits in, decoded into `container`.  Lossless: elements of the
    type `container` names (bf16, fp16, fp8 or fp32; a torch tensor's own
    dtype is used when it is one of those), restored bit for bit.
    """
    if lossless:
        if isinstance(w_bits, torch.Tensor) and w_bits.dtype in _TORCH_TO_LOSSLESS:
            container = _TORCH_TO_LOSSLESS[w_bits.dtype]
        w_bits = element_bits(w_bits, container)
    else:
        w_bits = bf16_bits(w_bits)
    if w_bits.ndim != 2:
        raise ValueError("expected a 2-D weight matrix")
    p = EpParams(MODE_LOSSLESS if lossless else MODE_LOSSY, float(target_bpp), CONTAINERS[container],
                 float(sample_frac), int(n_threads))
    out = ctypes.c_void_p(0)
    size = ctypes.c_size_t(0)
    check(lib.ep_encode(_ptr(w_bits), w_bits.shape[0], w_bits.shape[1], ctypes.byref(p), ctypes.byref(out),
                        ctypes.byref(size)), "ep_encode")
    try:
        return ctypes.string_at(out, size.value)
    finally:
        lib.ep_free(out)


def query(blob) -> dict:
    """ep_query: validated header fields of a host copy of a stream."""
    buf = np.frombuffer(blob, dtype=np.uint8) if isinstance(blob, (bytes, bytearray)) else blob
    info = EpInfo()
    check(lib.ep_query(_ptr(buf), buf.nbytes, ctypes.byref(info)), "ep_query")
    return {f: getattr(info, f) for f, _ in EpInfo._fields_}


def actual_bpp(blob) -> float:
    buf = np.frombuffer(blob, dtype=np.uint8) if isinstance(blob, (bytes, bytearray)) else blob
    v = ctypes.c_double(0)
    check(lib.ep_actual_bpp(_ptr(buf), buf.nbytes, ctypes.byref(v)), "ep_actual_bpp")
    return v.value


# ----------------------------------------------------------------- device side
class DeviceBlob:
    """A stream resident in HBM together with its (pinned) host copy and header."""

    def __init__(self, blob, device="cuda", pin: bool = True):
        host = np.frombuffer(bytes(blob), dtype=np.uint8) if isinstance(blob, (bytes, bytearray)) else blob
        self.info = query(host)
        self.host = torch.from_numpy(np.array(host, copy=True))
        if pin and torch.cuda.is_available():
            self.host = self.host.pin_memory()
        self.device = torch.empty(self.host.numel(), dtype=torch.uint8, device=device)
        self.device.copy_(self.host, non_blocking=False)
        self.nbytes = self.host.numel()

    @property
    def shape(self):
        return (self.info["rows"], self.info["cols"])

    @property
    def out_dtype(self):
        return CONTAINER_DTYPES[self.info["container"]]

    def alloc_out(self):
        return torch.empty(self.shape, dtype=self.out_dtype, device=self.device.device)


def decode_into(db: DeviceBlob, out: torch.Tensor, row_scale: torch.Tensor | None, status: torch.Tensor,
                stream=None, sym_out: torch.Tensor | None = None) -> None:
    """Enqueue ep_decode (or ep_decode_symbols) on `stream`; no synchronisation."""
    args = (_ptr(db.host), _ptr(db.device), db.nbytes, _ptr(out), _ptr(row_scale))
    if sym_out is None:
        check(lib.ep_decode(*args, _ptr(status), _stream_handle(stream)), "ep_decode")
    else:
        check(lib.ep_decode_symbols(*args, _ptr(sym_out), _ptr(status), _stream_handle(stream)), "ep_decode_symbols")


def sync_status(status: torch.Tensor, stream=None) -> None:
    check(lib.ep_sync_status(_ptr(status), _stream_handle(stream)), "ep_sync_status")


def decode(db: DeviceBlob, out: torch.Tensor | None = None, stream=None, symbols: bool = False):
    """Decode on the GPU; returns (weights, row_scale or None[, symbols]) after checking the status word."""
    out = db.alloc_out() if out is None else out
    dev = db.device.device
    row_scale = torch.empty(db.shape[0], dtype=torch.float32, device=dev) if db.info["has_row_scale"] else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sym = torch.empty(db.shape, dtype=torch.uint8, device=dev) if symbols else None
    decode_into(db, out, row_scale, status, stream, sym)
    sync_status(status, stream)
    return (out, row_scale, sym) if symbols else (out, row_scale)


class BatchDecoder:
    """Decode many streams in one persistent launch (ep_batch_prepare / ep_batch_decode).

    ``outs[i]`` receives stream ``blobs[i]``.  With ``ring = R > 0`` output
    buffers may repeat with period R (item i reuses item i - R's buffer) and
    the kernel orders the writes; with ``ring = 0`` outputs must be distinct.
    """

    def __init__(self, blobs, outs, ring: int = 0, row_scales=None):
        if len(blobs) != len(outs) or not blobs:
            raise ValueError("need one output per stream")
        dev = blobs[0].device.device
        self.blobs, self.outs, self.row_scales = list(blobs), list(outs), row_scales
        n = len(blobs)
        items = (EpBatchItem * n)()
        for i, (b, o) in enumerate(zip(blobs, outs)):
            rs = None if row_scales is None else row_scales[i]
            items[i] = EpBatchItem(b.host.data_ptr(), b.device.data_ptr(), b.nbytes, o.data_ptr(),
                                   0 if rs is None else rs.data_ptr())
        ws_bytes = lib.ep_batch_workspace_bytes(n)
        self.workspace = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        self.plan = EpBatchPlan()
        check(lib.ep_batch_prepare(items, n, int(ring), _ptr(self.workspace), ws_bytes, ctypes.byref(self.plan)),
              "ep_batch_prepare")
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def launch(self, stream=None, status: torch.Tensor | None = None) -> None:
        st = self.status if status is None else status
        check(lib.ep_batch_decode(ctypes.byref(self.plan), _ptr(st), _stream_handle(stream)), "ep_batch_decode")

    def __call__(self, stream=None) -> None:
        self.launch(stream)
        sync_status(self.status, stream)


# ------------------------------------------------------------------ linear
LINEAR_DECODE_THEN_GEMM, LINEAR_FUSED = 0, 1


def _check_bf16_2d(t: torch.Tensor, name: str) -> None:
    if t.dtype != torch.bfloat16 or t.dim() != 2 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D BF16 CUDA tensor")


def linear_bf16(x: torch.Tensor, w: torch.Tensor, out: torch.Tensor | None = None, status=None, stream=None):
    """ep_linear_bf16: Y = X W^T on the tcgen05 GEMM (dense BF16 W)."""
    _check_bf16_2d(x, "x")
    _check_bf16_2d(w, "w")
    if x.shape[1] != w.shape[1]:
        raise ValueError("x and w disagree on in_features")
    y = torch.empty((x.shape[0], w.shape[0]), dtype=torch.bfloat16, device=x.device) if out is None else out
    st = torch.zeros(1, dtype=torch.int32, device=x.device) if status is None else status
    check(lib.ep_linear_bf16(_ptr(x), _ptr(w), _ptr(y), x.shape[0], w.shape[0], w.shape[1], _ptr(st),
                             _stream_handle(stream)), "ep_linear_bf16")
    if status is None:
        sync_status(st, stream)
    return y


def compressed_linear(db: DeviceBlob, x: torch.Tensor, mode: int = LINEAR_DECODE_THEN_GEMM,
                      out: torch.Tensor | None = None, workspace: torch.Tensor | None = None, status=None,
                      stream=None):
    """ep_compressed_linear: Y = X W^T with W decoded from `db` by the library's kernels."""
    _check_bf16_2d(x, "x")
    rows, cols = db.shape
    if x.shape[1] != cols:
        raise ValueError("x does not match the stream's in_features")
    y = torch.empty((x.shape[0], rows), dtype=torch.bfloat16, device=x.device) if out is None else out
    if mode == LINEAR_DECODE_THEN_GEMM and workspace is None:
        workspace = torch.empty(rows * cols, dtype=torch.bfloat16, device=x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = torch.zeros(1, dtype=torch.int32, device=x.device) if status is None else status
    check(lib.ep_compressed_linear(_ptr(db.host), _ptr(db.device), db.nbytes, _ptr(x), x.shape[0], _ptr(y),
                                   int(mode), _ptr(workspace), ws_bytes, _ptr(st), _stream_handle(stream)),
          "ep_compressed_linear")
    if status is None:
        sync_status(st, stream)
    return y


# ------------------------------------------------------------ tensor-level API
@dataclass
class EntroPackLossyConfig:
    """Lossy E8 compression at a target bitrate (bits per parameter of coded payload)."""
    target_bpp: float = 4.0
    container: str = "bf16"
    sample_frac: float = 0.05


@dataclass
class TileANSConfig:
    """Lossless tiled ANS: the exponent byte (FP8: the whole element) entropy coded, the rest raw.

    Supported element types: BF16, FP16, FP8 e4m3 and FP32 (the tensor's own dtype).
    """


class CompressedTensor:
    def __init__(self, blob: bytes, config, device="cuda"):
        self.config = config
        self.blob = DeviceBlob(blob, device=device)

    @property
    def target_bpp(self) -> float:
        return self.blob.info["target_bpp"]

    @property
    def actual_bpp(self) -> float:
        return self.blob.info["actual_bpp"]

    @property
    def shape(self):
        return self.blob.shape


def compress(tensor: torch.Tensor, config=None, device="cuda") -> CompressedTensor:
    config = config or EntroPackLossyConfig()
    if isinstance(config, TileANSConfig):
        if tensor.dtype not in _TORCH_TO_LOSSLESS:
            raise TypeError(f"lossless compression supports bf16, fp16, float8_e4m3fn and fp32, not {tensor.dtype}")
        blob = encode(tensor, lossless=True)
    else:
        blob = encode(bf16_bits(tensor), config.target_bpp, config.container, sample_frac=config.sample_frac)
    return CompressedTensor(blob, config, device=device)


def decompress(ct: CompressedTensor, stream=None):
    """Decode to the container dtype; FP8/INT8 return (weights, per-row scales)."""
    out, scale = decode(ct.blob, stream=stream)
    return (out, scale) if scale is not None else out


class CompressedLinear(torch.nn.Module):
    """Linear layer whose weight stays entropy-coded in HBM and is decoded on each call.

    forward(x) = x @ W^T (+ bias): ep_compressed_linear decodes W with the
    library's decode kernel into a BF16 workspace and multiplies on the
    tcgen05 GEMM kernel; any leading batch dimensions of x are flattened.
    """

    def __init__(self, ct: CompressedTensor, bias: torch.Tensor | None = None):
        super().__init__()
        if ct.blob.info["container"] != 0:
            raise ValueError("CompressedLinear needs a BF16 container")
        self.ct = ct
        self.out_features, self.in_features = ct.shape
        self.bias = None if bias is None else torch.nn.Parameter(bias.detach().to(torch.bfloat16), requires_grad=False)
        self._ws = None
        self._status = None

    @classmethod
    def from_linear(cls, linear: torch.nn.Linear, config=None, device="cuda"):
        w = linear.weight.detach().to(torch.bfloat16)
        ct = compress(w, config or EntroPackLossyConfig(), device=device)
        bias = None if linear.bias is None else linear.bias.detach().to(device)
        return cls(ct, bias)

    def decoded_weight(self, stream=None) -> torch.Tensor:
        dev = self.ct.blob.device.device
        if self._ws is None:
            self._ws = torch.empty(self.ct.shape, dtype=torch.bfloat16, device=dev)
            self._status = torch.zeros(1, dtype=torch.int32, device=dev)
        decode_into(self.ct.blob, self._ws, None, self._status, stream)
        return self._ws

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        dev = self.ct.blob.device.device
        if self._ws is None:
            self._ws = torch.empty(self.ct.shape, dtype=torch.bfloat16, device=dev)
            self._status = torch.zeros(1, dtype=torch.int32, device=dev)
        lead = x.shape[:-1]
        x2 = x.reshape(-1, x.shape[-1]).to(torch.bfloat16).contiguous()
        y = compressed_linear(self.ct.blob, x2, LINEAR_DECODE_THEN_GEMM, workspace=self._ws, status=self._status)
        if self.bias is not None:
            y = y + self.bias
        return y.reshape(*lead, self.out_features)

    def check_status(self):
        if self._status is not None:
            sync_status(self._status)


__all__ = ["encode", "query", "actual_bpp", "DeviceBlob", "decode", "decode_into", "sync_status", "BatchDecoder",
           "linear_bf16", "compressed_linear", "LINEAR_DECODE_THEN_GEMM", "LINEAR_FUSED",
           "EntroPackLossyConfig", "TileANSConfig", "CompressedTensor", "compress", "decompress",
           "CompressedLinear", "EntroPackError", "CONTAINERS", "CONTAINER_DTYPES"]
