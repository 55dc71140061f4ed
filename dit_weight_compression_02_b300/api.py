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

from ._lib import EpBatchItem, EpBatchPlan, EpInfo, EpLayerRef, EpParams, EntroPackError, check, lib

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
           sample_frac: float = 0.05, n_threads: int = 0, j: int | None = None) -> bytes:
    """ep_encode: a rows x cols matrix -> stream bytes.

    Lossy: BF16 bits in, decoded into `container`.  Lossless: elements of the
    type `container` names (bf16, fp16, fp8 or fp32; a torch tensor's own
    dtype is used when it is one of those), restored bit for bit.  With `j`
    (lossy only) the stream is coded at that resolution index through
    ep_encode_at, with no rate search.
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
    if j is not None:
        if lossless:
            raise ValueError("a resolution index applies to lossy streams only")
        check(lib.ep_encode_at(_ptr(w_bits), w_bits.shape[0], w_bits.shape[1], ctypes.byref(p), int(j),
                               ctypes.byref(out), ctypes.byref(size)), "ep_encode_at")
    else:
        check(lib.ep_encode(_ptr(w_bits), w_bits.shape[0], w_bits.shape[1], ctypes.byref(p), ctypes.byref(out),
                            ctypes.byref(size)), "ep_encode")
    try:
        return ctypes.string_at(out, size.value)
    finally:
        lib.ep_free(out)


def estimate_bpp(w_bits, j: int, sample_frac: float = 0.05, n_threads: int = 0):
    """ep_estimate_bpp: (sampled coded bits per parameter at index j, smallest admissible index)."""
    w = bf16_bits(w_bits)
    bpp = ctypes.c_double(0.0)
    jmin = ctypes.c_int32(0)
    check(lib.ep_estimate_bpp(_ptr(w), w.shape[0], w.shape[1], float(sample_frac), int(j), int(n_threads),
                              ctypes.byref(bpp), ctypes.byref(jmin)), "ep_estimate_bpp")
    return bpp.value, jmin.value


def allocate_bits(weights, avg_bpp: float, sensitivities=None, sample_frac: float = 0.05, n_threads: int = 0) -> dict:
    """ep_allocate_bits: per-layer resolution indices for a model-level storage budget.

    weights: BF16 matrices (tensors or uint16 arrays); sensitivities: one
    positive weight per layer for its squared relative error (default 1).
    Returns {"t": shared index, "j": [...], "est_bpp": [...]}.
    """
    mats = [bf16_bits(w) for w in weights]
    n = len(mats)
    sens = [1.0] * n if sensitivities is None else [float(a) for a in sensitivities]
    if len(sens) != n:
        raise ValueError("one sensitivity per layer")
    refs = (EpLayerRef * n)(*[EpLayerRef(m.ctypes.data, m.shape[0], m.shape[1], a) for m, a in zip(mats, sens)])
    js = np.zeros(n, dtype=np.int32)
    est = np.zeros(n, dtype=np.float64)
    t = ctypes.c_int32(0)
    check(lib.ep_allocate_bits(refs, n, float(avg_bpp), float(sample_frac), int(n_threads), _ptr(js), _ptr(est),
                               ctypes.byref(t)), "ep_allocate_bits")
    return {"t": t.value, "j": [int(v) for v in js], "est_bpp": [float(v) for v in est]}


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
        # the stream validated once (ep_stream_open): hot paths launch from it
        # without parsing the host copy again
        self.handle = ctypes.c_void_p(0)
        check(lib.ep_stream_open(_ptr(self.host), self.nbytes, ctypes.byref(self.handle)), "ep_stream_open")

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            try:
                lib.ep_stream_close(h)
            except Exception:  # interpreter shutdown
                pass
            self.handle = ctypes.c_void_p(0)

    @property
    def shape(self):
        return (self.info["rows"], self.info["cols"])

    @property
    def out_dtype(self):
        return CONTAINER_DTYPES[self.info["container"]]

    def alloc_out(self):
        return torch.empty(self.shape, dtype=self.out_dtype, device=self.device.device)


def decode_into(db: DeviceBlob, out: torch.Tensor, row_scale: torch.Tensor | None, status: torch.Tensor,
                stream=None, sym_out: torch.Tensor | None = None, validated: bool = False) -> None:
    """Enqueue ep_decode (or ep_decode_symbols) on `stream`; no synchronisation.

    validated=True launches from the stream handle (ep_decode_h): the host copy
    was validated when the DeviceBlob was made and is not parsed again."""
    if validated and sym_out is None:
        check(lib.ep_decode_h(db.handle, _ptr(db.device), _ptr(out), _ptr(row_scale), _ptr(status),
                              _stream_handle(stream)), "ep_decode_h")
        return
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


class StreamingDecoder:
    """Decode streams whose bytes live in pinned host memory, uploading as it goes.

    The streams are taken in chunks of ``chunk`` consecutive items.  Each
    launch copies chunk k's bytes to the device on a copy stream and decodes
    chunk k on the compute stream (ep_batch_decode) as soon as they land, so
    the upload of chunk k + 1 overlaps the decode of chunk k.  Outputs must be
    distinct within a chunk and may repeat across chunks (decodes of
    successive chunks run in order on one stream).  The next launch's upload
    of a chunk waits for the previous launch's decode of it.
    """

    def __init__(self, blobs, outs, chunk: int = 7):
        if len(blobs) != len(outs) or not blobs or chunk < 1:
            raise ValueError("need one output per stream and a positive chunk")
        self.blobs = list(blobs)
        dev = self.blobs[0].device.device
        self.chunks = []
        for c0 in range(0, len(self.blobs), chunk):
            idx = list(range(c0, min(c0 + chunk, len(self.blobs))))
            if len({outs[i].data_ptr() for i in idx}) != len(idx):
                raise ValueError("outputs must be distinct within a chunk")
            self.chunks.append((idx, BatchDecoder([self.blobs[i] for i in idx], [outs[i] for i in idx])))
        self.status = torch.zeros(len(self.chunks), dtype=torch.int32, device=dev)
        self._any = torch.zeros(1, dtype=torch.int32, device=dev)
        self.copy_stream = torch.cuda.Stream(device=dev)
        self._landed = [torch.cuda.Event() for _ in self.chunks]
        self._decoded = [torch.cuda.Event() for _ in self.chunks]
        self._launched = False

    @property
    def upload_bytes(self) -> int:
        return sum(b.nbytes for b in self.blobs)

    def launch(self, stream=None) -> None:
        stream = torch.cuda.current_stream() if stream is None else stream
        for k, (idx, dec) in enumerate(self.chunks):
            with torch.cuda.stream(self.copy_stream):
                if self._launched:
                    self.copy_stream.wait_event(self._decoded[k])  # the previous decode of these bytes is done
                for i in idx:
                    self.blobs[i].device.copy_(self.blobs[i].host, non_blocking=True)
                self._landed[k].record(self.copy_stream)
            stream.wait_event(self._landed[k])
            dec.launch(stream, self.status[k:k + 1])
            self._decoded[k].record(stream)
        self._launched = True

    def check(self, stream=None) -> None:
        """Synchronise and raise EntroPackError if any chunk's decode reported corruption."""
        stream = torch.cuda.current_stream() if stream is None else stream
        with torch.cuda.stream(stream):
            torch.amax(self.status, dim=0, keepdim=True, out=self._any)
        sync_status(self._any, stream)

    def __call__(self, stream=None) -> None:
        self.launch(stream)
        self.check(stream)


# ------------------------------------------------------------------ linear
LINEAR_DECODE_THEN_GEMM, LINEAR_FUSED = 0, 1


def _check_bf16_2d(t: torch.Tensor, name: str) -> None:
    if t.dtype != torch.bfloat16 or t.dim() != 2 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D BF16 CUDA tensor")


def _check_bias(bias: torch.Tensor | None, rows: int) -> None:
    if bias is not None and (bias.dtype != torch.bfloat16 or bias.dim() != 1 or bias.shape[0] != rows
                             or not bias.is_cuda or not bias.is_contiguous()):
        raise ValueError("bias must be a contiguous 1-D BF16 CUDA tensor of out_features elements")


def linear_bf16(x: torch.Tensor, w: torch.Tensor, out: torch.Tensor | None = None, status=None, stream=None,
                bias: torch.Tensor | None = None):
    """ep_linear_bf16: Y = X W^T (+ bias) on the tcgen05 GEMM (dense BF16 W)."""
    _check_bf16_2d(x, "x")
    _check_bf16_2d(w, "w")
    if x.shape[1] != w.shape[1]:
        raise ValueError("x and w disagree on in_features")
    _check_bias(bias, w.shape[0])
    y = torch.empty((x.shape[0], w.shape[0]), dtype=torch.bfloat16, device=x.device) if out is None else out
    st = torch.zeros(1, dtype=torch.int32, device=x.device) if status is None else status
    check(lib.ep_linear_bf16(_ptr(x), _ptr(w), _ptr(y), _ptr(bias), x.shape[0], w.shape[0], w.shape[1], _ptr(st),
                             _stream_handle(stream)), "ep_linear_bf16")
    if status is None:
        sync_status(st, stream)
    return y


def compressed_linear(db: DeviceBlob, x: torch.Tensor, mode: int = LINEAR_DECODE_THEN_GEMM,
                      out: torch.Tensor | None = None, workspace: torch.Tensor | None = None, status=None,
                      stream=None, bias: torch.Tensor | None = None):
    """ep_compressed_linear: Y = X W^T (+ bias) with W decoded from `db` by the library's kernels.

    mode LINEAR_DECODE_THEN_GEMM decodes W into a BF16 workspace and runs the
    tensor-core GEMM on it; LINEAR_FUSED decodes W straight into shared memory
    as the tensor-core operand (no workspace; in_features % 128 == 0; tokens in
    passes of fused_tokens_per_pass(in_features), each decoding W again).
    """
    _check_bf16_2d(x, "x")
    rows, cols = db.shape
    if x.shape[1] != cols:
        raise ValueError("x does not match the stream's in_features")
    _check_bias(bias, rows)
    y = torch.empty((x.shape[0], rows), dtype=torch.bfloat16, device=x.device) if out is None else out
    if mode == LINEAR_DECODE_THEN_GEMM and workspace is None:
        workspace = torch.empty(rows * cols, dtype=torch.bfloat16, device=x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = torch.zeros(1, dtype=torch.int32, device=x.device) if status is None else status
    # launched from the stream handle: the host copy was validated when the DeviceBlob was made
    check(lib.ep_compressed_linear_h(db.handle, _ptr(db.device), _ptr(x), x.shape[0], _ptr(y), _ptr(bias),
                                     int(mode), _ptr(workspace), ws_bytes, _ptr(st), _stream_handle(stream)),
          "ep_compressed_linear_h")
    if status is None:
        sync_status(st, stream)
    return y


def fused_tokens_per_pass(in_features: int) -> int:
    """ep_fused_tokens_per_pass: tokens one fused pass covers (0: the shape is not served)."""
    return int(lib.ep_fused_tokens_per_pass(int(in_features)))


# ------------------------------------------------- fixed-width comparators
Q4_KINDS = {"nf4": 0, "int4": 1}


def q4_levels(kind: str = "nf4") -> np.ndarray:
    """ep_q4_levels: the 16 FP32 levels of the NF4 or INT4 comparator codebook."""
    lv = np.zeros(16, dtype=np.float32)
    check(lib.ep_q4_levels(Q4_KINDS[kind], _ptr(lv)), "ep_q4_levels")
    return lv


@dataclass
class Q4Tensor:
    """A block-absmax 4-bit comparator encoding (host arrays)."""
    codes: np.ndarray  # uint8, n / 2 (two codes per byte, low nibble first)
    scales: np.ndarray  # float32, one per block
    levels: np.ndarray  # float32[16]
    shape: tuple
    block: int

    @property
    def bits_per_weight(self) -> float:
        n = int(np.prod(self.shape))
        return 8.0 * (self.codes.nbytes + self.scales.nbytes) / n


def q4_encode(w_bits, kind: str = "nf4", block: int = 64, n_threads: int = 0) -> Q4Tensor:
    """ep_q4_encode: NF4 / INT4 encoding of BF16 weights on the host."""
    w = bf16_bits(w_bits)
    n = w.size
    codes = np.zeros(n // 2 + (n & 1), dtype=np.uint8)
    scales = np.zeros((n + block - 1) // block, dtype=np.float32)
    lv = q4_levels(kind)
    check(lib.ep_q4_encode(_ptr(w), n, block, _ptr(lv), _ptr(codes), _ptr(scales), int(n_threads)), "ep_q4_encode")
    return Q4Tensor(codes, scales, lv, tuple(w.shape), block)


def q4_decode(codes: torch.Tensor, scales: torch.Tensor, levels: np.ndarray, shape, block: int = 64,
              out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """ep_q4_decode: BF16 reconstruction of a comparator encoding on the GPU (device codes / scales)."""
    n = int(np.prod(shape))
    y = torch.empty(shape, dtype=torch.bfloat16, device=codes.device) if out is None else out
    lv = np.ascontiguousarray(levels, dtype=np.float32)
    check(lib.ep_q4_decode(_ptr(codes), _ptr(scales), n, block, _ptr(lv), _ptr(y), _stream_handle(stream)),
          "ep_q4_decode")
    return y


def fp8_row_encode(w_bits, n_threads: int = 0):
    """ep_fp8_row_encode: per-row-scaled FP8 E4M3 comparator on the host -> (codes uint8, FP32 row scales)."""
    w = bf16_bits(w_bits)
    if w.ndim != 2:
        raise ValueError("expected a 2-D weight matrix")
    codes = np.zeros(w.shape, dtype=np.uint8)
    scales = np.zeros(w.shape[0], dtype=np.float32)
    check(lib.ep_fp8_row_encode(_ptr(w), w.shape[0], w.shape[1], _ptr(codes), _ptr(scales), int(n_threads)),
          "ep_fp8_row_encode")
    return codes, scales


def fp8_row_decode(codes: torch.Tensor, scales: torch.Tensor, out: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """ep_fp8_row_decode: BF16 reconstruction of the FP8 comparator on the GPU."""
    rows, cols = codes.shape
    y = torch.empty((rows, cols), dtype=torch.bfloat16, device=codes.device) if out is None else out
    check(lib.ep_fp8_row_decode(_ptr(codes), _ptr(scales), rows, cols, _ptr(y), _stream_handle(stream)),
          "ep_fp8_row_decode")
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
        decode_into(self.ct.blob, self._ws, None, self._status, stream, validated=True)
        return self._ws

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        dev = self.ct.blob.device.device
        if self._ws is None:
            self._ws = torch.empty(self.ct.shape, dtype=torch.bfloat16, device=dev)
            self._status = torch.zeros(1, dtype=torch.int32, device=dev)
        lead = x.shape[:-1]
        x2 = x.reshape(-1, x.shape[-1]).to(torch.bfloat16).contiguous()
        y = compressed_linear(self.ct.blob, x2, LINEAR_DECODE_THEN_GEMM, workspace=self._ws, status=self._status,
                              bias=self.bias)  # the bias is added in the GEMM's epilogue
        return y.reshape(*lead, self.out_features)

    def check_status(self):
        if self._status is not None:
            sync_status(self._status)


def compress_linears(linears: dict, avg_bpp: float, sensitivities: dict | None = None, sample_frac: float = 0.05,
                     device="cuda"):
    """Compress several linear layers under one storage budget (ep_allocate_bits + ep_encode_at).

    linears: name -> torch.nn.Linear; sensitivities: name -> alpha (default 1).
    Returns (name -> CompressedLinear, record), where the record keeps, per
    layer, the sensitivity, the resolution index, the estimated and the actual
    bits per parameter, so the allocation can be reproduced and explained.
    """
    names = list(linears)
    weights = [linears[k].weight.detach().to(torch.bfloat16) for k in names]
    sens = [float((sensitivities or {}).get(k, 1.0)) for k in names]
    plan = allocate_bits(weights, avg_bpp, sens, sample_frac)
    out, record = {}, {"avg_bpp_budget": float(avg_bpp), "shared_index": plan["t"], "layers": {}}
    for k, w, a, j, e in zip(names, weights, sens, plan["j"], plan["est_bpp"]):
        blob = encode(bf16_bits(w), e, "bf16", sample_frac=sample_frac, j=j)
        ct = CompressedTensor(blob, EntroPackLossyConfig(e, "bf16", sample_frac), device=device)
        lin = linears[k]
        out[k] = CompressedLinear(ct, None if lin.bias is None else lin.bias.detach().to(device))
        record["layers"][k] = {"sensitivity": a, "j": j, "est_bpp": e, "actual_bpp": ct.actual_bpp,
                               "params": int(w.numel())}
    n_tot = sum(v["params"] for v in record["layers"].values())
    record["actual_bpp"] = sum(v["actual_bpp"] * v["params"] for v in record["layers"].values()) / n_tot
    return out, record


__all__ = ["encode", "query", "actual_bpp", "DeviceBlob", "decode", "decode_into", "sync_status", "BatchDecoder",
           "StreamingDecoder",
           "linear_bf16", "compressed_linear", "fused_tokens_per_pass", "LINEAR_DECODE_THEN_GEMM", "LINEAR_FUSED",
           "EntroPackLossyConfig", "TileANSConfig", "CompressedTensor", "compress", "decompress",
           "CompressedLinear", "EntroPackError", "CONTAINERS", "CONTAINER_DTYPES",
           "q4_levels", "q4_encode", "q4_decode", "Q4Tensor", "Q4_KINDS", "fp8_row_encode", "fp8_row_decode",
           "estimate_bpp", "allocate_bits", "compress_linears"]
