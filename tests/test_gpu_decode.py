"""GPU parity of the decode kernels against the CPU oracle (bit-exact).

For every configured workload the oracle encodes the weights, decodes them on
the CPU (container values, FP8/INT8 row scales, and the coded symbol byte of
every coordinate), and the sm_103a kernels decode the same stream through the
C ABI.  All of these must agree bit for bit.  Also covered: ragged tile
groups, single tiles, zero tensors, escape-heavy streams, long lanes (8 bpp),
device-side corruption reporting, the batched launch and its ring ordering.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    import dit_weight_compression_02_b300 as m
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return m


def _np(t: torch.Tensor) -> np.ndarray:
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).cpu().numpy()
    return t.cpu().numpy()


def _check(ep, blob, expect_bits=None):
    y_o, rs_o = oracle.decode_threaded(blob)
    sym_o = oracle.decode_symbols(blob)
    db = ep.DeviceBlob(blob)
    y_g, rs_g, sym_g = ep.decode(db, symbols=True)
    y_g, sym_g = _np(y_g), sym_g.cpu().numpy()
    assert (sym_g == sym_o).all(), f"symbol mismatch at {np.argwhere(sym_g != sym_o)[:5]}"
    bad = np.argwhere(y_g != y_o)
    assert bad.size == 0, f"{len(bad)} container mismatches, first {bad[:5]}"
    if rs_o is not None:
        assert (rs_g.cpu().numpy().view(np.uint32) == rs_o.view(np.uint32)).all()
    if expect_bits is not None:
        assert (y_g == expect_bits).all()
    # the plain decode path (no symbol dump) gives the same values
    y2, _ = ep.decode(db)
    assert (_np(y2) == y_o).all()
    return y_g


def test_c1_256x1024(ep):
    w = synth.normal_bf16(1, 256, 1024)
    blob = oracle.encode(w, 4.0)
    y = _check(ep, blob)
    W = synth.bf16_to_f32(w).astype(np.float64)
    rel = np.linalg.norm(oracle.container_to_f64(y, "bf16") - W) / np.linalg.norm(W)
    assert rel < 0.075 and 8 * len(blob) / w.size > 4.0


@pytest.mark.parametrize("target", [2.5, 3.0, 3.5, 4.0, 4.5])
def test_c2_4096_sweep(ep, target):
    w = synth.rows_outliers_bf16(2, 4096, 4096)
    _check(ep, oracle.encode(w, target))


@pytest.mark.parametrize("rows,cols,seed", [(3840, 3840, 3), (10240, 3840, 7), (3840, 10240, 9)])
def test_c3_layer_shapes(ep, rows, cols, seed):
    w = synth.student_t5_bf16(seed, rows, cols)
    _check(ep, oracle.encode(w, 4.0))


@pytest.mark.parametrize("container", ["fp16", "fp8", "int8"])
def test_c4a_containers_8192(ep, container):
    w = synth.normal_bf16(4, 8192, 8192)
    _check(ep, oracle.encode(w, 3.0, container))


def test_c4b_lossless_8192_specials(ep):
    w = synth.with_special_rows(synth.normal_bf16(4, 8192, 8192), seed=4)
    _check(ep, oracle.encode_lossless(w), expect_bits=w)


@pytest.mark.parametrize("dtype", ["fp16", "fp8", "fp32"])
@pytest.mark.parametrize("rows,cols", [(512, 1024), (45, 200), (8192, 1024)])
def test_lossless_other_dtypes(ep, dtype, rows, cols):
    npt = oracle.LOSSLESS_DTYPES[dtype][1]
    rng = np.random.default_rng(rows + cols)
    if dtype == "fp8":
        w = rng.integers(0, 256, size=(rows, cols), dtype=np.uint16).astype(np.uint8)
    else:
        # realistic exponents plus special values, so the coded byte is skewed
        f = rng.standard_normal((rows, cols)).astype(np.float32) * 0.02
        w = f.view(np.uint32) if dtype == "fp32" else f.astype(np.float16).view(np.uint16)
        w[0, :4] = [0, np.iinfo(npt).max, 1, 0]
    blob = oracle.encode_lossless(w, dtype)
    y_o, _ = oracle.decode(blob)
    db = ep.DeviceBlob(blob)
    y_g, rs, sym = ep.decode(db, symbols=True)
    assert rs is None
    as_bits = {"fp16": torch.int16, "fp8": torch.uint8, "fp32": torch.int32}[dtype]
    assert (y_g.view(as_bits).cpu().numpy().view(npt) == w).all() and (y_o == w).all()
    assert (sym.cpu().numpy() == oracle.decode_symbols(blob)).all()
    y2, _ = ep.decode(db)  # the production path (no symbol dump)
    assert (y2.view(as_bits).cpu().numpy().view(npt) == w).all()


def test_lossless_other_dtypes_batched(ep):
    rng = np.random.default_rng(3)
    ws = [rng.standard_normal((r, c)).astype(np.float32).view(np.uint32) for r, c in [(256, 512), (45, 200), (96, 384)]]
    blobs = [oracle.encode_lossless(w, "fp32") for w in ws]
    dbs = [ep.DeviceBlob(b) for b in blobs]
    outs = [d.alloc_out() for d in dbs]
    ep.BatchDecoder(dbs, outs, ring=0)()
    for w, o in zip(ws, outs):
        assert (o.view(torch.int32).cpu().numpy().view(np.uint32) == w).all()


def test_lossless_every_bf16_pattern(ep):
    w = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(512, 128)
    _check(ep, oracle.encode_lossless(w), expect_bits=w)


def test_large_matrix_two_lanes_per_thread(ep):
    # 16384 x 10240 = 40960 tiles = 5120 groups of 8: more than one wave of
    # warps, so the single-stream decode runs two lanes per thread (odd job
    # counts and ragged tails included in the grid's last CTAs)
    w = synth.student_t5_bf16(77, 16384, 10240)
    blob = oracle.encode(w, 4.0)
    db = ep.DeviceBlob(blob)
    y, _ = ep.decode(db)
    assert (_np(y) == oracle.decode_threaded(blob)[0]).all()


@pytest.mark.parametrize("rows,cols", [(32, 128), (96, 384), (224, 640), (32, 128 * 13)])
def test_ragged_and_single_tiles(ep, rows, cols):
    # 1, 9, 35 and 13 tiles: tile groups of 8 that end part-way
    w = synth.student_t5_bf16(rows + cols, rows, cols)
    _check(ep, oracle.encode(w, 4.0))
    _check(ep, oracle.encode(w, 3.0, "fp8"))


@pytest.mark.parametrize("rows,cols", [(1, 8), (45, 200), (33, 136), (100, 1000), (31, 120), (257, 3848)])
def test_general_shapes(ep, rows, cols):
    # tiles cover the matrix padded to 32 x 128 multiples; the GPU writes only
    # the true rows x cols values (row stride cols), bit for bit as the oracle
    w = synth.student_t5_bf16(rows * 3 + cols, rows, cols)
    for container in ("bf16", "fp16", "fp8", "int8"):
        _check(ep, oracle.encode(w, 4.0, container))
    _check(ep, oracle.encode_lossless(w), expect_bits=w)


def test_general_shapes_batched(ep):
    ws = [synth.student_t5_bf16(500 + i, r, c) for i, (r, c) in enumerate([(45, 200), (100, 1000), (1, 8), (33, 136)])]
    blobs = [oracle.encode(w, 4.0) for w in ws]
    dbs = [ep.DeviceBlob(b) for b in blobs]
    outs = [torch.full(d.shape, 5.0, dtype=torch.bfloat16, device="cuda") for d in dbs]
    ep.BatchDecoder(dbs, outs, ring=0)()
    for b, o in zip(blobs, outs):
        assert (_np(o) == oracle.decode(b)[0]).all()


def test_zero_and_constant_tensors(ep):
    _check(ep, oracle.encode(np.zeros((64, 256), np.uint16), 4.0))
    _check(ep, oracle.encode(np.full((64, 256), 0x3C4A, np.uint16), 4.0, "int8"))
    _check(ep, oracle.encode_lossless(np.zeros((64, 256), np.uint16)))


@pytest.mark.parametrize("container", ["bf16", "fp16", "fp8", "int8"])
def test_escape_heavy(ep, container):
    w = synth.rows_outliers_bf16(9, 256, 1024, frac=0.05, k_sigma=40.0)
    blob = oracle.encode(w, 6.0, container)
    assert (oracle.decode_symbols(blob)[:, 1::8] == 0).sum() > 100
    _check(ep, blob)


@pytest.mark.parametrize("container", ["bf16", "int8"])
def test_escapes_in_every_lanes_last_block(ep, container):
    # outliers in the last row of every tile's last K-slab: each lane's final
    # block (step 127) escapes, so the latency-bound decode's speculative
    # decode of the block after the last one is rolled back on the escape
    # path, and the lane must still end exactly at its last word
    w = synth.normal_bf16(17, 256, 1024)
    f = synth.bf16_to_f32(w)
    for q in range(4):  # the first coordinate of each lane's last block
        f[31::32, 96 + 8 * q::128] = 2.0 if q % 2 else -2.0
    w = (f.view(np.uint32) >> 16).astype(np.uint16)
    blob = oracle.encode(w, 7.0, container)
    sym = oracle.decode_symbols(blob)
    for q in range(4):  # s0 escaped: its byte is the coset bit, 0 or 1
        assert (sym[31::32, 96 + 8 * q::128] <= 1).all()
    _check(ep, blob)
    # the same stream through the batched kernel
    db = ep.DeviceBlob(blob)
    out = db.alloc_out()
    ep.BatchDecoder([db], [out], ring=0)()
    assert (_np(out) == oracle.decode(blob)[0]).all()


def test_long_lanes_8bpp(ep):
    _check(ep, oracle.encode(synth.normal_bf16(13, 256, 1024), 8.0))


def _status_after(ep, blob_host, blob_dev_bytes):
    db = ep.DeviceBlob(blob_host)
    db.device.copy_(torch.from_numpy(np.frombuffer(blob_dev_bytes, dtype=np.uint8).copy()).cuda())
    out = db.alloc_out()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.decode_into(db, out, None, status)
    torch.cuda.synchronize()
    return int(status.item())


def test_device_side_corruption_is_reported(ep):
    w = synth.normal_bf16(14, 256, 1024)
    blob = oracle.encode(w, 4.0)
    h = oracle.header(blob)
    b = bytearray(blob)
    for off in range(h["payload_off"] + 200, h["payload_off"] + 2000, 97):  # flip words in the first tiles
        b[off] ^= 0xFF
    assert _status_after(ep, blob, bytes(b)) & 0x1  # lane end state / word count
    b = bytearray(blob)
    big = np.array([1 << 40], dtype=np.uint64).tobytes()
    b[h["offsets_off"] + 8 * 3: h["offsets_off"] + 8 * 4] = big  # tile offset far outside the stream
    assert _status_after(ep, blob, bytes(b)) & 0x2
    assert _status_after(ep, blob, blob) == 0


def test_host_validation_rejects_before_launch(ep):
    blob = bytearray(oracle.encode(synth.normal_bf16(15, 64, 256), 4.0))
    db = ep.DeviceBlob(bytes(blob))
    blob[60] ^= 1  # tables offset
    db.host.copy_(torch.from_numpy(np.frombuffer(bytes(blob), dtype=np.uint8).copy()))
    with pytest.raises(ep.EntroPackError) as e:
        ep.decode(db)
    assert e.value.status == "EP_ERR_CORRUPT"


def _model_layers(n_blocks, hidden=3840, ffn=10240, seed=3):
    shapes = []
    for _ in range(n_blocks):
        shapes += [(hidden, hidden)] * 4 + [(ffn, hidden)] * 2 + [(hidden, ffn)]
    return [synth.student_t5_bf16(seed + i, r, c) for i, (r, c) in enumerate(shapes)]


def test_batch_distinct_outputs_matches_oracle(ep):
    ws = _model_layers(1)
    blobs = [oracle.encode(w, 4.0) for w in ws]
    dbs = [ep.DeviceBlob(b) for b in blobs]
    outs = [d.alloc_out() for d in dbs]
    bd = ep.BatchDecoder(dbs, outs, ring=0)
    bd()
    for b, o in zip(blobs, outs):
        assert (_np(o) == oracle.decode_threaded(b)[0]).all()


def test_batch_ring_orders_reused_buffers(ep):
    ws = [synth.student_t5_bf16(40 + i, 1024, 3840) for i in range(9)]
    blobs = [oracle.encode(w, 4.0) for w in ws]
    dbs = [ep.DeviceBlob(b) for b in blobs]
    R = 2
    bufs = [torch.empty((1024, 3840), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    bd = ep.BatchDecoder(dbs, [bufs[i % R] for i in range(len(dbs))], ring=R)
    for _ in range(3):
        bd()
        # each buffer holds the last item written to it, uncorrupted by earlier ones
        for k in range(R):
            last = max(i for i in range(len(dbs)) if i % R == k)
            assert (_np(bufs[k]) == oracle.decode_threaded(blobs[last])[0]).all()


def test_batch_fp8_row_scales(ep):
    ws = [synth.normal_bf16(50 + i, 512, 1024) for i in range(3)]
    blobs = [oracle.encode(w, 3.0, "fp8") for w in ws]
    dbs = [ep.DeviceBlob(b) for b in blobs]
    outs = [d.alloc_out() for d in dbs]
    scales = [torch.empty(512, dtype=torch.float32, device="cuda") for _ in dbs]
    ep.BatchDecoder(dbs, outs, ring=0, row_scales=scales)()
    for b, o, s in zip(blobs, outs, scales):
        y, rs = oracle.decode(b)
        assert (_np(o) == y).all()
        assert (s.cpu().numpy().view(np.uint32) == rs.view(np.uint32)).all()


def test_decode_in_cuda_graph(ep):
    w = synth.student_t5_bf16(60, 1024, 3840)
    blob = oracle.encode(w, 4.0)
    db = ep.DeviceBlob(blob)
    out = db.alloc_out()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ep.decode_into(db, out, None, status, stream=s)  # warm-up outside capture
    s.synchronize()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ep.decode_into(db, out, None, status, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert (_np(out) == oracle.decode(blob)[0]).all()


def test_compressed_linear_matches_fp64(ep):
    torch.manual_seed(0)
    w = synth.student_t5_bf16(61, 1024, 3840)
    x_bits = synth.normal_bf16(62, 256, 3840, std=1.0)
    lin = torch.nn.Linear(3840, 1024, bias=False)
    with torch.no_grad():
        lin.weight.copy_(torch.from_numpy(synth.bf16_to_f32(w)))
    cl = ep.CompressedLinear.from_linear(lin, ep.EntroPackLossyConfig(4.0))
    x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).cuda()
    y = cl(x).float().cpu().numpy().astype(np.float64)
    cl.check_status()
    blob = oracle.encode(w, 4.0)
    w_hat = oracle.container_to_f64(oracle.decode(blob)[0], "bf16")
    y_ref = oracle.gemm_f64(synth.bf16_to_f32(x_bits).astype(np.float64)[:64], w_hat)
    err = np.abs(y[:64] - y_ref).max() / np.abs(y_ref).max()
    assert err <= 2e-2, err


def test_c3_whole_model_in_bench_configuration(ep):
    """The benchmark's timed launch at full size, checked.

    30 DiT blocks at hidden 3840 (210 layers, 5.31 G params, Student-t nu = 5,
    4.0 bpp), encoded by the library, decoded by one batched launch into a ring
    of 16 reused BF16 buffers.  The status word must stay clean: every lane of
    all 1,296,000 tiles ended at x = L having consumed exactly its words, and
    no tile or escape check fired.  The ring's final contents (the last 16
    layers) are compared bit for bit with the oracle on sampled tile rows: the
    first, a middle and the last of each layer.  Then all 210 layers are
    decoded again by one batched launch into distinct buffers and every value
    of every layer is compared with the oracle.
    """
    shapes = []
    for _ in range(30):
        shapes += [(3840, 3840)] * 4 + [(10240, 3840)] * 2 + [(3840, 10240)]
    assert sum(r * c for r, c in shapes) == 5_308_416_000
    blobs = [ep.encode(synth.student_t5_bf16(3 + i, r, c), 4.0) for i, (r, c) in enumerate(shapes)]
    dbs = [ep.DeviceBlob(b, pin=False) for b in blobs]
    ring = 16
    bufs = [torch.empty(10240 * 3840, dtype=torch.bfloat16, device="cuda") for _ in range(ring)]
    outs = [bufs[i % ring][: r * c].view(r, c) for i, (r, c) in enumerate(shapes)]
    bd = ep.BatchDecoder(dbs, outs, ring=ring)
    bd()  # launches and checks the status word
    for i in range(len(shapes) - ring, len(shapes)):
        r, c = shapes[i]
        tpr = c // 128
        g = _np(outs[i])
        for tr in (0, (r // 32) // 2, r // 32 - 1):
            y_o, _ = oracle.decode(blobs[i], tr * tpr, (tr + 1) * tpr)
            rows = slice(tr * 32, tr * 32 + 32)
            assert (g[rows] == y_o[rows]).all(), (i, tr)
    del bufs, outs, bd
    # every layer, every value: the same batched launch with a distinct output
    # per layer (10.6 GB of BF16 in HBM), each layer compared with the
    # oracle's decode of it, one layer at a time to bound host memory
    outs = [torch.empty((r, c), dtype=torch.bfloat16, device="cuda") for r, c in shapes]
    ep.BatchDecoder(dbs, outs, ring=0)()
    for i, b in enumerate(blobs):
        assert (_np(outs[i]) == oracle.decode_threaded(b)[0]).all(), i
        outs[i] = None


def test_streaming_decoder_uploads_and_decodes(ep):
    """Chunks upload on a copy stream and decode as they land; outputs reused across chunks."""
    ws = [synth.student_t5_bf16(90 + i, 256, 1024) for i in range(7)]
    blobs = [oracle.encode(w, 3.5) for w in ws]
    dbs = [ep.DeviceBlob(b) for b in blobs]
    for db in dbs:
        db.device.zero_()  # the decoder must upload the bytes itself
    bufs = [torch.empty((256, 1024), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    outs = [bufs[i % 3] for i in range(7)]
    with pytest.raises(ValueError):
        ep.StreamingDecoder(dbs, outs, chunk=4)  # buffer 0 twice inside one chunk
    sd = ep.StreamingDecoder(dbs, outs, chunk=3)
    for _ in range(3):
        sd()
        for k in range(3):
            last = max(i for i in range(7) if i % 3 == k)
            assert (_np(bufs[k]) == oracle.decode(blobs[last])[0]).all()
    assert sd.upload_bytes == sum(len(b) for b in blobs)


def test_streaming_decoder_reports_corruption(ep):
    """Payload bytes that change in host memory after planning are caught by the device checks."""
    ws = [synth.normal_bf16(95 + i, 256, 1024) for i in range(4)]
    blobs = [oracle.encode(w, 4.0) for w in ws]
    dbs = [ep.DeviceBlob(b) for b in blobs]
    outs = [torch.empty((256, 1024), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    sd = ep.StreamingDecoder(dbs, outs, chunk=2)
    sd()
    h = oracle.header(blobs[3])
    host = dbs[3].host.numpy()
    saved = host.copy()
    for off in range(h["payload_off"] + 200, h["payload_off"] + 2000, 97):
        host[off] ^= 0xFF
    with pytest.raises(ep.EntroPackError) as e:
        sd()
    assert e.value.status == "EP_ERR_CORRUPT"
    host[:] = saved
    sd()  # clean again
    assert (_np(outs[3]) == oracle.decode(blobs[3])[0]).all()


def test_decode_from_validated_handle(ep):
    """ep_decode_h (the stream parsed once) matches the oracle, and device-side checks still fire."""
    w = synth.rows_outliers_bf16(97, 300, 1000)
    blob = oracle.encode(w, 3.5)
    db = ep.DeviceBlob(blob)
    out = db.alloc_out()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        ep.decode_into(db, out, None, status, validated=True)
        ep.sync_status(status)
        assert (_np(out) == oracle.decode(blob)[0]).all()
    h = oracle.header(blob)
    b = bytearray(blob)
    for off in range(h["payload_off"] + 200, h["payload_off"] + 2000, 97):
        b[off] ^= 0xFF
    db.device.copy_(torch.from_numpy(np.frombuffer(bytes(b), dtype=np.uint8).copy()).cuda())
    ep.decode_into(db, out, None, status, validated=True)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x1
