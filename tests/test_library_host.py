"""Host-side checks of libentropack.so (no GPU needed).

* the library loads and exports every function declared in include/entropack.h;
* ep_encode (the library's own threaded C++ encoder) produces byte-identical
  streams to the CPU oracle on the configured workloads (reduced sizes where
  the oracle would take minutes);
* ep_query / ep_actual_bpp / validation errors, and argument checks of the
  device entry points that return before touching the GPU.
"""
import ctypes
import os
import re

import numpy as np
import torch
import pytest

import oracle
import synth
from tests.conftest import ROOT


def _ep():
    import dit_weight_compression_02_b300 as ep
    return ep


def test_exports_every_declared_symbol():
    from dit_weight_compression_02_b300 import _lib
    hdr = open(os.path.join(ROOT, "include", "entropack.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    names = set(re.findall(r"\b(ep_[a-z_0-9]+)\s*\(", hdr))
    assert len(names) >= 10, names
    for n in sorted(names):
        assert hasattr(_lib.lib, n), f"{n} declared in entropack.h but not exported"
        assert n in _lib.SIGNATURES, f"{n} has no ctypes signature"
    assert _lib.lib.ep_version() == 1


CASES = [
    ("c1_256x1024_n002_4bpp", lambda: synth.normal_bf16(1, 256, 1024), 4.0, "bf16"),
    ("c2_1024x4096_rows_outliers_2p5", lambda: synth.rows_outliers_bf16(2, 1024, 4096), 2.5, "bf16"),
    ("c2_1024x4096_rows_outliers_4p5", lambda: synth.rows_outliers_bf16(2, 1024, 4096), 4.5, "bf16"),
    ("c3_q_3840x3840_t5_4bpp", lambda: synth.student_t5_bf16(3, 3840, 3840), 4.0, "bf16"),
    ("c4_1024x2048_fp16_3bpp", lambda: synth.normal_bf16(4, 1024, 2048), 3.0, "fp16"),
    ("c4_1024x2048_fp8_3bpp", lambda: synth.normal_bf16(4, 1024, 2048), 3.0, "fp8"),
    ("c4_1024x2048_int8_3bpp", lambda: synth.normal_bf16(4, 1024, 2048), 3.0, "int8"),
    ("escape_heavy_6bpp", lambda: synth.rows_outliers_bf16(9, 64, 512, frac=0.05, k_sigma=40.0), 6.0, "bf16"),
    ("tiny_rows_and_zero_rows", lambda: _tiny_rows(), 3.5, "int8"),
    ("ragged_45x200", lambda: synth.student_t5_bf16(30, 45, 200), 4.0, "bf16"),
    ("ragged_1x8", lambda: synth.normal_bf16(31, 1, 8), 4.0, "bf16"),
    ("ragged_100x1000_fp8", lambda: synth.normal_bf16(32, 100, 1000), 3.0, "fp8"),
    ("ragged_33x136_int8", lambda: synth.rows_outliers_bf16(33, 33, 136), 3.5, "int8"),
]


def _tiny_rows():
    w = synth.normal_bf16(10, 64, 256)
    w[0] = 0
    w[7] = synth.normal_bf16(11, 1, 256, std=1e-36)[0]
    w[9] = 0x0001  # smallest subnormal everywhere
    return w


@pytest.mark.parametrize("name,gen,target,container", CASES, ids=[c[0] for c in CASES])
def test_encoder_byte_identical_to_oracle(name, gen, target, container):
    ep = _ep()
    w = gen()
    b_lib = ep.encode(w, target, container)
    b_orc = oracle.encode(w, target, container)
    assert len(b_lib) == len(b_orc)
    assert b_lib == b_orc
    q = ep.query(b_lib)
    assert q["rows"] == w.shape[0] and q["cols"] == w.shape[1]
    assert q["actual_bpp"] == pytest.approx(8 * len(b_lib) / w.size)
    assert ep.actual_bpp(b_lib) == q["actual_bpp"]


def test_encoder_thread_count_does_not_change_bytes():
    ep = _ep()
    w = synth.rows_outliers_bf16(12, 512, 1024)
    ref = ep.encode(w, 3.5, n_threads=1)
    for t in (2, 3, 7):
        assert ep.encode(w, 3.5, n_threads=t) == ref


def test_lossless_byte_identical_and_exhaustive():
    ep = _ep()
    w = synth.with_special_rows(synth.normal_bf16(4, 512, 1024), seed=4)
    assert ep.encode(w, lossless=True) == oracle.encode_lossless(w)
    every = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(512, 128)
    assert ep.encode(every, lossless=True) == oracle.encode_lossless(every)


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp8", "fp32"])
@pytest.mark.parametrize("shape", [(64, 256), (45, 200), (1, 8), (100, 1000)])
def test_lossless_dtypes_byte_identical(dtype, shape):
    ep = _ep()
    npt = oracle.LOSSLESS_DTYPES[dtype][1]
    rng = np.random.default_rng(shape[0] * 1000 + shape[1])
    w = rng.integers(0, np.iinfo(npt).max, size=shape, dtype=npt, endpoint=True)
    blob = ep.encode(w, container=dtype, lossless=True)
    assert blob == oracle.encode_lossless(w, dtype)
    q = ep.query(blob)
    assert q["mode"] == 1 and q["container"] == oracle.LOSSLESS_DTYPES[dtype][0]
    assert q["out_elem_bytes"] == np.dtype(npt).itemsize


def test_errors():
    ep = _ep()
    w = synth.normal_bf16(5, 64, 256)
    bad = w.copy()
    bad[3, 3] = 0x7F80
    with pytest.raises(ep.EntroPackError) as e:
        ep.encode(bad)
    assert e.value.status == "EP_ERR_NONFINITE"
    with pytest.raises(ep.EntroPackError) as e:
        ep.encode(w[:, :204].copy())  # in_features not a multiple of 8
    assert e.value.status == "EP_ERR_SHAPE"
    with pytest.raises(ep.EntroPackError) as e:
        ep.encode(w[:0].copy())
    assert e.value.status == "EP_ERR_SHAPE"
    assert ep.query(ep.encode(w[:, :200].copy()))["cols"] == 200  # any multiple of 8 is accepted
    with pytest.raises(ep.EntroPackError) as e:
        ep.encode(w, target_bpp=-1.0)
    assert e.value.status == "EP_ERR_INVALID_ARG"
    # lossless accepts non-finite values
    assert oracle.decode(ep.encode(bad, lossless=True))[0][3, 3] == 0x7F80


def _flip(blob, pos, mask=0x5A):
    b = bytearray(blob)
    b[pos] ^= mask
    return bytes(b)


def test_query_rejects_corrupt_headers_and_layouts():
    ep = _ep()
    blob = ep.encode(synth.normal_bf16(6, 64, 256), 4.0)
    h = oracle.header(blob)
    for pos in (0, 4, 6, 7, 8, 16, 24, 48, 52, 53, 56, 64, 72, 80, 88,  # header fields
                h["tables_off"] + 2, h["offsets_off"] + 8, h["offsets_off"] + 8 * h["n_tiles"],
                h["payload_off"] + 16):  # a lane word count
        with pytest.raises(ep.EntroPackError) as e:
            ep.query(_flip(blob, pos))
        assert e.value.status == "EP_ERR_CORRUPT", pos
    with pytest.raises(ep.EntroPackError):
        ep.query(blob[:-16])
    with pytest.raises(ep.EntroPackError):
        ep.query(blob[:100])


def test_device_entry_points_validate_before_launch():
    """Errors found on the host return before any CUDA call (safe without a GPU)."""
    ep = _ep()
    from dit_weight_compression_02_b300._lib import lib
    blob = ep.encode(synth.normal_bf16(7, 64, 256), 4.0)
    host = np.frombuffer(blob, dtype=np.uint8)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    status = ctypes.c_void_p(1 << 21)
    # misaligned device pointers
    assert lib.ep_decode(host.ctypes.data, ctypes.c_void_p((1 << 20) + 8), len(blob), fake, None, status, None) == 1
    # corrupt host copy
    bad = np.frombuffer(_flip(blob, 0), dtype=np.uint8)
    assert lib.ep_decode(bad.ctypes.data, fake, len(blob), fake, None, status, None) == 4
    assert lib.ep_decode(host.ctypes.data, fake, len(blob) - 16, fake, None, status, None) == 4
    assert lib.ep_decode(host.ctypes.data, fake, len(blob), fake, None, None, None) == 1
    assert lib.ep_sync_status(None, None) == 1
    assert lib.ep_batch_workspace_bytes(0) == 0
    assert lib.ep_batch_workspace_bytes(5) > 0


# --------------------------------------------- fixed-width 4-bit comparators
@pytest.mark.parametrize("kind", ["nf4", "int4"])
def test_q4_levels_match_oracle(kind):
    ep = _ep()
    lv = ep.q4_levels(kind)
    np.testing.assert_array_equal(lv.view(np.uint32), oracle.q4_levels(kind).astype(np.float32).view(np.uint32))


@pytest.mark.parametrize("kind", ["nf4", "int4"])
@pytest.mark.parametrize("shape,block", [((64, 1024), 64), ((45, 200), 16), ((3, 136), 128), ((1, 8), 16),
                                         ((33, 1000), 1024)])
def test_q4_encoder_byte_identical(kind, shape, block):
    ep = _ep()
    w = synth.rows_outliers_bf16(shape[0] + block, *shape)
    w[0, :4] = 0
    q = ep.q4_encode(w, kind, block)
    codes, scales, _, bits = oracle.q4_roundtrip(w, kind, block)
    flat = codes.reshape(-1)
    np.testing.assert_array_equal(q.codes, (flat[0::2] | (flat[1::2] << 4)).astype(np.uint8))
    np.testing.assert_array_equal(q.scales.view(np.uint32), scales.view(np.uint32))
    assert q.bits_per_weight == pytest.approx(bits, abs=32.0 / w.size)
    for t in (1, 3):
        q2 = ep.q4_encode(w, kind, block, n_threads=t)
        assert (q2.codes == q.codes).all() and (q2.scales == q.scales).all()


def test_q4_errors():
    ep = _ep()
    from dit_weight_compression_02_b300._lib import lib
    w = synth.normal_bf16(40, 4, 64)
    with pytest.raises(ep.EntroPackError) as e:
        ep.q4_encode(w, "nf4", block=24)
    assert e.value.status == "EP_ERR_INVALID_ARG"
    bad = w.copy()
    bad[1, 5] = 0x7FC0  # NaN
    with pytest.raises(ep.EntroPackError) as e:
        ep.q4_encode(bad)
    assert e.value.status == "EP_ERR_NONFINITE"
    with pytest.raises(ep.EntroPackError) as e:
        ep.q4_encode(w.reshape(-1)[:7].copy())
    assert e.value.status == "EP_ERR_SHAPE"
    lv = np.zeros(16, np.float32)
    assert lib.ep_q4_levels(2, lv.ctypes.data) == 1
    # device entry point: argument errors return before any CUDA call
    fake = ctypes.c_void_p(1 << 20)
    assert lib.ep_q4_decode(fake, fake, 64, 64, lv.ctypes.data, ctypes.c_void_p((1 << 20) + 8), None) == 1
    assert lib.ep_q4_decode(ctypes.c_void_p((1 << 20) + 4), fake, 64, 64, lv.ctypes.data, fake, None) == 1
    assert lib.ep_q4_decode(fake, fake, 63, 64, lv.ctypes.data, fake, None) == 2
    assert lib.ep_q4_decode(fake, fake, 64, 8, lv.ctypes.data, fake, None) == 1
    assert lib.ep_q4_decode(fake, fake, 64, 64, None, fake, None) == 1


# ------------------------------------------------ per-layer bit allocation
def _alloc_layers():
    return [synth.student_t5_bf16(51, 64, 256), synth.normal_bf16(52, 45, 200),
            synth.rows_outliers_bf16(53, 32, 1024, frac=0.01, k_sigma=12.0)]


@pytest.mark.parametrize("sens", [None, [4.0, 1.0, 0.25], [2.0, 3.0, 0.7]])
@pytest.mark.parametrize("avg", [2.5, 4.0, 20.0, 0.01])
def test_allocation_identical_to_oracle(sens, avg):
    ep = _ep()
    layers = _alloc_layers()
    r_lib = ep.allocate_bits(layers, avg, sens)
    r_orc = oracle.allocate_bits(layers, avg, sens)
    assert r_lib["t"] == r_orc["t"] and r_lib["j"] == r_orc["j"]
    assert r_lib["est_bpp"] == r_orc["est_bpp"]  # bit-identical estimates


def test_estimate_and_encode_at_identical_to_oracle():
    ep = _ep()
    for w in _alloc_layers():
        jmin = oracle.smallest_valid_j(w)
        for j in (jmin, jmin + 37, 0, 128):
            bpp, jm = ep.estimate_bpp(w, j)
            assert jm == jmin and bpp == oracle.estimate_bpp(w, 0.05, j)
            assert ep.encode(w, 3.25, j=j) == oracle.encode_at(w, j, 3.25)
        for c in ("fp8", "int8"):
            assert ep.encode(w, 3.0, c, j=jmin + 64) == oracle.encode_at(w, jmin + 64, 3.0, c)


def test_allocation_errors():
    ep = _ep()
    layers = _alloc_layers()
    for sens in ([1.0, 0.0, 1.0], [1.0, -2.0, 1.0], [1.0, float("inf"), 1.0]):
        with pytest.raises(ep.EntroPackError) as e:
            ep.allocate_bits(layers, 4.0, sens)
        assert e.value.status == "EP_ERR_INVALID_ARG"
    with pytest.raises(ep.EntroPackError) as e:
        ep.allocate_bits(layers, 0.0)
    assert e.value.status == "EP_ERR_INVALID_ARG"
    bad = layers[0].copy()
    bad[2, 2] = 0x7F80
    with pytest.raises(ep.EntroPackError) as e:
        ep.allocate_bits([bad, layers[1]], 4.0)
    assert e.value.status == "EP_ERR_NONFINITE"
    with pytest.raises(ep.EntroPackError) as e:
        ep.allocate_bits([layers[0][:, :100].copy()], 4.0)
    assert e.value.status == "EP_ERR_SHAPE"
    jmin = oracle.smallest_valid_j(layers[0])
    for j in (jmin - 1, 129, -641):
        with pytest.raises(ep.EntroPackError) as e:
            ep.encode(layers[0], 4.0, j=j)
        assert e.value.status == "EP_ERR_INVALID_ARG"


def _wide_range_bf16(seed, rows, cols):
    """Weights spread over 2^-30 .. 2^0 with random signs: every E4M3 binade and the subnormals."""
    rng = np.random.default_rng(seed)
    v = np.exp2(rng.uniform(-30.0, 0.0, size=(rows, cols))) * rng.choice([-1.0, 1.0], size=(rows, cols))
    return torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("shape", [(48, 256), (5, 8), (100, 1000), (33, 136)])
def test_fp8_row_encoder_byte_identical(shape):
    ep = _ep()
    for w in (synth.rows_outliers_bf16(shape[0] + 7, *shape), _wide_range_bf16(shape[0], *shape)):
        w[0] = 0
        w[-1, :2] = 0x8000  # -0
        codes, scales = ep.fp8_row_encode(w)
        _, _, c_o, s_o = oracle.fp8_row_roundtrip(w, with_codes=True)
        np.testing.assert_array_equal(codes, c_o)
        np.testing.assert_array_equal(scales.view(np.uint32), s_o.view(np.uint32))


def test_fp8_row_errors():
    ep = _ep()
    from dit_weight_compression_02_b300._lib import lib
    w = synth.normal_bf16(41, 4, 64)
    bad = w.copy()
    bad[2, 7] = 0xFF80  # -inf
    with pytest.raises(ep.EntroPackError) as e:
        ep.fp8_row_encode(bad)
    assert e.value.status == "EP_ERR_NONFINITE"
    with pytest.raises(ep.EntroPackError) as e:
        ep.fp8_row_encode(w[:, :60].copy())
    assert e.value.status == "EP_ERR_SHAPE"
    fake = ctypes.c_void_p(1 << 20)
    assert lib.ep_fp8_row_decode(fake, fake, 4, 64, ctypes.c_void_p((1 << 20) + 8), None) == 1
    assert lib.ep_fp8_row_decode(ctypes.c_void_p((1 << 20) + 8), fake, 4, 64, fake, None) == 1
    assert lib.ep_fp8_row_decode(fake, fake, 4, 60, fake, None) == 2
    assert lib.ep_fp8_row_decode(None, fake, 4, 64, fake, None) == 1


def test_allocation_thread_count_does_not_change_the_plan():
    ep = _ep()
    layers = _alloc_layers()
    ref = ep.allocate_bits(layers, 3.0, [1.0, 2.0, 0.5], n_threads=1)
    for t in (2, 5):
        assert ep.allocate_bits(layers, 3.0, [1.0, 2.0, 0.5], n_threads=t) == ref


def test_stream_handles_validate_once():
    """ep_stream_open parses and validates like ep_query; the handle entry points check their arguments."""
    ep = _ep()
    from dit_weight_compression_02_b300._lib import lib
    blob = ep.encode(synth.normal_bf16(42, 64, 256), 4.0)
    host = np.frombuffer(blob, dtype=np.uint8)
    h = ctypes.c_void_p(0)
    assert lib.ep_stream_open(host.ctypes.data, len(blob), ctypes.byref(h)) == 0 and h.value
    fake = ctypes.c_void_p(1 << 20)
    status = ctypes.c_void_p(1 << 21)
    assert lib.ep_decode_h(h, ctypes.c_void_p((1 << 20) + 8), fake, None, status, None) == 1  # misaligned
    assert lib.ep_decode_h(None, fake, fake, None, status, None) == 1
    assert lib.ep_decode_h(h, fake, fake, None, None, None) == 1
    assert lib.ep_compressed_linear_h(None, fake, fake, 16, fake, None, 0, fake, 1 << 30, status, None) == 1
    assert lib.ep_compressed_linear_h(h, fake, fake, 16, fake, None, 1, fake, 1 << 30, status, None) == 5  # fused
    assert lib.ep_compressed_linear_h(h, fake, fake, 16, fake, None, 0, fake, 10, status, None) == 1  # workspace
    lib.ep_stream_close(h)
    lib.ep_stream_close(None)
    bad = np.frombuffer(_flip(blob, 0), dtype=np.uint8)
    h2 = ctypes.c_void_p(0)
    assert lib.ep_stream_open(bad.ctypes.data, len(blob), ctypes.byref(h2)) == 4 and not h2.value
    assert lib.ep_stream_open(host.ctypes.data, len(blob) - 16, ctypes.byref(h2)) == 4
    assert lib.ep_stream_open(None, len(blob), ctypes.byref(h2)) == 1


def test_allocation_identical_to_oracle_random_cases():
    """Seeded random sensitivities (FP32-exact) and budgets: library and oracle give the same plan."""
    ep = _ep()
    rng = np.random.default_rng(2024)
    layers = _alloc_layers()
    for _ in range(8):
        sens = [float(np.float32(v)) for v in np.exp2(rng.uniform(-3.0, 3.0, size=3))]
        avg = float(np.float32(rng.uniform(1.0, 7.0)))
        r_lib = ep.allocate_bits(layers, avg, sens)
        r_orc = oracle.allocate_bits(layers, avg, sens)
        assert (r_lib["t"], r_lib["j"]) == (r_orc["t"], r_orc["j"]), (sens, avg)
