"""Pins of the oracle's lossless tiled-ANS path.

Recovery must be bitwise ("EntroPack PyTorch Guide", "Start with a tensor
round trip": numeric closeness is not bitwise equality; include zeros,
repeated values and edge cases).  Exhaustive over all 65536 BF16 patterns.
"""
import numpy as np

import oracle
import synth


def test_all_bf16_patterns_bitwise():
    w = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(512, 128)
    blob = oracle.encode_lossless(w)
    y, rs = oracle.decode(blob)
    assert rs is None
    assert (y == w).all()


def test_special_rows_bitwise():
    w = synth.with_special_rows(synth.normal_bf16(4, 256, 512), seed=4)
    blob = oracle.encode_lossless(w)
    y, _ = oracle.decode(blob)
    assert (y == w).all()
    sym = oracle.decode_symbols(blob)
    assert (sym == ((w >> 7) & 0xFF)).all()


def test_single_exponent_tensor():
    w = np.full((32, 128), 0x3F80, dtype=np.uint16)  # all 1.0: one exponent symbol
    blob = oracle.encode_lossless(w)
    assert (oracle.decode(blob)[0] == w).all()


def test_lossless_rate():
    w = synth.normal_bf16(4, 256, 1024)
    blob = oracle.encode_lossless(w)
    e = ((w >> 7) & 0xFF).ravel()
    cnt = np.bincount(e, minlength=256).astype(np.float64)
    nz = cnt[cnt > 0]
    h = float((nz * np.log2(e.size / nz)).sum()) / e.size
    bpp = 8 * len(blob) / w.size
    assert 8 + h <= bpp <= 8 + h + 0.15


# ------------------------------------------------ other element types
def test_all_fp16_patterns_bitwise():
    w = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(512, 128)
    y, _ = oracle.decode(oracle.encode_lossless(w, "fp16"))
    assert y.dtype == np.uint16 and (y == w).all()


def test_all_fp8_patterns_bitwise():
    w = np.tile(np.arange(256, dtype=np.uint16).astype(np.uint8), 64).reshape(128, 128)
    blob = oracle.encode_lossless(w, "fp8")
    y, _ = oracle.decode(blob)
    assert y.dtype == np.uint8 and (y == w).all()
    # FP8 codes the whole byte: the coded symbol of every element is the element
    assert (oracle.decode_symbols(blob) == w).all()


def test_fp32_specials_and_random_bitwise():
    rng = np.random.default_rng(7)
    w = rng.integers(0, 2**32, size=(96, 384), dtype=np.uint64).astype(np.uint32)
    specials = np.array([0x00000000, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00001, 0xFFBFFFFF, 0x00000001,
                         0x807FFFFF, 0x3F800000, 0xBF800000, 0x7F7FFFFF, 0x00800000], dtype=np.uint32)
    w[5, :specials.size] = specials
    w[7] = 0x3F800000  # a repeated value
    blob = oracle.encode_lossless(w, "fp32")
    y, _ = oracle.decode(blob)
    assert y.dtype == np.uint32 and (y == w).all()
    # the coded symbol is the exponent field, bits 30..23
    assert (oracle.decode_symbols(blob) == ((w >> 23) & 0xFF)).all()


def test_fp16_and_fp32_rates_track_exponent_entropy():
    # the coded byte of FP32 is the exponent: bits/element = 24 raw + its entropy
    f = synth.bf16_to_f32(synth.normal_bf16(9, 256, 1024)).astype(np.float32)
    w = f.view(np.uint32)
    e = ((w >> 23) & 0xFF).ravel()
    cnt = np.bincount(e, minlength=256).astype(np.float64)
    nz = cnt[cnt > 0]
    h = float((nz * np.log2(e.size / nz)).sum()) / e.size
    bpp = 8 * len(oracle.encode_lossless(w, "fp32")) / w.size
    assert 24 + h <= bpp <= 24 + h + 0.15
