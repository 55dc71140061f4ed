"""Pins of the oracle's lossless tiled-ANS path (FORMAT.md §5).

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
