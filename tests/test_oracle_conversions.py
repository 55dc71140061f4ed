"""Pins of the oracle's container conversions.

The oracle rounds from the format definitions (nearest multiple of the
quantum of the binade, ties to even); these tests check it against torch's
and numpy's own conversions on random and adversarial fp32 inputs.
"""
import numpy as np
import pytest
import torch

import oracle
import synth


def _patterns(seed, n):
    bits = np.array([synth.u64(seed, 40, i) & 0xFFFFFFFF for i in range(n)], dtype=np.uint32)
    return bits.view(np.float32)


def _halfway_cases(mbits):
    # values exactly halfway between two representable neighbours, both parities
    out = []
    for e in (-130, -127, -20, -1, 0, 1, 7, 15, 100):
        for m in (0, 1, 2, 3, (1 << mbits) - 1, (1 << mbits) - 2):
            base = (1 + m / (1 << mbits)) * 2.0 ** e
            out += [base + 2.0 ** (e - mbits - 1), -(base + 2.0 ** (e - mbits - 1))]
    return np.array(out, dtype=np.float64).astype(np.float32)


def _finite(v):
    return v[np.isfinite(v)]


def test_bf16_against_torch():
    v = np.concatenate([_patterns(1, 60000), _halfway_cases(7),
                        np.array([0.0, -0.0, 1e-45, -1e-45, 3.4e38, -3.4e38, np.inf, -np.inf], np.float32)])
    got = oracle.convert_f32(v, "bf16")
    want = torch.from_numpy(v.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(v)
    assert (got[~nan] == want[~nan]).all()
    assert (((got[nan] & 0x7F80) == 0x7F80) & ((got[nan] & 0x7F) != 0)).all()


def test_fp16_against_numpy_and_torch():
    v = np.concatenate([_finite(_patterns(2, 60000)), _halfway_cases(10),
                        np.array([65504, 65519.99, 65520, -65520, 6e-8, 2.98e-8, 2.99e-8], np.float32)])
    got = oracle.convert_f32(v, "fp16")
    with np.errstate(over="ignore"):
        want_np = v.astype(np.float16).view(np.uint16)
    want_t = torch.from_numpy(v.copy()).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert (got == want_np).all()
    assert (got == want_t).all()


def test_e4m3_against_torch_in_range():
    v = _finite(_patterns(3, 60000))
    v = v[np.abs(v) <= 448.0]
    extra = np.array([448, -448, 0.001953125, 0.0009765625, 0.0014648438, 240, 232, 248, 17, 17.5, 18.5, 0, -0.0],
                     np.float32)
    sweep = (np.arange(-4600, 4601, dtype=np.float32) / 10.0)
    v = np.concatenate([v, extra, sweep])
    got = oracle.convert_f32(v, "fp8")
    want = torch.from_numpy(v.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (got == want).all()


def test_e4m3_satfinite_beyond_range():
    v = np.array([448.0, 449, 463.9, 464, 480, 1e6, 3e38, np.inf], np.float32)
    got = oracle.convert_f32(np.concatenate([v, -v]), "fp8")
    assert (got[:8] == 0x7E).all() and (got[8:] == 0xFE).all()


def test_int8_round_half_even_and_clamp():
    v = np.array([0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5, 127.49, 127.5, 300, -126.5, -127.6, -1000, 3.3, -3.7],
                 np.float32)
    want = np.array([0, 2, 2, 0, -2, -2, 126, 127, 127, 127, -126, -127, -127, 3, -4], np.int8)
    assert (oracle.convert_f32(v, "int8") == want).all()
    r = _finite(_patterns(4, 20000))
    r = r[np.abs(r) < 1e4]
    assert (oracle.convert_f32(r, "int8") == np.clip(np.rint(r.astype(np.float64)), -127, 127).astype(np.int8)).all()
