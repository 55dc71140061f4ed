"""Pins of the oracle's rANS coder and 12-bit normaliser.

Independent of the oracle itself: hand-computed golden streams, hand-worked
normaliser tables, and the information-theoretic code-length bounds of rANS
with a 32-bit state (each step changes log2(state) by log2(4096/f) +- log2(1+1/16)).
"""
import math
import os

import numpy as np
import pytest

import oracle
import synth


def _parse_pairs(s):
    out = {}
    for item in s.split(","):
        k, v = item.split(":")
        out[int(k)] = int(v)
    return out


def test_golden_streams(golden_dir):
    n = 0
    for line in open(os.path.join(golden_dir, "rans_tiny.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        fs, syms, state, words = [p.strip() for p in line.split("|")]
        F = np.zeros((1, 256), dtype=np.uint32)
        if fs == "uniform":
            F[0, :] = 16
        else:
            for k, v in _parse_pairs(fs).items():
                F[0, k] = v
        s = np.array([int(v) for v in syms.split()], dtype=np.uint8)
        ctx = np.zeros(s.size, dtype=np.uint8)
        st, w = oracle.rans_encode(s, ctx, F)
        assert st == int(state), line
        assert list(w) == [int(v) for v in words.split()], line
        assert (oracle.rans_decode(w, st, ctx, F) == s).all()
        n += 1
    assert n == 3


def test_golden_normalizer(golden_dir):
    n = 0
    for line in open(os.path.join(golden_dir, "normalizer.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        cs, fs = [p.strip() for p in line.split("|")]
        counts = np.zeros(256, dtype=np.uint64)
        for k, v in _parse_pairs(cs).items():
            counts[k] = v
        want = np.zeros(256, dtype=np.uint32)
        for k, v in _parse_pairs(fs).items():
            want[k] = v
        got = oracle.normalize(counts)
        assert (got == want).all(), (line, {i: int(got[i]) for i in np.nonzero(got)[0]})
        n += 1
    assert n >= 6


@pytest.mark.parametrize("seed", range(6))
def test_normalizer_invariants(seed):
    r = np.array([synth.u64(seed, 30, i) for i in range(256)], dtype=np.uint64)
    counts = np.where(r % 3 == 0, 0, r % (10 ** (1 + seed))).astype(np.uint64)
    counts[seed] += 1
    f = oracle.normalize(counts)
    assert int(f.sum()) == 4096
    assert ((f > 0) >= (counts > 0)).all()
    assert (f <= 4095).all()
    assert (oracle.normalize(counts) == f).all()


def _random_stream(seed, n, alphabet):
    p = np.array([1.0 / (1 + i) ** 1.5 for i in range(alphabet)])
    counts = np.floor(p / p.sum() * 1e6).astype(np.uint64) + 1
    F = oracle.normalize(np.pad(counts, (0, 256 - alphabet)))
    cum = np.concatenate([[0], np.cumsum(F)])
    u = np.array([synth.u64(seed, 31, i) % 4096 for i in range(n)])
    syms = (np.searchsorted(cum, u, side="right") - 1).astype(np.uint8)
    return syms, F


@pytest.mark.parametrize("seed,n,alphabet", [(1, 5000, 2), (2, 20000, 40), (3, 3000, 256), (4, 1, 5)])
def test_roundtrip_and_code_length(seed, n, alphabet):
    syms, F = _random_stream(seed, n, alphabet)
    ctx = np.zeros(n, dtype=np.uint8)
    st, w = oracle.rans_encode(syms, ctx, F[None])
    assert (1 << 16) <= st < (1 << 32)
    assert (oracle.rans_decode(w, st, ctx, F[None]) == syms).all()
    ideal = float(sum(math.log2(4096.0 / F[s]) for s in syms))
    content = 16 * len(w) + math.log2(st) - 16
    slack = n * math.log2(1 + 1 / 16)
    assert ideal - slack <= content <= ideal + slack
    if n >= 3000:  # typical states are far above 16 f, so the loss is tiny
        assert abs(content - ideal) <= 0.002 * ideal + 2


def test_extreme_frequencies_and_contexts():
    # f = 1 and f = 4095 symbols, two contexts interleaved
    F = np.zeros((2, 256), dtype=np.uint32)
    F[0, 0], F[0, 1] = 1, 4095
    F[1, 10], F[1, 11], F[1, 12] = 4094, 1, 1
    syms = np.array([0, 10, 1, 11, 0, 12, 0, 10] * 50, dtype=np.uint8)
    ctx = np.array([0, 1] * 200, dtype=np.uint8)
    st, w = oracle.rans_encode(syms, ctx, F)
    assert (oracle.rans_decode(w, st, ctx, F) == syms).all()


def test_corrupt_stream_detected():
    syms, F = _random_stream(9, 4000, 30)
    ctx = np.zeros(syms.size, dtype=np.uint8)
    st, w = oracle.rans_encode(syms, ctx, F[None])
    with pytest.raises(oracle.OracleError):
        oracle.rans_decode(w[:-1], st, ctx, F[None])
    bad = w.copy()
    bad[len(bad) // 2] ^= 0x1234
    try:
        out = oracle.rans_decode(bad, st, ctx, F[None])
        assert not (out == syms).all()
    except oracle.OracleError:
        pass
