"""Pins of the oracle's per-layer bitrate allocation and fixed-resolution encode.

The allocation gives layers with more weight on their error more bits under
one model-level budget ("EntroPack PyTorch Guide", "Separate reconstruction
metrics from application metrics"), driven by the sampled storage estimates
(EntroPack paper, Abstract).  Pins:
* exhaustive scan of the shared index on tiny layers: the result fits the
  budget and the next finer index does not (the bisection invariant), and
  equals the finest fitting index where the total is monotone;
* high-resolution rate-distortion theory: a sensitivity of 4 lowers the
  layer's index by 64 (Delta halved), which halves its relative L2 error and
  costs about one bit per parameter, measured by encoding and decoding;
* Jensen: at unit sensitivities the allocation's summed squared relative
  error is below that of giving every layer the average target, at no more
  storage;
* the fixed-resolution encode equals the rate-searched one at the index the
  search picks, and refuses indices that overflow a row.
"""
import math

import numpy as np
import pytest

import oracle
import synth


def _layers():
    return [synth.student_t5_bf16(41, 64, 256), synth.normal_bf16(42, 96, 512),
            synth.rows_outliers_bf16(43, 32, 1024, frac=0.01, k_sigma=12.0)]


def _rel(w, blob):
    y = oracle.container_to_f64(oracle.decode(blob)[0], "bf16")
    return oracle.rel_l2(y, synth.bf16_to_f32(w))


@pytest.mark.parametrize("sens", [None, [4.0, 1.0, 0.25], [2.0, 3.0, 0.7]])
@pytest.mark.parametrize("avg", [2.5, 4.0])
def test_shared_index_by_exhaustive_scan(sens, avg):
    layers = _layers()
    r = oracle.allocate_bits(layers, avg, sens)
    alphas = [1.0] * 3 if sens is None else sens
    off = [int(math.copysign(math.floor(abs(32 * math.log2(a)) + 0.5), math.log2(a))) for a in alphas]
    jmin = [oracle.smallest_valid_j(w) for w in layers]
    n = [w.size for w in layers]
    budget = float(np.float32(avg)) * sum(n)

    def total(t):
        return sum(n[l] * oracle.estimate_bpp(layers[l], 0.05, min(max(t - off[l], jmin[l]), 128)) for l in range(3))

    ts = list(range(min(jmin[l] + off[l] for l in range(3)), max(128 + off[l] for l in range(3)) + 1))
    fits = [t for t in ts if total(t) <= budget]
    assert fits, "budget reachable in these cases"
    t = r["t"]
    assert total(t) <= budget and (t == ts[0] or total(t - 1) > budget)
    totals = [total(x) for x in ts]
    if all(a >= b for a, b in zip(totals, totals[1:])):
        assert t == fits[0]
    assert r["j"] == [min(max(t - off[l], jmin[l]), 128) for l in range(3)]
    assert r["est_bits"] <= r["budget_bits"]


def test_sensitivity_four_halves_the_error_for_one_bit():
    w = synth.normal_bf16(44, 256, 1024)
    r = oracle.allocate_bits([w, w.copy()], 4.0, [4.0, 1.0])
    j_hi, j_lo = r["j"]
    assert j_lo - j_hi == 64  # Delta_hi = Delta_lo / 2
    b_hi, b_lo = oracle.encode_at(w, j_hi), oracle.encode_at(w, j_lo)
    ratio = _rel(w, b_hi) / _rel(w, b_lo)
    assert 0.47 < ratio < 0.53, ratio
    d_bits = r["est_bpp"][0] - r["est_bpp"][1]
    assert 0.9 < d_bits < 1.1, d_bits
    assert r["est_bpp"][0] + r["est_bpp"][1] <= 8.0  # the average stays within the budget


def test_allocation_beats_uniform_targets():
    layers = _layers()
    avg = 3.5
    r = oracle.allocate_bits(layers, avg)
    alloc = [oracle.encode_at(w, j) for w, j in zip(layers, r["j"])]
    uniform = [oracle.encode(w, avg) for w in layers]
    n = [w.size for w in layers]

    def objective(blobs):
        return sum(nl * _rel(w, b) ** 2 for nl, w, b in zip(n, layers, blobs))

    def coded_bits(blobs):
        return sum(8 * len(b) for b in blobs)

    assert objective(alloc) < 0.97 * objective(uniform)
    assert coded_bits(alloc) <= 1.01 * coded_bits(uniform)
    # equal sensitivities and no clamping: one shared index
    assert len(set(r["j"])) == 1


def test_encode_at_matches_rate_search_and_refuses_overflow():
    w = synth.student_t5_bf16(45, 64, 512)
    j, j_lo = oracle.select_j(w, 3.0)
    assert oracle.encode_at(w, j, 3.0) == oracle.encode(w, 3.0)
    assert oracle.smallest_valid_j(w) == j_lo
    with pytest.raises(oracle.OracleError):
        oracle.encode_at(w, j_lo - 1)
    with pytest.raises(oracle.OracleError):
        oracle.encode_at(w, 129)
