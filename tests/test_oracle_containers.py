"""Exact pin of the oracle's container step for lossy streams.

The container rule ("EntroPack: Fast and Accurate Entropy-Coded Weight
Compression at Arbitrary Bitrates", Abstract: floating-point and integer
weight containers BF16, FP16, FP8 and INT8, the storage bitrate independent
of the container) is read as: each container value is one fp32 product
rounded to the container.  BF16 / FP16 take y = container(fp32(g_r * q));
FP8 e4m3 and INT8 take a per-row multiplier m_r, y = container(fp32(q * m_r)),
with output scale t_r = fp32(g_r / m_r) so that w ~ t_r * y:

  FP8   m_r = TR7(448 / Q_r)                                  (1 if Q_r = 0)
  INT8  m_r = 2 if 2 Q_r <= 127, else TR7(127 / Q_r)          (1 if Q_r = 0)

where Q_r = max_k |q_rk| and TR7 truncates to 7 significant bits.

This test recomputes all of it from the decoded lattice points alone
(oracle.decode_lattice gives k = 2q for every coordinate) and the row steps
g_r stored in the stream: TR7 in exact rational arithmetic (fractions), the
products, divisions and casts with torch's own fp32 arithmetic and its
bfloat16 / float16 / float8_e4m3fn conversions.  Every container value, m_r
and t_r must equal what oracle.decode returns and what the stream stores,
bit for bit.  Independent bounds pin the truncation direction: FP8 and INT8
never need saturation (|q * m_r| stays within 448 and 127) while each row's
maximum lands within one part in 64 of the limit, so rounding m_r to nearest
instead of truncating, or a wrong INT8 branch, fails here.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth


def _tr7(v: Fraction) -> Fraction:
    """Largest n * 2^e <= v with an integer 64 <= n < 128 (v > 0), exactly."""
    e = v.numerator.bit_length() - v.denominator.bit_length() - 7
    while v / Fraction(2) ** e >= 128:
        e += 1
    while v / Fraction(2) ** e < 64:
        e -= 1
    n = (v / Fraction(2) ** e).numerator // (v / Fraction(2) ** e).denominator
    assert 64 <= n < 128
    return n * Fraction(2) ** e


def _row_meta(blob: bytes, n: int):
    h = oracle.header(blob)
    mp = 32 * ((h["M"] + 31) // 32)
    off = h["rowmeta_off"]
    meta = np.frombuffer(blob, dtype=np.float32, count=n * mp, offset=off).reshape(n, mp)
    return h, mp, meta


def _f32(a) -> torch.Tensor:
    return torch.from_numpy(np.array(a, dtype=np.float32))


def _expected(blob: bytes, container: str):
    """Container values, m_r and t_r recomputed from the lattice points and g_r."""
    k = oracle.decode_lattice(blob)  # 2q, int32, M x K
    n_meta = 3 if container in ("fp8", "int8") else 1
    h, mp, meta = _row_meta(blob, n_meta)
    M = h["M"]
    g = meta[0]
    q = _f32(k.astype(np.float64) / 2.0)  # exact: |k| <= 30002
    if container in ("bf16", "fp16"):
        prod = q * _f32(g[:M])[:, None]  # one fp32 product, rounded to nearest even
        dt = torch.bfloat16 if container == "bf16" else torch.float16
        return prod.to(dt).view(torch.int16).numpy().view(np.uint16), None, None, prod
    Q = np.abs(k).max(axis=1) / 2.0 if k.shape[1] else np.zeros(M)
    m = np.ones(mp, dtype=np.float32)
    for r in range(M):
        if Q[r] == 0:
            continue
        if container == "int8" and 2 * Q[r] <= 127:
            m[r] = 2.0
        else:
            lim = 448 if container == "fp8" else 127
            mr = _tr7(Fraction(lim) / Fraction(Q[r]))
            assert float(np.float32(mr)) == mr  # 7 significant bits: exact in fp32
            m[r] = np.float32(mr)
    t = (_f32(g) / _f32(m)).numpy()  # one fp32 division, rounded to nearest even
    prod = q * _f32(m[:M])[:, None]
    if container == "fp8":
        y = prod.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    else:
        y = torch.clamp(torch.round(prod), -127, 127).to(torch.int8).numpy()
    return y, m, t, prod


def _blobs():
    zero_row = synth.normal_bf16(21, 64, 256)
    zero_row[5] = 0
    heavy = synth.rows_outliers_bf16(9, 256, 1024, frac=0.05, k_sigma=40.0)
    heavy[17] = 0  # an all-zero row among escape-heavy ones
    return [
        ("gauss_2.5bpp", zero_row, 2.5),              # small lattice points: the INT8 m = 2 branch
        ("escape_heavy_6bpp", heavy, 6.0),            # escapes on every row: the TR7 branch
        ("ragged_45x200_4bpp", synth.student_t5_bf16(22, 45, 200), 4.0),  # padded rows and columns
    ]


@pytest.mark.parametrize("container", ["bf16", "fp16", "fp8", "int8"])
def test_container_step_bit_exact(container):
    branches = set()
    for name, w, bpp in _blobs():
        blob = oracle.encode(w, bpp, container)
        y_exp, m_exp, t_exp, prod = _expected(blob, container)
        y, rs = oracle.decode(blob)
        if container in ("bf16", "fp16"):
            assert rs is None
            assert (y == y_exp).all(), name
            continue
        h, mp, meta = _row_meta(blob, 3)
        M = h["M"]
        # the stream's multipliers and scales, and the oracle's row scales
        assert (meta[1].view(np.uint32) == m_exp.view(np.uint32)).all(), name
        assert (meta[2].view(np.uint32) == t_exp.view(np.uint32)).all(), name
        assert (rs.view(np.uint32) == t_exp[:M].view(np.uint32)).all(), name
        assert (y.view(np.uint8) == y_exp.view(np.uint8)).all(), name
        # padding rows keep m = 1 and t = 0
        assert (meta[1][M:] == 1.0).all() and (meta[2][M:] == 0.0).all()
        # no saturation is ever needed, and each row's largest |q| lands just
        # below the limit (TR7 loses less than one part in 64)
        lim = 448.0 if container == "fp8" else 127.0
        p = prod.abs().numpy().astype(np.float64)
        assert p.max() <= lim, name
        k = oracle.decode_lattice(blob)
        for r in range(M):
            Q = np.abs(k[r]).max() / 2.0
            if Q == 0:
                assert meta[1][r] == 1.0 and (y[r] == 0).all()
                branches.add("zero")
            elif container == "int8" and 2 * Q <= 127:
                assert meta[1][r] == 2.0 and p[r].max() == 2 * Q
                branches.add("m2")
            else:
                assert lim * (1 - 2.0 ** -6) < p[r].max() <= lim, (name, r)
                branches.add("tr7")
    if container == "fp8":
        assert branches == {"zero", "tr7"}
    elif container == "int8":
        assert branches == {"zero", "m2", "tr7"}


def test_tr7_reference_values():
    # hand-checked: 448/3 = 149.33 -> 148 = 74 * 2 (74 = 1001010b, 7 bits); 127/100 = 1.27 ->
    # 1.265625 (81/64); 448/0.5 = 896 exactly (7 bits); 127/63.5 = 2 exactly
    assert _tr7(Fraction(448, 3)) == 148
    assert _tr7(Fraction(127, 100)) == Fraction(81, 64)
    assert _tr7(Fraction(896)) == 896
    assert _tr7(Fraction(127) / Fraction(127, 2)) == 2
    assert oracle.tr7(448 / 3) == 148.0 and oracle.tr7(1.27) == 81 / 64
