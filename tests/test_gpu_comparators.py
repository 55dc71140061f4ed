"""GPU parity of the fixed-width 4-bit comparators (ep_q4_decode) with the oracle.

The kernel reconstructs BF16(level * scale) from packed codes; the oracle's
reconstruction of the same weights is the reference, bit for bit.  Sizes span
many groups of 16 with ragged tails (n % 16 != 0), short last blocks and
several block sizes; one case is a full FFN-sized layer (10240 x 3840).
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


def _run(ep, w, kind, block):
    q = ep.q4_encode(w, kind, block)
    codes = torch.from_numpy(q.codes).cuda()
    scales = torch.from_numpy(q.scales).cuda()
    y = ep.q4_decode(codes, scales, q.levels, w.shape, block)
    torch.cuda.synchronize()
    return y.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("kind", ["nf4", "int4"])
@pytest.mark.parametrize("shape,block", [((64, 1024), 64), ((45, 200), 16), ((3, 136), 128), ((1, 8), 16),
                                         ((33, 1000), 1024), ((257, 3840), 64)])
def test_q4_decode_bit_exact(ep, kind, shape, block):
    w = synth.rows_outliers_bf16(shape[0] * 7 + block, *shape)
    w[0, :4] = 0
    y = _run(ep, w, kind, block)
    _, _, recon, _ = oracle.q4_roundtrip(w, kind, block)
    np.testing.assert_array_equal(y, recon)


def test_q4_decode_ffn_layer(ep):
    w = synth.student_t5_bf16(5, 10240, 3840)
    y = _run(ep, w, "nf4", 64)
    _, _, recon, _ = oracle.q4_roundtrip(w, "nf4", 64)
    np.testing.assert_array_equal(y, recon)


def test_q4_decode_into_offset_views(ep):
    """Decoding into a 16-byte aligned slice of a larger buffer leaves the rest untouched."""
    w = synth.normal_bf16(6, 16, 512)
    q = ep.q4_encode(w, "nf4", 64)
    buf = torch.full((w.size + 64,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[8: 8 + w.size].view(w.shape)
    ep.q4_decode(torch.from_numpy(q.codes).cuda(), torch.from_numpy(q.scales).cuda(), q.levels, w.shape, 64, out=out)
    torch.cuda.synchronize()
    _, _, recon, _ = oracle.q4_roundtrip(w, "nf4", 64)
    assert (out.view(torch.int16).cpu().numpy().view(np.uint16) == recon).all()
    rest = torch.cat([buf[:8], buf[8 + w.size:]]).float()
    assert (rest == 7.0).all()


@pytest.mark.parametrize("shape", [(48, 256), (5, 8), (100, 1000), (1024, 3840)])
def test_fp8_row_decode_bit_exact(ep, shape):
    w = synth.rows_outliers_bf16(shape[0] + 11, *shape)
    w[0] = 0
    codes, scales = ep.fp8_row_encode(w)
    y = ep.fp8_row_decode(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda())
    torch.cuda.synchronize()
    recon, _ = oracle.fp8_row_roundtrip(w)
    np.testing.assert_array_equal(y.view(torch.int16).cpu().numpy().view(np.uint16), recon)


def test_fp8_row_decode_every_code(ep):
    """All 254 finite E4M3 bytes under a few scales, against the oracle's decoder."""
    b = np.array([v for v in range(256) if v not in (0x7F, 0xFF)] * 2, dtype=np.uint8)[:504].reshape(1, 504)
    codes = np.repeat(b, 3, axis=0)
    scales = np.array([1.0, 2.0 ** -20, 3.5], dtype=np.float32)
    y = ep.fp8_row_decode(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda())
    torch.cuda.synchronize()
    got = y.float().cpu().numpy().astype(np.float64)
    q = np.array([[oracle.e4m3_to_f64(v) for v in row] for row in codes])
    ref = torch.from_numpy((q.astype(np.float32) * scales[:, None]).astype(np.float32)).to(torch.bfloat16)
    np.testing.assert_array_equal(got, ref.float().numpy().astype(np.float64))
