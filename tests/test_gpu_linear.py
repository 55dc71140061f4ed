"""GPU checks of the tcgen05 linear kernels against the fp64 oracle GEMM.

ep_linear_bf16 (dense BF16 W) and ep_compressed_linear (W decoded from a
stream) compute Y = X W^T in fp32 and round Y to BF16 once.  The reference
is the oracle's plain fp64 triple loop over the same BF16 X and the oracle's
decode of W.  Bars:
  * the CompressedLinear bar of max |Y - Y_ref| / max |Y_ref| <= 2e-2;
  * elementwise |Y - Y_ref| <= 2^-8 |Y_ref| + 1e-6 * sum_k |x_k w_k|: one
    BF16 rounding (2^-9 relative) plus fp32 accumulation over K terms;
which a transposed operand, a wrong swizzle or a dropped K block all fail.
Shapes span several tiles with ragged tails in every dimension; the full
CompressedLinear size (8192 x 3840 by 10240 x 3840) is checked on sampled
token rows.
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


def _bf16_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()


def _check(y: torch.Tensor, x_bits: np.ndarray, w64: np.ndarray, rows=None, bias_bits=None):
    x64 = synth.bf16_to_f32(x_bits).astype(np.float64)
    if rows is not None:
        x64 = x64[rows]
    y_ref = oracle.gemm_f64(x64, w64)
    mag = oracle.gemm_f64(np.abs(x64), np.abs(w64))
    if bias_bits is not None:  # one more fp32 addend before the single rounding
        b64 = synth.bf16_to_f32(bias_bits).astype(np.float64)
        y_ref = y_ref + b64
        mag = mag + np.abs(b64)
    yg = y.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        yg = yg[rows]
    err = np.abs(yg - y_ref)
    assert err.max() / np.abs(y_ref).max() <= 2e-2
    bound = 2.0 ** -8 * np.abs(y_ref) + 1e-6 * mag + 1e-30
    bad = np.argwhere(err > bound)
    assert bad.size == 0, f"{len(bad)} elements out of bound, first {bad[:5]} err {err[tuple(bad[0])]}"


@pytest.mark.parametrize("T,N,K", [(128, 256, 64), (300, 544, 200), (257, 3840, 384), (1000, 512, 1024)])
def test_dense_gemm_ragged(ep, T, N, K):
    x = synth.normal_bf16(100 + T, T, K, std=1.0)
    w = synth.student_t5_bf16(200 + N, N, K)
    y = ep.linear_bf16(_bf16_dev(x), _bf16_dev(w))
    _check(y, x, synth.bf16_to_f32(w).astype(np.float64))


@pytest.mark.parametrize("T,N,K", [(300, 544, 200), (77, 1000, 1000)])
def test_bias_in_epilogue(ep, T, N, K):
    x = synth.normal_bf16(300 + T, T, K, std=1.0)
    w = synth.student_t5_bf16(400 + N, N, K)
    b = synth.normal_bf16(500 + N, 1, N, std=0.5)[0]
    bd = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).cuda()
    y = ep.linear_bf16(_bf16_dev(x), _bf16_dev(w), bias=bd)
    _check(y, x, synth.bf16_to_f32(w).astype(np.float64), bias_bits=b)
    blob = oracle.encode(w, 4.0)
    yc = ep.compressed_linear(ep.DeviceBlob(blob), _bf16_dev(x), bias=bd)
    _check(yc, x, oracle.container_to_f64(oracle.decode(blob)[0], "bf16"), bias_bits=b)
    # a zero bias changes no value (only -0 may become +0)
    y0 = ep.linear_bf16(_bf16_dev(x), _bf16_dev(w))
    y1 = ep.linear_bf16(_bf16_dev(x), _bf16_dev(w), bias=torch.zeros_like(bd))
    assert torch.equal(y0.float(), y1.float())


def test_dense_gemm_matches_torch_closely(ep):
    x = synth.normal_bf16(7, 512, 1024, std=1.0)
    w = synth.normal_bf16(8, 768, 1024)
    xd, wd = _bf16_dev(x), _bf16_dev(w)
    y = ep.linear_bf16(xd, wd).float()
    ref = (xd.float() @ wd.float().t())
    rel = ((y - ref).abs().max() / ref.abs().max()).item()
    assert rel < 4e-3


def test_compressed_linear_small(ep):
    w = synth.student_t5_bf16(61, 1024, 3840)
    x = synth.normal_bf16(62, 333, 3840, std=1.0)
    blob = oracle.encode(w, 4.0)
    db = ep.DeviceBlob(blob)
    y = ep.compressed_linear(db, _bf16_dev(x))
    w_hat = oracle.container_to_f64(oracle.decode(blob)[0], "bf16")
    _check(y, x, w_hat)


@pytest.mark.parametrize("T,N,K", [(77, 1000, 1000), (5, 48, 200), (300, 264, 136)])
def test_compressed_linear_general_shapes(ep, T, N, K):
    w = synth.student_t5_bf16(N + K, N, K)
    x = synth.normal_bf16(T + K, T, K, std=1.0)
    blob = oracle.encode(w, 4.0)
    y = ep.compressed_linear(ep.DeviceBlob(blob), _bf16_dev(x))
    assert y.shape == (T, N)
    _check(y, x, oracle.container_to_f64(oracle.decode(blob)[0], "bf16"))


def test_compressed_linear_full_size_sampled(ep):
    # X 8192 x 3840 N(0,1), W 10240 x 3840 Student-t at 4 bpp
    w = synth.student_t5_bf16(5, 10240, 3840)
    x = synth.normal_bf16(5, 8192, 3840, std=1.0)
    blob = ep.encode(w, 4.0)
    assert blob == oracle.encode(w, 4.0)
    db = ep.DeviceBlob(blob)
    y = ep.compressed_linear(db, _bf16_dev(x))
    w_hat = oracle.container_to_f64(oracle.decode_threaded(blob)[0], "bf16")
    # one token row in every 128-row M tile (at a different offset in each),
    # so every (M tile, N tile) output tile of the persistent GEMM schedule is
    # checked, plus the first and last rows
    rows = np.unique(np.r_[[t * 128 + (37 * t + 5) % 128 for t in range(8192 // 128)], 0, 8191])
    _check(y, x, w_hat, rows=rows)


@pytest.mark.parametrize("T,N,K,with_bias", [(128, 10240, 3840, False), (77, 1000, 1024, True),
                                              (300, 544, 384, False), (5, 48, 256, True), (700, 256, 1024, False)])
def test_fused_linear_matches_fp64(ep, T, N, K, with_bias):
    # W decoded straight into shared memory as the tensor-core operand.  The
    # shapes cover the CompressedLinear layer at 128 tokens (three tile rows
    # per CTA, one wave), ragged tile rows (N % 32 != 0), an odd number of
    # tiles per row (K = 384), several token tiles per pass (T = 300) and two
    # passes (T = 700 > 640 tokens per pass for K = 1024); the outlier rows
    # put escapes into every layer
    w = synth.rows_outliers_bf16(N + K, N, K, frac=0.002, k_sigma=40.0)
    x = synth.normal_bf16(T + 3 * K, T, K, std=1.0)
    blob = oracle.encode(w, 4.0)
    sym = oracle.decode_symbols(blob)
    assert (sym.reshape(N, -1, 8)[:, :, 1:] == 0).any()  # escaped coordinates exist
    b = synth.normal_bf16(N, 1, N, std=0.5)[0] if with_bias else None
    bd = None if b is None else torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).cuda()
    y = ep.compressed_linear(ep.DeviceBlob(blob), _bf16_dev(x), mode=ep.LINEAR_FUSED, bias=bd)
    assert y.shape == (T, N)
    _check(y, x, oracle.container_to_f64(oracle.decode(blob)[0], "bf16"), bias_bits=b)


@pytest.mark.parametrize("T,N,K", [(100, 15360, 128), (300, 15360, 256)])
def test_fused_linear_several_units_per_cta(ep, T, N, K):
    # more units (three tile rows each) than SMs: CTAs take a second unit, so
    # the accumulators are read back and reused, and the half-slab barriers
    # carry on across units
    w = synth.student_t5_bf16(N + 7 * K, N, K)
    x = synth.normal_bf16(T + 11 * K, T, K, std=1.0)
    blob = oracle.encode(w, 4.0)
    n_units = -(-(N // 32) // 3)
    assert n_units > torch.cuda.get_device_properties(0).multi_processor_count
    y = ep.compressed_linear(ep.DeviceBlob(blob), _bf16_dev(x), mode=ep.LINEAR_FUSED)
    _check(y, x, oracle.container_to_f64(oracle.decode(blob)[0], "bf16"))


def test_fused_linear_reports_corruption(ep):
    # payload words changed on the device after the host validated the stream:
    # the fused kernel's end-of-lane checks must flag it in the status word
    w = synth.normal_bf16(68, 256, 512)
    blob = oracle.encode(w, 4.0)
    db = ep.DeviceBlob(blob)
    h = oracle.header(blob)
    b = bytearray(blob)
    for off in range(h["payload_off"] + 200, h["payload_off"] + 2000, 97):
        b[off] ^= 0xFF
    db.device.copy_(torch.from_numpy(np.frombuffer(bytes(b), dtype=np.uint8).copy()).cuda())
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.compressed_linear(db, _bf16_dev(synth.normal_bf16(69, 64, 512, std=1.0)), mode=ep.LINEAR_FUSED, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 0x1
    db.device.copy_(db.host.cuda())  # the clean stream again: no flag
    ep.compressed_linear(db, _bf16_dev(synth.normal_bf16(69, 64, 512, std=1.0)), mode=ep.LINEAR_FUSED, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def test_fused_linear_unsupported_shapes(ep):
    assert ep.fused_tokens_per_pass(3840) == 640 and ep.fused_tokens_per_pass(200) == 0
    w = synth.normal_bf16(66, 64, 200)  # in_features not a multiple of 128
    db = ep.DeviceBlob(oracle.encode(w, 4.0))
    with pytest.raises(ep.EntroPackError) as e:
        ep.compressed_linear(db, _bf16_dev(synth.normal_bf16(67, 8, 200)), mode=ep.LINEAR_FUSED)
    assert e.value.status == "EP_ERR_UNSUPPORTED"


def test_compressed_linear_rejects_bad_args(ep):
    w = synth.normal_bf16(63, 64, 256)
    db = ep.DeviceBlob(oracle.encode(w, 4.0))
    x = _bf16_dev(synth.normal_bf16(64, 16, 256))
    with pytest.raises(ep.EntroPackError) as e:
        ep.compressed_linear(db, x, workspace=torch.empty(10, dtype=torch.bfloat16, device="cuda"))
    assert e.value.status == "EP_ERR_INVALID_ARG"
    db8 = ep.DeviceBlob(oracle.encode(w, 3.0, "fp8"))
    with pytest.raises(ep.EntroPackError) as e:
        ep.compressed_linear(db8, x)
    assert e.value.status == "EP_ERR_UNSUPPORTED"


def test_compressed_linear_module(ep):
    torch.manual_seed(0)
    w = synth.student_t5_bf16(65, 512, 1024)
    lin = torch.nn.Linear(1024, 512, bias=True)
    with torch.no_grad():
        lin.weight.copy_(torch.from_numpy(synth.bf16_to_f32(w)))
    cl = ep.CompressedLinear.from_linear(lin, ep.EntroPackLossyConfig(4.0))
    x = torch.randn(2, 50, 1024).to(torch.bfloat16).cuda()
    y = cl(x)
    assert y.shape == (2, 50, 512)
    w_hat = oracle.container_to_f64(oracle.decode(oracle.encode(w, 4.0))[0], "bf16")
    b_bits = lin.bias.detach().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    x_bits = x.reshape(-1, 1024).cpu().view(torch.int16).numpy().view(np.uint16)
    _check(y.reshape(-1, 512), x_bits, w_hat, bias_bits=b_bits)


def test_compress_linears_with_allocation(ep):
    """Three layers under one 3.5-bit budget: each forward matches the oracle's decode at its allocated index."""
    torch.manual_seed(1)
    shapes = {"attn.q": (256, 512), "ffn.up": (1024, 512), "ffn.down": (512, 1024)}
    gens = {"attn.q": synth.normal_bf16, "ffn.up": synth.student_t5_bf16, "ffn.down": synth.student_t5_bf16}
    lins, bits = {}, {}
    for i, (k, (n, kk)) in enumerate(shapes.items()):
        bits[k] = gens[k](70 + i, n, kk)
        lin = torch.nn.Linear(kk, n, bias=(k != "ffn.down"))
        with torch.no_grad():
            lin.weight.copy_(torch.from_numpy(synth.bf16_to_f32(bits[k])))
        lins[k] = lin
    sens = {"attn.q": 4.0}
    cls, record = ep.compress_linears(lins, 3.5, sens)
    plan = oracle.allocate_bits([bits[k] for k in shapes], 3.5, [sens.get(k, 1.0) for k in shapes])
    assert [record["layers"][k]["j"] for k in shapes] == plan["j"]
    assert record["layers"]["attn.q"]["j"] == plan["t"] - 64
    for k, (n, kk) in shapes.items():
        blob = oracle.encode_at(bits[k], plan["j"][list(shapes).index(k)],
                                record["layers"][k]["est_bpp"])
        assert cls[k].ct.blob.host.numpy().tobytes() == blob
        x_bits = synth.normal_bf16(80, 100, kk, std=1.0)
        y = cls[k](_bf16_dev(x_bits))
        w_hat = oracle.container_to_f64(oracle.decode(blob)[0], "bf16")
        if lins[k].bias is None:
            _check(y, x_bits, w_hat)
        else:
            b = lins[k].bias.detach().to(torch.bfloat16).double().numpy()
            ref = oracle.gemm_f64(synth.bf16_to_f32(x_bits).astype(np.float64), w_hat) + b
            err = np.abs(y.double().cpu().numpy() - ref).max() / np.abs(ref).max()
            assert err < 2e-2
