"""GPU check of ep_batch_decode_static, the allocation-free batched decode.

Callers that cannot allocate device memory (code running under another
framework's allocator or memory budget, plug-ins inside a host process that
owns every allocation, latency-critical paths where cudaMalloc would stall)
use this entry point; its scratch lives in a device array inside the
library.  The test calls it through the C ABI twice in a row, with two
different sets of streams, and compares each result bit for bit with the
workspace-based entry point (ep_batch_prepare + ep_batch_decode) and with the
CPU oracle's decode of the same streams.  A third call passes more streams
than the entry point stages per host chunk, so the descriptor and unit-table
copies at nonzero offsets are exercised too.  It also checks that an
oversized batch is refused before any work is enqueued.

The file name sorts last so that a run which stops at the first failure has
already run every other test.
"""
import ctypes

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


def _items(ep, blobs, outs):
    from dit_weight_compression_02_b300._lib import EpBatchItem
    arr = (EpBatchItem * len(blobs))()
    for i, (b, o) in enumerate(zip(blobs, outs)):
        arr[i] = EpBatchItem(b.host.data_ptr(), b.device.data_ptr(), b.nbytes, o.data_ptr(), 0)
    return arr


def _static_call(ep, blobs, outs, ring):
    from dit_weight_compression_02_b300._lib import check, lib
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    check(lib.ep_batch_decode_static(_items(ep, blobs, outs), len(blobs), ring, ctypes.c_void_p(status.data_ptr()),
                                     ctypes.c_void_p(stream.cuda_stream)), "ep_batch_decode_static")
    ep.sync_status(status)


def _workspace_call(ep, blobs, ring, shapes):
    outs = [torch.zeros(s, dtype=torch.bfloat16, device="cuda") for s in shapes]
    ep.BatchDecoder(blobs, outs, ring=ring)()
    return outs


def _bits(t):
    return t.view(torch.int16).cpu().numpy()


def test_static_batch_matches_workspace_entry_twice(ep):
    # call 1: seven layers of one transformer block with distinct outputs
    shapes1 = [(512, 3840)] * 4 + [(1024, 3840)] * 2 + [(512, 1024)]
    host1 = [oracle.encode(synth.student_t5_bf16(300 + i, r, c), 4.0) for i, (r, c) in enumerate(shapes1)]
    blobs1 = [ep.DeviceBlob(b) for b in host1]
    ref1 = _workspace_call(ep, blobs1, 0, shapes1)
    outs1 = [torch.full(s, 7.0, dtype=torch.bfloat16, device="cuda") for s in shapes1]
    _static_call(ep, blobs1, outs1, ring=0)
    for a, b, h in zip(outs1, ref1, host1):
        assert (_bits(a) == _bits(b)).all()
        assert (_bits(a).view(np.uint16) == oracle.decode(h)[0]).all()

    # call 2: a different batch (ragged tile groups, a ring of two reused
    # buffers), so the array's leftover descriptors and counters from call 1
    # must not leak into the result
    shapes2 = [(96, 384), (224, 640), (96, 384), (224, 640), (96, 384)]
    blobs2 = [ep.DeviceBlob(ep.encode(synth.rows_outliers_bf16(400 + i, r, c), 3.5)) for i, (r, c) in enumerate(shapes2)]
    ref2 = _workspace_call(ep, blobs2, 0, shapes2)
    ring_bufs = [torch.full(shapes2[k], 3.0, dtype=torch.bfloat16, device="cuda") for k in range(2)]
    _static_call(ep, blobs2, [ring_bufs[i % 2] for i in range(len(blobs2))], ring=2)
    for k in range(2):
        last = max(i for i in range(len(blobs2)) if i % 2 == k)
        assert (_bits(ring_bufs[k]) == _bits(ref2[last])).all()
        assert (_bits(ring_bufs[k]).view(np.uint16) == oracle.decode(blobs2[last].host.numpy().tobytes())[0]).all()


def test_static_batch_more_items_than_one_host_chunk(ep):
    # 57 small streams: the entry point stages descriptors 32 at a time, so the
    # second chunk's copies land at a nonzero offset of the array, and the
    # unit table's final entry is written after both chunks
    shapes = [(32 * (1 + i % 3), 128 * (1 + i % 4)) for i in range(57)]
    host = [oracle.encode(synth.normal_bf16(700 + i, r, c), 3.0 + 0.5 * (i % 3)) for i, (r, c) in enumerate(shapes)]
    blobs = [ep.DeviceBlob(b) for b in host]
    ref = _workspace_call(ep, blobs, 0, shapes)
    outs = [torch.full(s, -1.0, dtype=torch.bfloat16, device="cuda") for s in shapes]
    _static_call(ep, blobs, outs, ring=0)
    for a, b, h in zip(outs, ref, host):
        assert (_bits(a) == _bits(b)).all()
        assert (_bits(a).view(np.uint16) == oracle.decode(h)[0]).all()


def test_static_batch_rejects_oversized_batch(ep):
    from dit_weight_compression_02_b300._lib import EpBatchItem, lib
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    n = 1025  # one more than the library's fixed capacity
    items = (EpBatchItem * n)()
    rc = lib.ep_batch_decode_static(items, n, 0, ctypes.c_void_p(status.data_ptr()),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 1  # EP_ERR_INVALID_ARG, before any work is enqueued
    assert int(status.item()) == 0
