"""The allocation-free tile-wise prune, tw_prune_compress_noalloc.

Some callers cannot allocate device memory during a call (a plugin inside an
inference engine that only gets its input and output buffers, a serving loop
that must not call cudaMalloc/cudaFree). For them the library keeps the score
scratch in a fixed device array. This test calls that entry point through the
C ABI twice in a row, on two different weights, and checks each result against
the ordinary entry point (which takes a caller workspace): offsets, indices,
schedule, packed operand and metadata must be bit-identical, including on
weights with several tiles of equal kept length (the schedule's tie order). The
refusal of problems beyond the fixed limits is a host-only test in test_abi.py
(no device may see a refused problem). The file sorts last so that
a run stopping at the first failure has run every other test before it; it must
also pass on its own in a fresh process.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from gpu_helpers import dev_tensor, lib, rand_bits

pytestmark = pytest.mark.gpu


def _call_noalloc(ss, W: torch.Tensor, keep: np.ndarray, tvw: bool):
    M, K = W.shape
    dt = ss._DT[W.dtype]
    sz = ss.tw_sizes(dt, tvw, M, K, keep)
    nt = (M + 127) // 128
    dev = W.device
    offsets = torch.full((nt + 1,), -1, dtype=torch.int32, device=dev)
    indices = torch.full((max(1, sz["indices_count"]),), -1, dtype=torch.int32, device=dev)
    schedule = torch.full((4 * nt,), -1, dtype=torch.int32, device=dev)
    packed = torch.zeros(max(8, sz["packed_bytes"] // 2), dtype=W.dtype, device=dev)
    meta = torch.zeros(max(16, sz["meta_bytes"]), dtype=torch.uint8, device=dev) if tvw else None
    meta_hw = torch.zeros(max(16, sz["meta_hw_bytes"]), dtype=torch.uint8, device=dev) if tvw else None
    k = np.ascontiguousarray(keep, dtype=np.int32)
    st = ss.lib.tw_prune_compress_noalloc(
        dt, int(tvw), W.data_ptr(), M, K, W.stride(0), k.ctypes.data_as(C.POINTER(C.c_int32)),
        offsets.data_ptr(), indices.data_ptr(), schedule.data_ptr(), packed.data_ptr(),
        None if meta is None else meta.data_ptr(), None if meta_hw is None else meta_hw.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert st == 0, ss.status_str(st)
    torch.cuda.synchronize()
    n = sz["indices_count"]
    return (offsets.cpu(), indices[:n].cpu(), schedule.cpu(), packed[:sz["packed_bytes"] // 2].cpu(),
            None if meta is None else meta[:sz["meta_bytes"]].cpu(),
            None if meta_hw is None else meta_hw[:sz["meta_hw_bytes"]].cpu())


def _call_ordinary(ss, W, keep, tvw):
    f = ss.tw_prune_compress(W, keep, tvw)
    torch.cuda.synchronize()
    return (f.offsets.cpu(), f.indices.cpu(), f.schedule.cpu(), f.packed.cpu(),
            None if f.meta is None else f.meta.cpu(), None if f.meta_hw is None else f.meta_hw.cpu())


def _same(a, b):
    for x, y in zip(a, b):
        if x is None or y is None:
            assert x is None and y is None
        else:
            assert torch.equal(x.view(torch.uint8) if x.dtype != torch.int32 else x,
                               y.view(torch.uint8) if y.dtype != torch.int32 else y)


def test_noalloc_matches_ordinary_entry_point_two_calls_in_a_row():
    ss = lib()
    cases = [
        (512, 1024, np.array([256, 0, 516, 1024], dtype=np.int32), True),   # TVW, an empty and a full tile
        (300, 200, np.array([7, 0, 200], dtype=np.int32), False),          # TW, ragged M and L
        # several tiles of equal length: the schedule's tie order (length
        # descending, tile ascending) computed on the device must match the host's
        (1000, 512, np.array([128, 64, 128, 64, 128, 0, 64, 128], dtype=np.int32), True),
        (1024, 256, np.array([64, 64, 64, 64, 64, 64, 64, 64], dtype=np.int32), False),
    ]
    for i, (M, K, keep, tvw) in enumerate(cases):
        W = dev_tensor(rand_bits(9100 + i, (M, K), "bf16", 0.02), "bf16")
        got = _call_noalloc(ss, W, keep, tvw)
        want = _call_ordinary(ss, W, keep, tvw)
        _same(got, want)
        assert ss.check_device_error() == 0
