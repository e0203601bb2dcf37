"""GPU parity of the block-wise (BW) path through the C ABI: the prune (block
selection, offsets, schedule, packed operand) bit-exact against the oracle, and
the block-sparse GEMM (with and without the fused epilogue) within the bound,
on ragged M, empty and full tiles, and the 4096^3 tile-wise shape."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import REL, bits_of, canary_intact, dev_padded, dev_tensor, guarded_output, lib, rand_bits
from structured_sparse_dnn_gb300 import inputs as I

pytestmark = pytest.mark.gpu

CASES = [
    (300, 256, 40, [1, 4, 0]),              # ragged M, a full tile and an empty one
    (512, 1024, 72, [3, 16, 7, 1]),
    (128, 64, 256, [1]),
]


def _check_form(form, ref):
    assert np.array_equal(form.offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(form.indices.cpu().numpy(), ref["indices"])
    assert np.array_equal(form.schedule.cpu().numpy(), ref["schedule_table"])
    assert np.array_equal(bits_of(form.packed), ref["packed"])


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("case", CASES)
def test_bw_prune_and_gemm(dt, case):
    ss = lib()
    M, K, N, keep = case
    keep = np.array(keep, dtype=np.int32)
    W = rand_bits(900 + M + K, (M, K), dt, 0.5)
    X = rand_bits(910 + N, (K, N), dt, 1.0)
    form = ss.bw_prune_compress(dev_tensor(W, dt), keep)
    Y, buf = guarded_output(M, N, torch.bfloat16 if dt == "bf16" else torch.float16)
    ss.bw_gemm(form, dev_padded(X, dt), out=Y)
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    ref = oracle.bw.prune(W, dt, keep)
    _check_form(form, ref)
    Y_ref, B = oracle.bw.gemm(ref, keep, X, dt, dt, M)
    ok = oracle.gemm.within_bound(bits_of(Y), Y_ref, B, dt, REL[dt])
    assert ok.all(), f"{(~ok).sum()} outside the bound"
    assert canary_intact(buf, M, N)


def test_bw_gemm_fused_epilogue():
    ss = lib()
    M, K, N = 384, 512, 264
    keep = np.array([2, 8, 0], dtype=np.int32)
    W = rand_bits(920, (M, K), "bf16", 0.5)
    X = rand_bits(921, (K, N), "bf16", 1.0)
    bias = (np.random.default_rng(4).standard_normal(M) * 0.5).astype(np.float32)
    form = ss.bw_prune_compress(dev_tensor(W, "bf16"), keep)
    Y, buf = guarded_output(M, N, torch.float8_e4m3fn, pad_cols=24)   # 288-byte rows
    ss.bw_gemm(form, dev_padded(X, "bf16"), out=Y, alpha=0.5, bias=torch.from_numpy(bias).cuda(), act="gelu",
               y_scale=4.0)
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    ref = oracle.bw.prune(W, "bf16", keep)
    Wm = oracle.bw.masked_dense(W, ref, keep)
    want = oracle.epilogue.gemm_dense_ep(Wm, X, "bf16", "e4m3", 0.5, bias.astype(np.float64), "gelu", 4.0)
    B = oracle.gemm.bound(Wm, X, "bf16", 0.5)
    ok = oracle.epilogue.within_bound_ep(bits_of(Y), want, B, "e4m3", REL["bf16"], "gelu", 4.0)
    assert ok.all(), f"{(~ok).sum()} outside the bound"
    assert canary_intact(buf, M, N)


def test_bw_tile_wise_workload_sampled_tiles():
    """The 4096^3 bf16 shape with per-tile kept blocks drawn like the tile-wise
    kept fractions (15-35 %), in the configuration the benchmark times."""
    ss = lib()
    wl = I.WORKLOADS["tile_wise_4096_bf16"]
    d = wl.make()
    keep = (d["keep"] // 64).astype(np.int32)
    form = ss.bw_prune_compress(I.torch_view(d["W"], "bf16").cuda(), keep)
    Y = ss.bw_gemm(form, I.torch_view(d["X"], "bf16").cuda())
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    ref = oracle.bw.prune(d["W"], "bf16", keep)
    _check_form(form, ref)
    order = ref["schedule_table"].reshape(-1, 4)[:, 0]
    tiles = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})
    Y_ref, B = oracle.bw.gemm(ref, keep, d["X"], "bf16", "bf16", wl.M, tiles=tiles)
    yb = bits_of(Y)
    for t in tiles:
        sl = slice(128 * t, 128 * (t + 1))
        ok = oracle.gemm.within_bound(yb[sl], Y_ref[sl], B[sl], "bf16", REL["bf16"])
        assert ok.all(), f"tile {t}: {(~ok).sum()} outside the bound"
