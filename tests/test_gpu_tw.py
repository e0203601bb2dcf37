"""GPU parity of the tile-wise (TW) and tile-vector-wise (TVW) path through the
C ABI: offsets, indices, schedule, packed operand and metadata bit-exact
against the oracle; the fused gather GEMM within the elementwise bound;
empty, full and ragged tiles."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import REL, bits_of, canary_intact, dev_tensor, guarded_output, lib, rand_bits

pytestmark = pytest.mark.gpu

CASES = [
    # M, K, N, keep (one entry per 128-row tile)
    (256, 256, 64, [64, 128]),
    (300, 200, 72, [8, 0, 200]),
    (384, 1024, 256, [1024, 0, 516]),
    (128, 4096, 320, [1000]),
    (512, 512, 512, [4, 96, 260, 512]),
]


@pytest.mark.parametrize("tvw", [False, True])
@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_tw_prune_bit_exact_and_gemm(tvw, case, dt):
    ss = lib()
    M, K, N, keep = case
    keep = np.array(keep, dtype=np.int32)
    if not tvw:
        keep = np.where(keep % 4 == 0, keep, keep)  # TW accepts any L
    elif (keep % 4).any():
        pytest.skip("TVW needs L % 4 == 0")
    W = rand_bits(600 + M + K, (M, K), dt, 0.02)
    X = rand_bits(700 + N, (K, N), dt, 1.0)
    form = ss.tw_prune_compress(dev_tensor(W, dt), keep, tvw=tvw)
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    ref = oracle.tw.prune(W, dt, keep, tvw)
    assert np.array_equal(form.offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(form.indices.cpu().numpy(), ref["indices"])
    assert np.array_equal(form.schedule.cpu().numpy(), ref["schedule_table"])
    assert np.array_equal(bits_of(form.packed), ref["packed"])
    if tvw:
        assert np.array_equal(bits_of(form.meta), ref["meta"])
        assert np.array_equal(bits_of(form.meta_hw), ref["meta_hw"])
    Y, buf = guarded_output(M, N, torch.bfloat16 if dt == "bf16" else torch.float16)
    ss.tvw_gemm(form, dev_tensor(X, dt), out=Y)
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    Y_ref, B = oracle.tw.gemm(ref, keep, X, dt, dt, M, tvw)
    ok = oracle.gemm.within_bound(bits_of(Y), Y_ref, B, dt, REL[dt])
    assert ok.all(), f"{(~ok).sum()} outside the bound"
    assert canary_intact(buf, M, N)


def test_all_tiles_empty_gives_zero():
    ss = lib()
    M, K, N = 256, 128, 64
    W = rand_bits(1, (M, K), "bf16", 0.02)
    keep = np.zeros(2, dtype=np.int32)
    form = ss.tw_prune_compress(dev_tensor(W, "bf16"), keep, tvw=False)
    Y = torch.full((M, N), 5.0, dtype=torch.bfloat16, device="cuda")
    ss.tvw_gemm(form, dev_tensor(rand_bits(2, (K, N), "bf16"), "bf16"), out=Y)
    assert (Y == 0).all()


def test_full_keep_matches_dense_gemm_bits_within_bound():
    ss = lib()
    M, K, N = 256, 256, 128
    W = rand_bits(3, (M, K), "bf16", 0.02)
    X = rand_bits(4, (K, N), "bf16")
    keep = np.full(2, K, dtype=np.int32)
    form = ss.tw_prune_compress(dev_tensor(W, "bf16"), keep, tvw=False)
    Y = ss.tvw_gemm(form, dev_tensor(X, "bf16"))
    Y_ref = oracle.gemm.gemm_dense(W, X, "bf16", "bf16")
    B = oracle.gemm.bound(W, X, "bf16")
    assert oracle.gemm.within_bound(bits_of(Y), Y_ref, B, "bf16", 1e-2).all()


@pytest.mark.parametrize("pattern", ["tw", "tvw", "bw", "ew"])
def test_prune_into_existing_result_matches_fresh(pattern):
    """out= overwrites an earlier result in place: pruning a second weight into the
    first weight's buffers gives exactly what a fresh call on it gives."""
    ss = lib()
    M, K, dt = 384, 512, "bf16"
    W1 = dev_tensor(rand_bits(901, (M, K), dt, 0.02), dt)
    W2 = dev_tensor(rand_bits(902, (M, K), dt, 0.02), dt)
    if pattern in ("tw", "tvw"):
        keep = np.array([128, 64, 256], dtype=np.int32)
        tvw = pattern == "tvw"
        work = torch.empty(ss.tw_sizes(ss.BF16, tvw, M, K, keep)["workspace_bytes"], dtype=torch.uint8,
                           device="cuda")
        form = ss.tw_prune_compress(W1, keep, tvw, work)
        fresh = ss.tw_prune_compress(W2, keep, tvw, work)
        again = ss.tw_prune_compress(W2, keep, tvw, work, out=form)
        names = ["offsets", "indices", "schedule", "packed"] + (["meta", "meta_hw"] if tvw else [])
    elif pattern == "bw":
        keep = np.array([2, 0, 8], dtype=np.int32)
        work = torch.empty(ss.bw_sizes(ss.BF16, M, K, keep)["workspace_bytes"], dtype=torch.uint8, device="cuda")
        form = ss.bw_prune_compress(W1, keep, work)
        fresh = ss.bw_prune_compress(W2, keep, work)
        again = ss.bw_prune_compress(W2, keep, work, out=form)
        names = ["offsets", "indices", "schedule", "packed"]
    else:
        k = 51
        work = torch.empty(ss.ew_sizes(ss.BF16, M, K, k)["workspace_bytes"], dtype=torch.uint8, device="cuda")
        form = ss.ew_prune_compress(W1, k, work)
        fresh = ss.ew_prune_compress(W2, k, work)
        again = ss.ew_prune_compress(W2, k, work, out=form)
        names = ["row_ptr", "col_idx", "vals"]
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    assert again is form
    for n in names:
        a, b = getattr(again, n), getattr(fresh, n)
        assert torch.equal(a.view(torch.uint8) if a.dtype != torch.int32 else a,
                           b.view(torch.uint8) if b.dtype != torch.int32 else b), n
    with pytest.raises(ValueError):
        if pattern in ("tw", "tvw"):
            ss.tw_prune_compress(W2, keep + 4, pattern == "tvw", work, out=form)
        elif pattern == "bw":
            ss.bw_prune_compress(W2, keep + 1, work, out=form)
        else:
            ss.ew_prune_compress(W2, k + 1, work, out=form)
