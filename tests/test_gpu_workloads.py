"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times: compression bit-exact in full; Y within the elementwise
bound in full where the oracle finishes in seconds, else on sampled rows
(first and last 128 and a seeded random set) or sampled tiles."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import REL, bits_of, lib
from structured_sparse_dnn_gb300 import inputs as I

pytestmark = pytest.mark.gpu

SMALL = ["toy_fp16", "bert_ffn_up_bf16", "bert_ffn_down_bf16", "resnet50_1x1_fp16"]
LARGE = ["llm_ffn_e4m3", "llm_ffn_bf16"]


def _run_sp24(ss, wl, d):
    Wd = I.torch_view(d["W"], wl.dt).cuda()
    Xd = I.torch_view(d["X"], wl.dt).cuda()
    f = ss.sp24_prune_compress(Wd)
    Y = ss.sp24_gemm(f, Xd, alpha=d["alpha"], out_dtype=torch.bfloat16 if wl.out_dt == "bf16" else torch.float16)
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    return f, Y, Wd, Xd


@pytest.mark.parametrize("name", SMALL)
def test_small_workload_full(name):
    ss = lib()
    wl = I.WORKLOADS[name]
    d = wl.make()
    f, Y, _, _ = _run_sp24(ss, wl, d)
    v_ref, m_ref = oracle.sp24.compress(d["W"], wl.dt)
    assert np.array_equal(bits_of(f.values), v_ref)
    assert np.array_equal(bits_of(f.meta), m_ref)
    assert np.array_equal(bits_of(f.meta_hw), oracle.sp24.meta_hw_from_canonical(m_ref, wl.M, wl.K, wl.dt))
    Y_ref = oracle.gemm.gemm_sp24(v_ref, m_ref, wl.K, d["X"], wl.dt, wl.out_dt, d["alpha"])
    B = oracle.gemm.bound(oracle.sp24.decompress(v_ref, m_ref, wl.K), d["X"], wl.dt, d["alpha"])
    ok = oracle.gemm.within_bound(bits_of(Y), Y_ref, B, wl.out_dt, REL[wl.dt])
    assert ok.all(), f"{(~ok).sum()} outside the bound"


def _sample_rows(M, seed=0, n=256):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([np.arange(128), np.arange(M - 128, M), rng.choice(M, n, replace=False)]))


@pytest.mark.parametrize("name", LARGE)
def test_large_workload_compress_full_gemm_sampled(name):
    ss = lib()
    wl = I.WORKLOADS[name]
    d = wl.make()
    f, Y, Wd, Xd = _run_sp24(ss, wl, d)
    v_ref, m_ref = oracle.sp24.compress(d["W"], wl.dt)
    assert np.array_equal(bits_of(f.values), v_ref)
    assert np.array_equal(bits_of(f.meta), m_ref)
    assert np.array_equal(bits_of(f.meta_hw), oracle.sp24.meta_hw_from_canonical(m_ref, wl.M, wl.K, wl.dt))
    rows = _sample_rows(wl.M)
    Yr = bits_of(Y[torch.from_numpy(rows).cuda()])
    Y_ref = oracle.gemm.gemm_sp24(v_ref, m_ref, wl.K, d["X"], wl.dt, wl.out_dt, d["alpha"], rows=rows)
    B = oracle.gemm.bound(oracle.sp24.decompress(v_ref[rows], m_ref[rows], wl.K), d["X"], wl.dt, d["alpha"])
    ok = oracle.gemm.within_bound(Yr, Y_ref, B, wl.out_dt, REL[wl.dt])
    assert ok.all(), f"{(~ok).sum()} outside the bound"
    # the dense GEMM of the same family on the same shape (sampled rows)
    Yd = ss.dense_gemm(Wd, Xd, alpha=d["alpha"], out_dtype=torch.bfloat16 if wl.out_dt == "bf16" else torch.float16)
    Ydr = bits_of(Yd[torch.from_numpy(rows).cuda()])
    Yd_ref = oracle.gemm.gemm_dense(d["W"], d["X"], wl.dt, wl.out_dt, d["alpha"], rows=rows)
    Bd = oracle.gemm.bound(d["W"], d["X"], wl.dt, d["alpha"], rows=rows)
    ok = oracle.gemm.within_bound(Ydr, Yd_ref, Bd, wl.out_dt, REL[wl.dt])
    assert ok.all(), f"dense: {(~ok).sum()} outside the bound"


@pytest.mark.parametrize("tvw", [False, True])
def test_tile_wise_workload(tvw):
    ss = lib()
    wl = I.WORKLOADS["tile_wise_4096_bf16"]
    d = wl.make()
    keep = d["keep"] if not tvw else (d["keep"] // 4) * 4
    Wd = I.torch_view(d["W"], "bf16").cuda()
    Xd = I.torch_view(d["X"], "bf16").cuda()
    form = ss.tw_prune_compress(Wd, keep, tvw=tvw)
    Y = ss.tvw_gemm(form, Xd)
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    ref = oracle.tw.prune(d["W"], "bf16", keep, tvw)
    assert np.array_equal(form.offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(form.indices.cpu().numpy(), ref["indices"])
    assert np.array_equal(form.schedule.cpu().numpy(), ref["schedule_table"])
    assert np.array_equal(bits_of(form.packed), ref["packed"])
    if tvw:
        assert np.array_equal(bits_of(form.meta), ref["meta"])
        assert np.array_equal(bits_of(form.meta_hw), ref["meta_hw"])
    order = ref["schedule"]
    tiles = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})
    Y_ref, B = oracle.tw.gemm(ref, keep, d["X"], "bf16", "bf16", wl.M, tvw, tiles=tiles)
    yb = bits_of(Y)
    for t in tiles:
        sl = slice(t * 128, (t + 1) * 128)
        ok = oracle.gemm.within_bound(yb[sl], Y_ref[sl], B[sl], "bf16", 1e-2)
        assert ok.all(), f"tile {t}: {(~ok).sum()} outside the bound"
