"""GPU parity of the fused layer epilogue (per-row bias, ReLU / GELU, output
scale, e4m3 output) through the C ABI, against the oracle's epilogue: 2:4,
dense and tile-wise GEMMs, ragged shapes, untouched canaries, the empty product
(K == 0) and an empty tile, and the LLM FFN shape on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import REL, bits_of, canary_intact, dev_padded, dev_tensor, guarded_output, lib, rand_bits
from structured_sparse_dnn_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TORCH_OUT = {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}


def _bias(seed, M):
    return (np.random.default_rng(seed).standard_normal(M) * 0.5).astype(np.float32)


def _check(Y, ref, B, out_dt, rel, act, ys):
    ok = oracle.epilogue.within_bound_ep(bits_of(Y), ref, B, out_dt, rel, act, ys)
    if not ok.all():
        i, j = np.argwhere(~ok)[0]
        y = oracle.codecs.decode(bits_of(Y)[i, j], out_dt)
        r = oracle.codecs.decode(ref[i, j], out_dt)
        raise AssertionError(f"{(~ok).sum()} of {ok.size} outside the bound; first at {i},{j}: gpu {y} ref {r}")


@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3"])
@pytest.mark.parametrize("act", ["none", "relu", "gelu"])
@pytest.mark.parametrize("out_e4m3", [False, True])
@pytest.mark.parametrize("tile", [0, 9256, 19256])
def test_sp24_gemm_epilogue(dt, act, out_e4m3, tile):
    """The fused epilogue on the shape's own tiles (variant 0) and on forced SM-pair
    tiles with one- and two-step stages (9256, 19256)."""
    ss = lib()
    M, N, K = 300, 264, 520
    W = rand_bits(610 + M, (M, K), dt, 0.5)
    X = rand_bits(620 + N, (K, N), dt, 1.0)
    out_dt = "e4m3" if out_e4m3 else ("bf16" if dt == "e4m3" else dt)
    alpha = 0.75 if dt == "e4m3" else 1.0
    ys = 4.0 if out_e4m3 else 0.5
    bias = _bias(7, M)
    f = ss.sp24_prune_compress(dev_tensor(W, dt), canonical_meta=False)
    Y, buf = guarded_output(M, N, TORCH_OUT[out_dt])
    ss.sp24_gemm(f, dev_padded(X, dt), alpha=alpha, out=Y, bias=torch.from_numpy(bias).cuda(), act=act, y_scale=ys,
                 variant=tile)
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    v, m = oracle.sp24.compress(W, dt)
    ref = oracle.epilogue.gemm_sp24_ep(v, m, K, X, dt, out_dt, alpha, bias.astype(np.float64), act, ys)
    B = oracle.gemm.bound(oracle.sp24.decompress(v, m, K), X, dt, alpha)
    _check(Y, ref, B, out_dt, REL[dt], act, ys)
    assert canary_intact(buf, M, N)


@pytest.mark.parametrize("act", ["relu", "gelu"])
@pytest.mark.parametrize("dt", ["bf16", "e4m3"])
def test_dense_gemm_epilogue(act, dt):
    ss = lib()
    M, N, K = 384, 264, 512
    W = rand_bits(630, (M, K), dt, 0.5)
    X = rand_bits(640, (K, N), dt, 1.0)
    bias = _bias(8, M)
    Y, buf = guarded_output(M, N, torch.float8_e4m3fn)
    ss.dense_gemm(dev_padded(W, dt), dev_padded(X, dt), out=Y, bias=torch.from_numpy(bias).cuda(), act=act,
                  y_scale=2.0)
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    ref = oracle.epilogue.gemm_dense_ep(W, X, dt, "e4m3", 1.0, bias.astype(np.float64), act, 2.0)
    B = oracle.gemm.bound(W, X, dt)
    _check(Y, ref, B, "e4m3", REL[dt], act, 2.0)
    assert canary_intact(buf, M, N)


@pytest.mark.parametrize("tvw", [False, True])
@pytest.mark.parametrize("out_dt", ["bf16", "e4m3"])
def test_tile_wise_gemm_epilogue_with_an_empty_tile(tvw, out_dt):
    ss = lib()
    M, N, K = 512, 272, 384
    keep = np.array([128, 0, 200, 96], dtype=np.int32)          # tile 1 keeps nothing: rows = act(bias)
    W = rand_bits(650, (M, K), "bf16", 0.5)
    X = rand_bits(660, (K, N), "bf16", 1.0)
    bias = _bias(9, M)
    ys = 4.0 if out_dt == "e4m3" else 1.0
    form = ss.tw_prune_compress(dev_tensor(W, "bf16"), keep, tvw=tvw)
    Y, buf = guarded_output(M, N, TORCH_OUT[out_dt], pad_cols=16)
    ss.tvw_gemm(form, dev_padded(X, "bf16"), out=Y, alpha=0.5, bias=torch.from_numpy(bias).cuda(), act="gelu",
                y_scale=ys)
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    ref = oracle.tw.prune(W, "bf16", keep, tvw)
    yb = bits_of(Y)
    for t in range(len(keep)):
        sl = slice(t * 128, (t + 1) * 128)
        # the tile's masked dense weight (kept columns only; TVW also 2:4 within them)
        Wt = _masked_dense(ref, keep, t, K, tvw)
        acc = oracle.gemm.dense_product(Wt, X, "bf16", 0.5)
        want = oracle.codecs.encode(oracle.epilogue.apply(acc, bias[sl].astype(np.float64), "gelu", ys), out_dt)
        B = oracle.gemm.bound(Wt, X, "bf16", 0.5)
        ok = oracle.epilogue.within_bound_ep(yb[sl], want, B, out_dt, 1e-2, "gelu", ys)
        assert ok.all(), f"tile {t}: {(~ok).sum()} outside the bound"
    assert canary_intact(buf, M, N)


def _masked_dense(ref, keep, t, K, tvw):
    """The 128 x K weight tile t contributes: its kept block (TVW: after 2:4)
    scattered to its K indices, zeros elsewhere."""
    o, L = int(ref["offsets"][t]), int(keep[t])
    blk = oracle.tw.unpack_tile(ref, keep, t, tvw, "bf16")
    Wt = np.zeros((128, K), dtype=blk.dtype)
    Wt[:, ref["indices"][o:o + L]] = blk
    return Wt


@pytest.mark.parametrize("out_dt", ["bf16", "e4m3"])
def test_empty_product_is_the_activated_bias(out_dt):
    ss = lib()
    M, N = 200, 48
    bias = _bias(10, M)
    Y, buf = guarded_output(M, N, TORCH_OUT[out_dt], pad_cols=16)
    X = torch.zeros((0, N), dtype=torch.bfloat16, device="cuda")
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    ss.sp24_gemm(ss.Sp24(ss.BF16, M, 0, z, None, z), X, out=Y, bias=torch.from_numpy(bias).cuda(), act="gelu",
                 y_scale=3.0)
    torch.cuda.synchronize()
    want = oracle.codecs.encode(oracle.epilogue.apply(np.zeros((M, N)), bias.astype(np.float64), "gelu", 3.0),
                                out_dt)
    ok = oracle.epilogue.within_bound_ep(bits_of(Y), want, np.zeros((M, N)), out_dt, 0.0, "gelu", 3.0)
    assert ok.all()
    assert canary_intact(buf, M, N)


def test_llm_ffn_e4m3_epilogue_sampled_rows():
    """The LLM FFN up-projection shape, e4m3 in and e4m3 out with bias + GELU, in
    the launch configuration of the plain GEMM; rows sampled."""
    ss = lib()
    wl = I.WORKLOADS["llm_ffn_e4m3"]
    d = wl.make()
    bias = _bias(11, wl.M)
    f = ss.sp24_prune_compress(I.torch_view(d["W"], "e4m3").cuda(), canonical_meta=False)
    Y = torch.empty((wl.M, wl.N), dtype=torch.float8_e4m3fn, device="cuda")
    ss.sp24_gemm(f, I.torch_view(d["X"], "e4m3").cuda(), alpha=d["alpha"], out=Y,
                 bias=torch.from_numpy(bias).cuda(), act="gelu", y_scale=8.0)
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(128), np.arange(wl.M - 128, wl.M), rng.choice(wl.M, 128, False)]))
    v, m = oracle.sp24.compress(d["W"], "e4m3")
    ref = oracle.epilogue.gemm_sp24_ep(v, m, wl.K, d["X"], "e4m3", "e4m3", d["alpha"], bias.astype(np.float64),
                                       "gelu", 8.0, rows=rows)
    B = oracle.gemm.bound(oracle.sp24.decompress(v[rows], m[rows], wl.K), d["X"], "e4m3", d["alpha"])
    yr = bits_of(Y.view(torch.uint8)[torch.from_numpy(rows).cuda()])
    ok = oracle.epilogue.within_bound_ep(yr, ref, B, "e4m3", REL["e4m3"], "gelu", 8.0)
    assert ok.all(), f"{(~ok).sum()} outside the bound"


@pytest.mark.parametrize("out_dt", ["bf16", "e4m3"])
@pytest.mark.parametrize("tile", [0, 19256])
def test_gelu_at_chosen_values(out_dt, tile):
    """GELU through the GEMM on chosen inputs: a 2:4 identity weight makes each
    accumulator exactly one X value (zero, tiny, moderate, large and far into either
    tail, both signs), with and without a bias. The accumulator is exact here, so the
    result must be the oracle's exact GELU to within the kernel's erf approximation
    (Abramowitz-Stegun 7.1.26: GELU error <= 1.7e-7 max(|x|, 1), absolute; relative to
    the tiny values of the far negative tail that is several output ulps) and one
    output ulp."""
    ss = lib()
    K = N = 256
    M = 256
    W = np.zeros((M, K))
    W[np.arange(M), np.arange(M) % K] = 1.0
    Wb = oracle.codecs.encode(W, "bf16")
    vals = np.array([0.0, -0.0, 1e-30, -1e-30, 1e-3, -1e-3, 0.25, -0.25, 0.5, -0.5, 1.0, -1.0, 1.5, -1.5, 2.0, -2.0,
                     3.0, -3.0, 4.5, -4.5, 5.5, -5.5, 8.0, -8.0, 12.0, -12.0, 20.0, -20.0, 100.0, -100.0, 1e4, -1e4])
    X = np.tile(vals, (K, N // len(vals)))
    X = X * (1.0 + np.arange(K)[:, None] / K)              # a different scale per row of X
    Xb = oracle.codecs.encode(X, "bf16")
    bias = np.where(np.arange(M) % 3 == 0, 0.0, np.where(np.arange(M) % 3 == 1, 2.0, -2.0)).astype(np.float32)
    ys = 4.0 if out_dt == "e4m3" else 1.0
    f = ss.sp24_prune_compress(dev_tensor(Wb, "bf16"), canonical_meta=False)
    Y, buf = guarded_output(M, N, TORCH_OUT[out_dt], pad_cols=16)  # row pitch a multiple of 16 bytes
    ss.sp24_gemm(f, dev_padded(Xb, "bf16"), out=Y, bias=torch.from_numpy(bias).cuda(), act="gelu", y_scale=ys,
                 variant=tile)
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    acc = oracle.codecs.decode(Wb, "bf16") @ oracle.codecs.decode(Xb, "bf16")
    z = acc + bias.astype(np.float64)[:, None]
    want = oracle.codecs.encode(oracle.epilogue.apply(acc, bias.astype(np.float64), "gelu", ys), out_dt)
    y = oracle.codecs.decode(bits_of(Y), out_dt)
    r = oracle.codecs.decode(want, out_dt)
    slack = ys * 1.7e-7 * np.maximum(np.abs(z), 1.0) + oracle.epilogue.ulp(np.maximum(np.abs(y), np.abs(r)), out_dt)
    bad = ~((np.abs(y - r) <= slack) & np.isfinite(y))
    assert not bad.any(), f"{bad.sum()} off; first at z = {z[bad][0]}: gpu {y[bad][0]} ref {r[bad][0]}"
    # inside |z| <= 3 the approximation is far below half an ulp: one ulp at most
    near = np.abs(z) <= 3.0
    assert (np.abs(y - r)[near] <= oracle.epilogue.ulp(np.maximum(np.abs(y), np.abs(r)), out_dt)[near]).all()
    assert canary_intact(buf, M, N)
