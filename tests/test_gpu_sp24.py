"""GPU parity of the 2:4 path through the C ABI: prune/compress bit-exact
against the oracle, sparse and dense GEMMs within the elementwise bound,
ragged shapes, edge values, strided operands and untouched canaries."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (CANARY, REL, bits_of, canary_intact, dev_padded, dev_tensor, guarded_output, lib,
                         rand_bits)

pytestmark = pytest.mark.gpu

SHAPES_C = [(1, 4), (5, 36), (128, 128), (130, 260), (257, 1000), (64, 4096)]


@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3"])
@pytest.mark.parametrize("shape", SHAPES_C)
def test_compress_bit_exact(dt, shape):
    ss = lib()
    M, K = shape
    W = rand_bits(100 + M + K, shape, dt, 0.02 if dt != "f16" else 1.0)
    f = ss.sp24_prune_compress(dev_tensor(W, dt))
    torch.cuda.synchronize()
    v_ref, m_ref = oracle.sp24.compress(W, dt)
    assert np.array_equal(bits_of(f.values), v_ref)
    assert np.array_equal(bits_of(f.meta), m_ref)
    assert np.array_equal(bits_of(f.meta_hw), oracle.sp24.meta_hw_from_canonical(m_ref, M, K, dt))
    assert ss.check_device_error() == 0


def test_compress_strided_input():
    ss = lib()
    M, K, ld = 70, 200, 264
    big = rand_bits(5, (M, ld), "bf16")
    Wt = dev_tensor(big, "bf16")[:, :K]
    f = ss.sp24_prune_compress(Wt)
    v_ref, m_ref = oracle.sp24.compress(np.ascontiguousarray(big[:, :K]), "bf16")
    assert np.array_equal(bits_of(f.values), v_ref) and np.array_equal(bits_of(f.meta), m_ref)


@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3"])
def test_compress_edge_values(dt):
    ss = lib()
    rng = np.random.default_rng(0)
    if dt == "e4m3":
        pool = np.array([0x00, 0x80, 0x01, 0x81, 0x07, 0x08, 0x38, 0xB8, 0x7E, 0xFE, 0x7D, 0x40], np.uint8)
    else:
        sgn = 0x8000
        pool = np.array([0, sgn, 1, sgn | 1, 0x3FF, 0x400, 0x3C00, sgn | 0x3C00, 0x7BFF, sgn | 0x7BFF,
                         0x3C01, 0x3BFF], np.uint16)
    W = pool[rng.integers(0, len(pool), size=(96, 512))]
    W[0, :] = pool[6]                       # all-equal groups
    W[1, :] = 0                             # all-zero groups
    f = ss.sp24_prune_compress(dev_tensor(W, dt))
    v_ref, m_ref = oracle.sp24.compress(W, dt)
    assert np.array_equal(bits_of(f.values), v_ref)
    assert np.array_equal(bits_of(f.meta), m_ref)


# The tile chooser gives the small shapes 128x64 tiles (16-bit) or 128x128
# (e4m3); (1280, 1000, 192) takes 128x128 and (3072, 1000, 128) 128x256 tiles,
# both with a ragged N; the last shape selects the 256-row tiles (two 128-row
# sub-tiles per CTA) with a ragged M.
GEMM_SHAPES = [(128, 256, 64), (200, 72, 136), (256, 512, 1024), (300, 40, 8), (64, 1000, 96), (384, 264, 520),
               (1280, 1000, 192), (3072, 1000, 128), (2000, 8192, 256)]


def _check_y(Y, Y_ref, B, out_dt, rel):
    yb = bits_of(Y)
    ok = oracle.gemm.within_bound(yb, Y_ref, B, out_dt, rel)
    if not ok.all():
        bad = np.argwhere(~ok)
        i, j = bad[0]
        y = oracle.codecs.decode(yb[i, j], out_dt)
        r = oracle.codecs.decode(Y_ref[i, j], out_dt)
        raise AssertionError(f"{(~ok).sum()} of {ok.size} outside the bound; first at {i},{j}: "
                             f"gpu {y} ref {r} bound {B[i, j] * rel}")


@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3"])
@pytest.mark.parametrize("shape", GEMM_SHAPES)
def test_sp24_gemm_within_bound(dt, shape):
    ss = lib()
    M, N, K = shape
    W = rand_bits(200 + M, (M, K), dt, 0.5)
    X = rand_bits(300 + N, (K, N), dt, 1.0)
    out_dt = "bf16" if dt == "e4m3" else dt
    alpha = 0.75 if dt == "e4m3" else 1.0
    f = ss.sp24_prune_compress(dev_tensor(W, dt), canonical_meta=False)
    Y, buf = guarded_output(M, N, torch.bfloat16 if out_dt == "bf16" else torch.float16)
    ss.sp24_gemm(f, dev_padded(X, dt), alpha=alpha, out=Y)
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    v_ref, m_ref = oracle.sp24.compress(W, dt)
    Y_ref = oracle.gemm.gemm_sp24(v_ref, m_ref, K, X, dt, out_dt, alpha)
    B = oracle.gemm.bound(oracle.sp24.decompress(v_ref, m_ref, K), X, dt, alpha)
    _check_y(Y, Y_ref, B, out_dt, REL[dt])
    assert canary_intact(buf, M, N)


@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3"])
@pytest.mark.parametrize("shape", GEMM_SHAPES)
def test_dense_gemm_within_bound(dt, shape):
    ss = lib()
    M, N, K = shape
    W = rand_bits(400 + M, (M, K), dt, 0.5)
    X = rand_bits(500 + N, (K, N), dt, 1.0)
    out_dt = "bf16" if dt == "e4m3" else dt
    Y, buf = guarded_output(M, N, torch.bfloat16 if out_dt == "bf16" else torch.float16)
    ss.dense_gemm(dev_padded(W, dt), dev_padded(X, dt), alpha=1.0, out=Y)
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    Y_ref = oracle.gemm.gemm_dense(W, X, dt, out_dt)
    B = oracle.gemm.bound(W, X, dt)
    _check_y(Y, Y_ref, B, out_dt, REL[dt])
    assert canary_intact(buf, M, N)


def test_sp24_gemm_identity_is_exact():
    """X = I gives Y = the pruned W exactly (each output is a single product)."""
    ss = lib()
    M, K = 256, 256
    W = rand_bits(9, (M, K), "bf16", 1.0)
    X = oracle.codecs.encode(np.eye(K), "bf16")
    f = ss.sp24_prune_compress(dev_tensor(W, "bf16"))
    Y = ss.sp24_gemm(f, dev_tensor(X, "bf16"))
    assert np.array_equal(bits_of(Y), oracle.sp24.prune(W, "bf16"))


def test_k_zero_and_empty():
    ss = lib()
    X = torch.zeros((0, 16), dtype=torch.bfloat16, device="cuda")
    Y = torch.full((8, 16), 3.0, dtype=torch.bfloat16, device="cuda")
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    ss.sp24_gemm(ss.Sp24(ss.BF16, 8, 0, z, None, z), X, out=Y)
    assert (Y == 0).all()


def test_two_calls_in_a_row_agree():
    ss = lib()
    M, N, K = 256, 256, 512
    W = rand_bits(11, (M, K), "f16")
    X = rand_bits(12, (K, N), "f16")
    f = ss.sp24_prune_compress(dev_tensor(W, "f16"))
    Xd = dev_tensor(X, "f16")
    a = ss.sp24_gemm(f, Xd)
    b = ss.sp24_gemm(f, Xd)
    assert torch.equal(a, b)


def test_bounded_wait_reports_timeout_without_fault():
    """Failure detection on the device: a wait that nothing completes gives up
    after its limit, the kernel returns, the host reads SSDNN_ERR_TIMEOUT from
    the error word, and the context keeps working afterwards."""
    ss = lib()
    assert ss.check_device_error() == 0
    ss.selftest_wait_timeout(2000)
    assert ss.check_device_error() == 4          # SSDNN_ERR_TIMEOUT
    assert ss.check_device_error() == 0          # the word was cleared
    # the context is still usable: a GEMM right after runs and is exact
    M, K = 128, 128
    W = rand_bits(13, (M, K), "bf16", 1.0)
    X = oracle.codecs.encode(np.eye(K), "bf16")
    f = ss.sp24_prune_compress(dev_tensor(W, "bf16"))
    Y = ss.sp24_gemm(f, dev_tensor(X, "bf16"))
    assert np.array_equal(bits_of(Y), oracle.sp24.prune(W, "bf16"))
    assert ss.check_device_error() == 0


@pytest.mark.parametrize("dt", ["bf16", "e4m3"])
@pytest.mark.parametrize("sparse", [False, True])
def test_mma_rate_microbenchmark_runs_clean(dt, sparse):
    """The on-chip tensor-core rate kernel completes on every SM without a device
    error, for each instruction shape the bench measures."""
    ss = lib()
    for n in (128, 192, 256):
        ss.mma_rate(ss.BF16 if dt == "bf16" else ss.E4M3, sparse, n, 64)
    ss.mma_rate_pair(ss.BF16 if dt == "bf16" else ss.E4M3, sparse, 64)
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0


# Every tile variant, forced through the variant entry points (MT * 1000 + BN; 9000 + BN
# for an SM pair: two CTAs of a cluster run M = 256 MMAs, each holding 128 rows of
# W and half of the X panel), on a shape with ragged M (the odd CTA of the last
# pair has no rows), ragged N and a partial last K stage, and on a multi-wave shape.
FORCED_SHAPES = [(300, 264, 520), (2000, 8192, 256)]


def _forced_tiles(dt, sparse):
    """Every tile variant the operand type has (sp24_gemm_variant / dense_gemm_variant)."""
    tiles = [1128, 1256, 9256] + ([1064] if dt != "e4m3" else [])
    if sparse:
        tiles += [2192, 19256, 11128] + ([11064] if dt != "e4m3" else [])
    return tiles + ([] if sparse else [2256])


@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3"])
@pytest.mark.parametrize("shape", FORCED_SHAPES)
@pytest.mark.parametrize("sparse", [True, False])
def test_forced_tiles_within_bound(dt, shape, sparse):
    ss = lib()
    M, N, K = shape
    W = rand_bits(700 + M, (M, K), dt, 0.5)
    X = rand_bits(710 + N, (K, N), dt, 1.0)
    out_dt = "bf16" if dt == "e4m3" else dt
    alpha = 0.75 if dt == "e4m3" else 1.0
    if sparse:
        v_ref, m_ref = oracle.sp24.compress(W, dt)
        Y_ref = oracle.gemm.gemm_sp24(v_ref, m_ref, K, X, dt, out_dt, alpha)
        B = oracle.gemm.bound(oracle.sp24.decompress(v_ref, m_ref, K), X, dt, alpha)
        f = ss.sp24_prune_compress(dev_tensor(W, dt), canonical_meta=False)
    else:
        Y_ref = oracle.gemm.gemm_dense(W, X, dt, out_dt, alpha)
        B = oracle.gemm.bound(W, X, dt, alpha)
    Xd = dev_padded(X, dt)
    for tile in _forced_tiles(dt, sparse):
        # 19256: SM-pair stages of two 128-byte K steps
        Y, buf = guarded_output(M, N, torch.bfloat16 if out_dt == "bf16" else torch.float16)
        if sparse:
            ss.sp24_gemm(f, Xd, alpha=alpha, out=Y, variant=tile)
        else:
            ss.dense_gemm(dev_padded(W, dt), Xd, alpha=alpha, out=Y, variant=tile)
        torch.cuda.synchronize()
        assert ss.check_device_error() == 0, tile
        _check_y(Y, Y_ref, B, out_dt, REL[dt])
        assert canary_intact(buf, M, N), tile


@pytest.mark.parametrize("dt", ["bf16", "e4m3"])
@pytest.mark.parametrize("shape", [(1000, 264, 512), (4096, 4104, 256)])
def test_sp24_gemm_host_direct_output(dt, shape):
    """Y_dev None: the epilogue stores straight into page-locked host memory. The
    result is bit-identical to the device output of the same shape (same tiles:
    single-CTA tiles for the small shape, SM-pair tiles for the large one), and
    nothing outside the M x N view of the pinned buffer is written."""
    ss = lib()
    M, N, K = shape
    W = rand_bits(811, (M, K), dt, 0.5)
    X = rand_bits(812, (K, N), dt, 1.0)
    f = ss.sp24_prune_compress(dev_tensor(W, dt), canonical_meta=False)
    Xd = dev_padded(X, dt)
    ld = Xd.stride(0)                       # rows padded to 16 bytes, as the GEMM requires
    X_host = torch.empty((K, ld), dtype=Xd.dtype).pin_memory()
    X_host.copy_(Xd.as_strided((K, ld), (ld, 1)))
    X_host = X_host[:, :N]
    X_dev = torch.empty((K, ld), dtype=Xd.dtype, device="cuda")[:, :N]
    out = torch.bfloat16
    Y_dev = torch.empty((M, N), dtype=out, device="cuda")
    ss.sp24_gemm(f, Xd, alpha=0.5, out=Y_dev)
    buf = torch.empty((M + 2, N + 8), dtype=out).pin_memory()
    buf.view(torch.uint8).fill_(CANARY)
    Y_host = buf[:M, :N]
    ss.sp24_gemm_host(f, X_host, Y_host, X_dev, None, alpha=0.5)
    torch.cuda.current_stream().synchronize()
    assert ss.check_device_error() == 0
    assert np.array_equal(bits_of(Y_host), bits_of(Y_dev))
    b = buf.view(torch.uint8).numpy().reshape(M + 2, -1)
    assert (b[:M, 2 * N:] == CANARY).all() and (b[M:] == CANARY).all()
    v_ref, m_ref = oracle.sp24.compress(W, dt)
    Y_ref = oracle.gemm.gemm_sp24(v_ref, m_ref, K, X, dt, "bf16", 0.5)
    B = oracle.gemm.bound(oracle.sp24.decompress(v_ref, m_ref, K), X, dt, 0.5)
    _check_y(Y_host, Y_ref, B, "bf16", REL[dt])


def test_host_memory_operands_refused():
    """Pageable host memory as the direct output, or host memory as an input of the
    device GEMM, is refused on the host before anything is launched."""
    ss = lib()
    M, N, K = 256, 128, 256
    W = rand_bits(821, (M, K), "bf16", 0.5)
    X = rand_bits(822, (K, N), "bf16", 1.0)
    f = ss.sp24_prune_compress(dev_tensor(W, "bf16"), canonical_meta=False)
    Xd = dev_tensor(X, "bf16")
    X_host = Xd.cpu().pin_memory()
    with pytest.raises(ss.SsdnnError) as e:
        ss.sp24_gemm_host(f, X_host, torch.empty((M, N), dtype=torch.bfloat16), torch.empty_like(Xd), None)
    assert e.value.status == 1
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = ss.lib.sp24_gemm(ss.BF16, ss.BF16, M, N, K, f.values.data_ptr(), f.meta_hw.data_ptr(), X_host.data_ptr(),
                          N, Y.data_ptr(), N, 1.0, torch.cuda.current_stream().cuda_stream)
    assert st == 1
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0


@pytest.mark.parametrize("copy_stream", [False, True])
@pytest.mark.parametrize("rows_per_block", [0, 256])
def test_sp24_gemm_host_buffers(copy_stream, rows_per_block):
    """The host-buffer form: X copied in from pinned memory, Y computed in row
    blocks and copied out (overlapped on a second stream), against the oracle."""
    ss = lib()
    M, N, K, dt = 1000, 264, 520, "bf16"
    W = rand_bits(801, (M, K), dt, 0.5)
    X = rand_bits(802, (K, N), dt, 1.0)
    f = ss.sp24_prune_compress(dev_tensor(W, dt), canonical_meta=False)
    X_host = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).pin_memory()
    Y_host = torch.full((M, N), 7.0, dtype=torch.bfloat16).pin_memory()
    X_dev = torch.empty((K, N), dtype=torch.bfloat16, device="cuda")
    Y_dev = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    cs = torch.cuda.Stream() if copy_stream else None
    ss.sp24_gemm_host(f, X_host, Y_host, X_dev, Y_dev, rows_per_block=rows_per_block, copy_stream=cs)
    torch.cuda.current_stream().synchronize()
    assert ss.check_device_error() == 0
    v_ref, m_ref = oracle.sp24.compress(W, dt)
    Y_ref = oracle.gemm.gemm_sp24(v_ref, m_ref, K, X, dt, dt)
    B = oracle.gemm.bound(oracle.sp24.decompress(v_ref, m_ref, K), X, dt)
    _check_y(Y_host, Y_ref, B, dt, REL[dt])


@pytest.mark.parametrize("dt", ["bf16", "e4m3"])
def test_compress_into_existing_result_matches_fresh(dt):
    """out= overwrites an earlier 2:4 result in place: compressing a second weight into
    the first weight's buffers gives exactly what a fresh call on it gives; a result of
    another shape is refused before any device work."""
    ss = lib()
    M, K = 200, 520
    W1 = dev_tensor(rand_bits(911, (M, K), dt, 0.5), dt)
    W2 = dev_tensor(rand_bits(912, (M, K), dt, 0.5), dt)
    form = ss.sp24_prune_compress(W1)
    fresh = ss.sp24_prune_compress(W2)
    again = ss.sp24_prune_compress(W2, out=form)
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    assert again is form
    for name in ("values", "meta", "meta_hw"):
        a, b = getattr(again, name), getattr(fresh, name)
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), name
    with pytest.raises(ValueError):
        ss.sp24_prune_compress(dev_tensor(rand_bits(913, (M, K + 32), dt, 0.5), dt), out=form)
