"""The C-ABI library builds, loads and exports every function include/ssdnn.h
declares; host-only entry points (sizes, status strings, argument checks that
fail before any CUDA call) behave as documented. No GPU needed."""
import ctypes as C
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssdnn.h")


@pytest.fixture(scope="module")
def ssdnn():
    from structured_sparse_dnn_gb300 import build
    build.build()
    from structured_sparse_dnn_gb300 import ssdnn as mod
    return mod


class Buffers:
    """Operand addresses for calls that must be refused on the host. With a GPU
    present they are real device allocations (64 KB each, 256-byte aligned, large
    enough for every small shape used here), so that a refusal that regressed
    would launch on valid memory; without one they are distinct dummy addresses,
    which nothing can dereference because no kernel can run."""

    def __init__(self):
        import torch
        self.cuda = torch.cuda.is_available()
        self._keep = []
        self._next = 1 << 20

    def dev(self, nbytes: int = 1 << 16) -> int:
        if self.cuda:
            import torch
            t = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device="cuda")
            self._keep.append(t)
            return t.data_ptr()
        self._next += max(nbytes, 256) + 4096
        return self._next

    def host(self, nbytes: int = 1 << 16) -> int:
        a = np.zeros(max(nbytes, 256) + 256, dtype=np.uint8)
        self._keep.append(a)
        p = a.ctypes.data
        return p + (-p % 256)


@pytest.fixture
def bufs():
    return Buffers()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_api():
    names = _declared()
    for n in ("sp24_prune_compress", "sp24_gemm", "tw_prune_compress", "tvw_gemm", "dense_gemm",
              "sp24_sizes", "tw_sizes", "ssdnn_status_str", "ssdnn_check_device_error", "ssdnn_version"):
        assert n in names


def test_every_declared_symbol_is_exported(ssdnn):
    lib = C.CDLL(os.path.join(ROOT, "structured_sparse_dnn_gb300", "lib", "libssdnn.so"))
    for n in _declared():
        assert hasattr(lib, n), n
    assert set(ssdnn.EXPORTED) <= set(_declared())


def test_status_strings_and_version(ssdnn):
    assert ssdnn.status_str(0) == "ok"
    assert "unsupported" in ssdnn.status_str(2)
    assert ssdnn.status_str(99) == "unknown status"
    assert ssdnn.lib.ssdnn_version() >= 100


def test_sp24_sizes(ssdnn):
    assert ssdnn.sp24_sizes(ssdnn.BF16, 256, 256) == (256 * 128 * 2, 256 * 32, 2 * 4 * 2048)
    assert ssdnn.sp24_sizes(ssdnn.E4M3, 14336, 4096) == (14336 * 2048, 14336 * 512, 112 * 32 * 2048)
    v, m, h = ssdnn.sp24_sizes(ssdnn.F16, 5, 36)           # Kp = 64
    assert (v, m, h) == (5 * 32 * 2, 5 * 8, 1 * 1 * 2048)
    with pytest.raises(ssdnn.SsdnnError) as e:
        ssdnn.sp24_sizes(ssdnn.F16, 4, 6)
    assert e.value.status == 2
    with pytest.raises(ssdnn.SsdnnError) as e:
        ssdnn.sp24_sizes(7, 4, 8)
    assert e.value.status == 1


def test_tw_sizes_match_layout(ssdnn):
    keep = np.array([832, 0, 64, 100], dtype=np.int32)
    s = ssdnn.tw_sizes(ssdnn.BF16, False, 500, 1024, keep)
    R = [832, 0, 64, 128]
    assert s["packed_bytes"] == 128 * sum(R) * 2
    assert s["indices_count"] == keep.sum()
    assert s["workspace_bytes"] == 4 * 1024 * 4
    assert s["meta_bytes"] == 0 and s["meta_hw_bytes"] == 0
    with pytest.raises(ssdnn.SsdnnError):                    # TVW needs L % 4 == 0
        ssdnn.tw_sizes(ssdnn.BF16, True, 500, 1024, np.array([832, 0, 64, 102], dtype=np.int32))
    keep4 = np.array([832, 0, 64, 100], dtype=np.int32)
    s = ssdnn.tw_sizes(ssdnn.BF16, True, 500, 1024, keep4)
    assert s["packed_bytes"] == 64 * sum(R) * 2
    assert s["meta_bytes"] == 16 * sum(R)
    assert s["meta_hw_bytes"] == 2048 * (13 + 0 + 1 + 2)
    with pytest.raises(ssdnn.SsdnnError):                    # L > K
        ssdnn.tw_sizes(ssdnn.BF16, False, 128, 64, np.array([65], dtype=np.int32))
    with pytest.raises(ssdnn.SsdnnError) as e:               # e4m3 tile-wise is not implemented
        ssdnn.tw_sizes(ssdnn.E4M3, False, 128, 64, np.array([64], dtype=np.int32))
    assert e.value.status == 2


def test_argument_errors_before_any_device_work(ssdnn, bufs):
    lib = ssdnn.lib
    d = [bufs.dev() for _ in range(6)]
    # bad dtype, negative sizes, K % 4 != 0: rejected on the host
    assert lib.sp24_prune_compress(9, None, 4, 8, 8, None, None, None, None) == 1
    assert lib.sp24_prune_compress(0, None, -1, 8, 8, None, None, None, None) == 1
    assert lib.sp24_prune_compress(0, None, 4, 6, 6, None, None, None, None) == 2
    assert lib.sp24_gemm(0, 2, 4, 4, 8, None, None, None, 4, None, 4, 1.0, None) == 2   # out e4m3
    assert lib.sp24_gemm(0, 0, 4, 4, 8, None, None, None, 4, None, 4, 1.0, None) == 1   # null Y
    assert lib.dense_gemm(0, 0, 4, 8, 8, d[0], 8, d[1], 4, d[2], 8, 1.0, None) == 1     # ldx < N
    assert lib.tvw_gemm(2, 0, 4, 4, 8, None, None, None, None, None, None, None, 4, None, 4, None) == 2
    # empty problems are valid no-ops
    assert lib.sp24_gemm(0, 0, 0, 4, 8, None, None, None, 4, None, 4, 1.0, None) == 0
    assert lib.sp24_prune_compress(0, None, 0, 8, 8, None, None, None, None) == 0
    # the wait-timeout self-test takes a limit of 1 us .. 1 s
    assert lib.ssdnn_selftest_wait_timeout(0, None) == 1
    assert lib.ssdnn_selftest_wait_timeout(1000001, None) == 1
    # the tensor-core rate microbenchmark validates its arguments on the host
    assert lib.ssdnn_mma_rate(7, 0, 128, 16, None) == 1
    assert lib.ssdnn_mma_rate(1, 2, 128, 16, None) == 1
    assert lib.ssdnn_mma_rate(1, 0, 128, 0, None) == 1
    assert lib.ssdnn_mma_rate_pair(7, 0, 16, None) == 1
    assert lib.ssdnn_mma_rate_pair(1, 2, 16, None) == 1
    assert lib.ssdnn_mma_rate_pair(1, 0, 0, None) == 1
    assert lib.ssdnn_mma_rate_pair(2, 1, (1 << 18) + 1, None) == 1
    assert lib.ssdnn_mma_rate(1, 0, 96, 16, None) == 2
    # fused epilogue: unknown activation, non-finite scale, misaligned bias, e4m3 pitch
    ep = ssdnn.Epilogue(None, 5, 1.0)
    assert lib.dense_gemm_ep(0, 0, 4, 8, 8, d[0], 8, d[1], 8, d[2], 8, 1.0, C.byref(ep), None) == 1
    ep = ssdnn.Epilogue(None, 1, float("inf"))
    assert lib.sp24_gemm_ep(0, 0, 4, 8, 8, d[0], d[3], d[1], 8, d[2], 8, 1.0, C.byref(ep), None) == 1
    ep = ssdnn.Epilogue(d[4] + 2, 1, 1.0)                                                   # bias not 4-byte aligned
    assert lib.sp24_gemm_ep(0, 0, 4, 8, 8, d[0], d[3], d[1], 8, d[2], 8, 1.0, C.byref(ep), None) == 2
    assert lib.sp24_gemm_ep(0, 2, 4, 8, 8, d[0], d[3], d[1], 8, d[2], 8, 1.0, None, None) == 2  # e4m3 row pitch 8 B
    assert lib.sp24_gemm(0, 2, 4, 16, 8, d[0], d[3], d[1], 16, d[2], 16, 1.0, None) == 2      # plain call: no e4m3 out
    # explicit tile variants: unknown values, and variants the operand type lacks
    assert lib.sp24_gemm_variant(1, 1, 4, 8, 8, d[0], d[3], d[1], 8, d[2], 8, 1.0, None, 1234, None) == 2
    assert lib.sp24_gemm_variant(2, 1, 4, 16, 8, d[0], d[3], d[1], 16, d[2], 16, 1.0, None, 1064, None) == 2
    assert lib.dense_gemm_variant(1, 1, 4, 8, 8, d[0], 8, d[1], 8, d[2], 8, 1.0, None, 19256, None) == 2
    assert lib.dense_gemm_variant(1, 1, 4, 8, 8, d[0], 8, d[1], 8, d[2], 8, 1.0, None, 2192, None) == 2
    # the host-buffer GEMM: block height a multiple of 128, host buffers required
    hx, hy = bufs.host(), bufs.host()
    assert lib.sp24_gemm_host(1, 1, 256, 8, 64, d[0], d[3], hx, 8, hy, 8, 1.0, d[1], d[2], 100, None, None) == 1
    assert lib.sp24_gemm_host(1, 1, 256, 8, 64, d[0], d[3], None, 8, hy, 8, 1.0, d[1], d[2], 128, None, None) == 1
    # block-wise: K % 64, kept blocks within range, e4m3 unsupported
    k = np.array([1, 2], dtype=np.int32)
    assert lib.bw_sizes(1, 256, 100, k.ctypes.data_as(C.POINTER(C.c_int32)), None, None, None) == 2
    k3 = np.array([5, 0], dtype=np.int32)
    assert lib.bw_sizes(1, 256, 256, k3.ctypes.data_as(C.POINTER(C.c_int32)), None, None, None) == 1
    assert lib.bw_sizes(2, 256, 256, k.ctypes.data_as(C.POINTER(C.c_int32)), None, None, None) == 2


def test_bw_sizes_match_layout(ssdnn):
    s = ssdnn.bw_sizes(ssdnn.BF16, 300, 256, np.array([1, 4, 0], dtype=np.int32))
    assert s["packed_bytes"] == 128 * 64 * 5 * 2
    assert s["indices_count"] == 5
    assert s["workspace_bytes"] >= 3 * 256 * 4 + 3 * 4 * 4 + 4 * 4 + 64 * 5 * 4
    # element-wise: k > K invalid, e4m3 unsupported
    assert ssdnn.lib.ew_sizes(1, 8, 16, 17, None, None, None) == 1
    assert ssdnn.lib.ew_sizes(2, 8, 16, 4, None, None, None) == 2


def test_conv_argument_checks(ssdnn, bufs):
    lib = ssdnn.lib
    d = [bufs.dev() for _ in range(4)]
    # C_in not a multiple of 64, image wider than 224, e4m3
    assert lib.sp24_conv3x3(1, 1, 128, 32, 1, 8, 8, d[0], d[1], d[2], d[3], 64, 1.0, None) == 2
    assert lib.sp24_conv3x3(1, 1, 128, 64, 1, 8, 256, d[0], d[1], d[2], d[3], 2048, 1.0, None) == 2
    assert lib.dense_conv3x3(2, 1, 128, 64, 1, 8, 8, d[0], 576, d[2], d[3], 64, 1.0, None) == 2


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="host-only: the refused problems exceed the fixed scratch, so a regressed "
                           "refusal must never reach a GPU")
def test_noalloc_refusals_host_only(ssdnn):
    """tw_prune_compress_noalloc refuses, before any CUDA call, problems beyond its
    fixed limits: more than SSDNN_NOALLOC_MAX_TILES tiles (the kept counts travel
    as a fixed-size kernel parameter), and more than SSDNN_NOALLOC_MAX_SCORES
    scores. Dummy addresses only: nothing here may run on a device."""
    lib = ssdnn.lib
    max_tiles, max_scores = 2048, 1 << 21
    hdr = open(HEADER).read()
    assert f"#define SSDNN_NOALLOC_MAX_TILES {max_tiles}" in hdr
    assert "#define SSDNN_NOALLOC_MAX_SCORES (1 << 21)" in hdr
    P = C.POINTER(C.c_int32)
    # nt = max_tiles + 1 tiles, K small (nt * K well inside the score scratch)
    nt = max_tiles + 1
    keep = np.full(nt, 4, dtype=np.int32)
    st = lib.tw_prune_compress_noalloc(1, 0, 1 << 20, 128 * nt, 16, 16, keep.ctypes.data_as(P),
                                       2 << 20, 3 << 20, 4 << 20, 5 << 20, None, None, None)
    assert st == 2
    # exactly max_tiles tiles passes the tile limit; it is then refused only for a null W
    keep = np.full(max_tiles, 4, dtype=np.int32)
    st = lib.tw_prune_compress_noalloc(1, 0, None, 128 * max_tiles, 16, 16, keep.ctypes.data_as(P),
                                       2 << 20, 3 << 20, 4 << 20, 5 << 20, None, None, None)
    assert st == 1
    # two tiles whose scores exceed the scratch by one tile row
    K = max_scores // 2 + 64
    keep = np.array([64, 64], dtype=np.int32)
    st = lib.tw_prune_compress_noalloc(1, 0, 1 << 20, 256, K, K, keep.ctypes.data_as(P),
                                       2 << 20, 3 << 20, 4 << 20, 5 << 20, None, None, None)
    assert st == 2


def test_out_refusals_come_before_any_library_call(ssdnn, monkeypatch):
    """The prune helpers' out= forms refuse a result made for another shape, type,
    kept counts or k (and a missing workspace) on the host, before any call into the
    library: the library is replaced by an object that fails on any attribute access."""
    import torch

    class NoLib:
        def __getattr__(self, name):
            raise AssertionError(f"library called: {name}")

    monkeypatch.setattr(ssdnn, "lib", NoLib())
    t = torch.zeros(4, dtype=torch.uint8)
    W = torch.zeros(256, 512, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ssdnn.sp24_prune_compress(W, out=ssdnn.Sp24(ssdnn.BF16, 256, 544, t, None, t))
    with pytest.raises(ValueError):
        ssdnn.sp24_prune_compress(W, out=ssdnn.Sp24(ssdnn.F16, 256, 512, t, None, t))
    keep = np.array([128, 64], dtype=np.int32)
    tw = ssdnn.TileWise(ssdnn.BF16, True, 256, 512, keep, t, t, t, t, t, t)
    with pytest.raises(ValueError):
        ssdnn.tw_prune_compress(W, np.array([128, 68], dtype=np.int32), True, t, out=tw)
    with pytest.raises(ValueError):
        ssdnn.tw_prune_compress(W, keep, False, t, out=tw)
    with pytest.raises(ValueError):
        ssdnn.tw_prune_compress(W, keep, True, None, out=tw)
    kb = np.array([2, 1], dtype=np.int32)
    bw = ssdnn.BlockWise(ssdnn.BF16, 256, 512, kb, t, t, t, t)
    with pytest.raises(ValueError):
        ssdnn.bw_prune_compress(W, np.array([2, 2], dtype=np.int32), t, out=bw)
    with pytest.raises(ValueError):
        ssdnn.bw_prune_compress(W, kb, None, out=bw)
    ew = ssdnn.ElementWise(ssdnn.BF16, 256, 512, 51, t, t, t, t, t)
    with pytest.raises(ValueError):
        ssdnn.ew_prune_compress(W, 52, t, out=ew)
    with pytest.raises(ValueError):
        ssdnn.ew_prune_compress(W, 51, None, out=ew)
