"""Thin ctypes binding of libssdnn.so (include/ssdnn.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels. Functions carry the C names; the tensor-level helpers allocate the
outputs with torch (the library itself allocates nothing) and pass raw device
pointers plus the current CUDA stream. There is no CPU fallback: importing this
module raises if the library cannot be loaded.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

import numpy as np
import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libssdnn.so")

if not os.path.exists(_LIB_PATH):
    raise ImportError(f"libssdnn.so not built ({_LIB_PATH}); run structured_sparse_dnn_gb300.build.build()")
lib = C.CDLL(_LIB_PATH)

F16, BF16, E4M3 = 0, 1, 2
_DT = {torch.float16: F16, torch.bfloat16: BF16, torch.float8_e4m3fn: E4M3}
_TORCH = {F16: torch.float16, BF16: torch.bfloat16, E4M3: torch.float8_e4m3fn}

_i64, _ptr, _sz, _i32p = C.c_int64, C.c_void_p, C.c_size_t, C.POINTER(C.c_int32)

ACT = {"none": 0, "relu": 1, "gelu": 2}


class Epilogue(C.Structure):
    """ssdnn_epilogue: per-row fp32 bias (device pointer or None), activation, output scale."""
    _fields_ = [("bias", C.c_void_p), ("act", C.c_int), ("y_scale", C.c_float)]


_epp = C.POINTER(Epilogue)
_SIGS = {
    "ssdnn_status_str": ([C.c_int], C.c_char_p),
    "ssdnn_version": ([], C.c_int),
    "ssdnn_check_device_error": ([_ptr], C.c_int),
    "ssdnn_selftest_wait_timeout": ([C.c_uint32, _ptr], C.c_int),
    "ssdnn_mma_rate": ([C.c_int, C.c_int, C.c_int, C.c_int, _ptr], C.c_int),
    "ssdnn_mma_rate_pair": ([C.c_int, C.c_int, C.c_int, _ptr], C.c_int),
    "sp24_sizes": ([C.c_int, _i64, _i64, C.POINTER(_sz), C.POINTER(_sz), C.POINTER(_sz)], C.c_int),
    "sp24_prune_compress": ([C.c_int, _ptr, _i64, _i64, _i64, _ptr, _ptr, _ptr, _ptr], C.c_int),
    "sp24_gemm": ([C.c_int, C.c_int, _i64, _i64, _i64, _ptr, _ptr, _ptr, _i64, _ptr, _i64, C.c_float, _ptr],
                  C.c_int),
    "dense_gemm": ([C.c_int, C.c_int, _i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, C.c_float, _ptr],
                   C.c_int),
    "sp24_gemm_ep": ([C.c_int, C.c_int, _i64, _i64, _i64, _ptr, _ptr, _ptr, _i64, _ptr, _i64, C.c_float, _epp,
                      _ptr], C.c_int),
    "dense_gemm_ep": ([C.c_int, C.c_int, _i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, C.c_float, _epp,
                       _ptr], C.c_int),
    "tvw_gemm_ep": ([C.c_int, C.c_int, C.c_int, _i64, _i64, _i64, _i32p, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _i64,
                     _ptr, _i64, C.c_float, _epp, _ptr], C.c_int),
    "sp24_gemm_host": ([C.c_int, C.c_int, _i64, _i64, _i64, _ptr, _ptr, _ptr, _i64, _ptr, _i64, C.c_float, _ptr,
                        _ptr, _i64, _ptr, _ptr], C.c_int),
    "bw_sizes": ([C.c_int, _i64, _i64, _i32p, C.POINTER(_sz), C.POINTER(_sz), C.POINTER(_sz)], C.c_int),
    "bw_prune_compress": ([C.c_int, _ptr, _i64, _i64, _i64, _i32p, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr], C.c_int),
    "bw_gemm": ([C.c_int, _i64, _i64, _i64, _i32p, _ptr, _ptr, _ptr, _ptr, _ptr, _i64, _ptr, _i64, _ptr], C.c_int),
    "bw_gemm_ep": ([C.c_int, C.c_int, _i64, _i64, _i64, _i32p, _ptr, _ptr, _ptr, _ptr, _ptr, _i64, _ptr, _i64,
                    C.c_float, _epp, _ptr], C.c_int),
    "ew_sizes": ([C.c_int, _i64, _i64, _i64, C.POINTER(_sz), C.POINTER(_sz), C.POINTER(_sz)], C.c_int),
    "ew_prune_compress": ([C.c_int, _ptr, _i64, _i64, _i64, _i64, _ptr, _ptr, _ptr, _ptr, _ptr], C.c_int),
    "ew_spmm": ([C.c_int, _i64, _i64, _i64, _ptr, _ptr, _ptr, _ptr, _i64, _ptr, _i64, _ptr], C.c_int),
    "sp24_conv3x3": ([C.c_int, C.c_int, _i64, _i64, _i64, _i64, _i64, _ptr, _ptr, _ptr, _ptr, _i64, C.c_float,
                      _ptr], C.c_int),
    "dense_conv3x3": ([C.c_int, C.c_int, _i64, _i64, _i64, _i64, _i64, _ptr, _i64, _ptr, _ptr, _i64, C.c_float,
                       _ptr], C.c_int),
    "tw_conv3x3": ([C.c_int, C.c_int, _i64, _i64, _i64, _i64, _i64, _i32p, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _i64,
                    C.c_float, _ptr], C.c_int),
    "tw_sizes": ([C.c_int, C.c_int, _i64, _i64, _i32p, C.POINTER(_sz), C.POINTER(_sz), C.POINTER(_sz),
                  C.POINTER(_sz), C.POINTER(_sz)], C.c_int),
    "tw_prune_compress": ([C.c_int, C.c_int, _ptr, _i64, _i64, _i64, _i32p, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr,
                           _ptr, _ptr], C.c_int),
    "tvw_gemm": ([C.c_int, C.c_int, _i64, _i64, _i64, _i32p, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _i64, _ptr,
                  _i64, _ptr], C.c_int),
    "sp24_gemm_variant": ([C.c_int, C.c_int, _i64, _i64, _i64, _ptr, _ptr, _ptr, _i64, _ptr, _i64, C.c_float, _epp,
                           C.c_int, _ptr], C.c_int),
    "dense_gemm_variant": ([C.c_int, C.c_int, _i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, C.c_float, _epp,
                            C.c_int, _ptr], C.c_int),
    "tw_prune_compress_noalloc": ([C.c_int, C.c_int, _ptr, _i64, _i64, _i64, _i32p, _ptr, _ptr, _ptr, _ptr, _ptr,
                                   _ptr, _ptr], C.c_int),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = _res

EXPORTED = tuple(_SIGS)


class SsdnnError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {lib.ssdnn_status_str(status).decode()} (status {status})")
        self.status = status


def _check(status: int, where: str):
    if status != 0:
        raise SsdnnError(status, where)


def _stream(dev) -> int:
    return torch.cuda.current_stream(dev).cuda_stream


def _p(t: torch.Tensor | None):
    return None if t is None else t.data_ptr()


def _keep_arr(keep) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(keep, dtype=np.int32))


def _kp(keep: np.ndarray):
    return keep.ctypes.data_as(_i32p)


def status_str(status: int) -> str:
    return lib.ssdnn_status_str(status).decode()


def check_device_error(stream: int | None = None) -> int:
    """Synchronises the stream and returns (and clears) the device error status."""
    return lib.ssdnn_check_device_error(stream if stream is not None else _stream(None))


def mma_rate(dt: int, sparse: bool, n: int, iters: int, stream: int | None = None) -> None:
    """Launches the tensor-core rate microbenchmark (one CTA per SM, `iters`
    steps of 2 * 128 * n * (128 / elem bytes) dense-equivalent flops each)."""
    _check(lib.ssdnn_mma_rate(dt, int(sparse), n, iters, stream if stream is not None else _stream(None)),
           "ssdnn_mma_rate")


def mma_rate_pair(dt: int, sparse: bool, iters: int, stream: int | None = None) -> None:
    """The microbenchmark on SM pairs (M = 256, N = 256 per pair; `iters` steps of
    2 * 256 * 256 * (128 / elem bytes) dense-equivalent flops per pair)."""
    _check(lib.ssdnn_mma_rate_pair(dt, int(sparse), iters, stream if stream is not None else _stream(None)),
           "ssdnn_mma_rate_pair")


def selftest_wait_timeout(limit_us: int = 1000, stream: int | None = None) -> None:
    """Launches the bounded-wait self-test: a wait that nothing completes gives up
    after limit_us and records a timeout; check_device_error() then reports it."""
    _check(lib.ssdnn_selftest_wait_timeout(limit_us, stream if stream is not None else _stream(None)),
           "ssdnn_selftest_wait_timeout")


# ---------------------------------------------------------------------- 2:4
def sp24_sizes(dt: int, M: int, K: int) -> tuple[int, int, int]:
    """(values, meta, meta_hw) sizes in bytes."""
    v, m, h = _sz(), _sz(), _sz()
    _check(lib.sp24_sizes(dt, M, K, C.byref(v), C.byref(m), C.byref(h)), "sp24_sizes")
    return v.value, m.value, h.value


@dataclass
class Sp24:
    """A 2:4-compressed weight on the device: the values (M x Kp/2), the canonical
    metadata (optional) and the metadata in the tensor-core operand order."""
    dt: int
    M: int
    K: int
    values: torch.Tensor
    meta: torch.Tensor | None
    meta_hw: torch.Tensor


def sp24_prune_compress(W: torch.Tensor, canonical_meta: bool = True, out: Sp24 | None = None) -> Sp24:
    """W (M x K, fp16/bf16/e4m3, CUDA) -> its 2:4-compressed form. `out`, a result of
    an earlier call with the same shape and type, is overwritten in place (no
    allocation; its canonical metadata too, if it has any)."""
    dt = _DT[W.dtype]
    M, K = W.shape
    assert W.stride(1) == 1
    if out is not None:
        if (out.dt, out.M, out.K) != (dt, M, K):
            raise ValueError("sp24_prune_compress: out was made for another weight shape or type")
        _check(lib.sp24_prune_compress(dt, _p(W), M, K, W.stride(0), _p(out.values), _p(out.meta), _p(out.meta_hw),
                                       _stream(W.device)), "sp24_prune_compress")
        return out
    vb, mb, hb = sp24_sizes(dt, M, K)
    Kp = (K + 31) // 32 * 32
    values = torch.empty((M, Kp // 2), dtype=W.dtype, device=W.device)
    meta = torch.empty((M, Kp // 8), dtype=torch.uint8, device=W.device) if canonical_meta else None
    meta_hw = torch.empty(max(16, hb), dtype=torch.uint8, device=W.device)
    _check(lib.sp24_prune_compress(dt, _p(W), M, K, W.stride(0), _p(values), _p(meta), _p(meta_hw),
                                   _stream(W.device)), "sp24_prune_compress")
    return Sp24(dt, M, K, values, meta, meta_hw[:hb])


def _epilogue(bias: torch.Tensor | None, act: str, y_scale: float, M: int):
    """The ssdnn_epilogue for these arguments, or None for the plain conversion."""
    if bias is None and act == "none" and y_scale == 1.0:
        return None
    if bias is not None:
        assert bias.dtype == torch.float32 and bias.is_cuda and bias.numel() == M and bias.is_contiguous()
    return Epilogue(None if bias is None else bias.data_ptr(), ACT[act], float(y_scale))


def sp24_gemm(form: Sp24, X: torch.Tensor, out_dtype: torch.dtype | None = None, alpha: float = 1.0,
              out: torch.Tensor | None = None, bias: torch.Tensor | None = None, act: str = "none",
              y_scale: float = 1.0, variant: int = 0):
    """Y = round(y_scale * act(alpha * decompress(form) . X + bias[:, None]))  (M x N).
    variant != 0 forces a tile variant (sp24_gemm_variant)."""
    dt = _DT[X.dtype]
    assert dt == form.dt and X.shape[0] == form.K
    N = X.shape[1]
    out_dtype = out_dtype or (torch.bfloat16 if dt == E4M3 else X.dtype)
    if out is None:
        out = torch.empty((form.M, N), dtype=out_dtype, device=X.device)
    ep = _epilogue(bias, act, y_scale, form.M)
    args = (dt, _DT[out.dtype], form.M, N, form.K, _p(form.values), _p(form.meta_hw), _p(X), X.stride(0), _p(out),
            out.stride(0), alpha)
    if variant:
        _check(lib.sp24_gemm_variant(*args, None if ep is None else C.byref(ep), variant, _stream(X.device)),
               "sp24_gemm_variant")
    elif ep is None and out.dtype != torch.float8_e4m3fn:
        _check(lib.sp24_gemm(*args, _stream(X.device)), "sp24_gemm")
    else:
        _check(lib.sp24_gemm_ep(*args, None if ep is None else C.byref(ep), _stream(X.device)), "sp24_gemm_ep")
    return out


def sp24_gemm_host(form: Sp24, X_host: torch.Tensor, Y_host: torch.Tensor, X_dev: torch.Tensor,
                   Y_dev: torch.Tensor | None, alpha: float = 1.0, rows_per_block: int = 0,
                   copy_stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Y_host = alpha * decompress(form) . X_host through the device buffers X_dev and
    Y_dev, the copies of Y overlapped with the GEMM of later row blocks when a
    copy stream is given; with Y_dev None the GEMM stores into the pinned Y_host
    itself. Enqueues only: Y_host is complete once the current stream is."""
    dt = _DT[X_host.dtype]
    assert dt == form.dt and X_host.shape == X_dev.shape and X_host.stride(0) == X_dev.stride(0)
    assert Y_dev is None or (Y_host.shape == Y_dev.shape and Y_host.stride(0) == Y_dev.stride(0))
    N = X_host.shape[1]
    cs = copy_stream.cuda_stream if copy_stream is not None else None
    _check(lib.sp24_gemm_host(dt, _DT[Y_host.dtype], form.M, N, form.K, _p(form.values), _p(form.meta_hw),
                              X_host.data_ptr(), X_host.stride(0), Y_host.data_ptr(), Y_host.stride(0), alpha,
                              _p(X_dev), None if Y_dev is None else _p(Y_dev), rows_per_block,
                              _stream(X_dev.device), cs), "sp24_gemm_host")
    return Y_host


def dense_gemm(W: torch.Tensor, X: torch.Tensor, out_dtype: torch.dtype | None = None, alpha: float = 1.0,
               out: torch.Tensor | None = None, bias: torch.Tensor | None = None, act: str = "none",
               y_scale: float = 1.0, variant: int = 0):
    """Y = round(y_scale * act(alpha * W . X + bias[:, None])) on the dense tensor cores.
    variant != 0 forces a tile variant (dense_gemm_variant)."""
    dt = _DT[W.dtype]
    M, K = W.shape
    N = X.shape[1]
    out_dtype = out_dtype or (torch.bfloat16 if dt == E4M3 else W.dtype)
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=X.device)
    ep = _epilogue(bias, act, y_scale, M)
    args = (dt, _DT[out.dtype], M, N, K, _p(W), W.stride(0), _p(X), X.stride(0), _p(out), out.stride(0), alpha)
    if variant:
        _check(lib.dense_gemm_variant(*args, None if ep is None else C.byref(ep), variant, _stream(X.device)),
               "dense_gemm_variant")
    elif ep is None and out.dtype != torch.float8_e4m3fn:
        _check(lib.dense_gemm(*args, _stream(X.device)), "dense_gemm")
    else:
        _check(lib.dense_gemm_ep(*args, None if ep is None else C.byref(ep), _stream(X.device)), "dense_gemm_ep")
    return out


# ---------------------------------------------------------------- TW / TVW
@dataclass
class TileWise:
    """A tile-wise (or tile-vector-wise) compressed weight, as laid out on the device."""
    dt: int
    tvw: bool
    M: int
    K: int
    keep: np.ndarray
    offsets: torch.Tensor
    indices: torch.Tensor
    schedule: torch.Tensor
    packed: torch.Tensor
    meta: torch.Tensor | None
    meta_hw: torch.Tensor | None


def tw_sizes(dt: int, tvw: bool, M: int, K: int, keep) -> dict:
    k = _keep_arr(keep)
    out = [_sz() for _ in range(5)]
    _check(lib.tw_sizes(dt, int(tvw), M, K, _kp(k), *[C.byref(o) for o in out]), "tw_sizes")
    return dict(zip(("packed_bytes", "indices_count", "meta_bytes", "meta_hw_bytes", "workspace_bytes"),
                    (o.value for o in out)))


def tw_prune_compress(W: torch.Tensor, keep, tvw: bool, workspace: torch.Tensor | None = None,
                      out: TileWise | None = None) -> TileWise:
    """Tile-wise (tvw=False) or tile-vector-wise prune + pack. `out`, a result of an
    earlier call with the same shape, type, pattern and kept counts, is overwritten
    in place (no allocation)."""
    dt = _DT[W.dtype]
    M, K = W.shape
    assert W.stride(1) == 1
    k = _keep_arr(keep)
    if out is not None:
        if (out.dt, out.tvw, out.M, out.K) != (dt, bool(tvw), M, K) or not np.array_equal(out.keep, k):
            raise ValueError("tw_prune_compress: out was made for another weight shape or kept counts")
        if workspace is None:
            raise ValueError("tw_prune_compress: out= needs a workspace")
        _check(lib.tw_prune_compress(dt, int(tvw), _p(W), M, K, W.stride(0), _kp(out.keep), _p(out.offsets),
                                     _p(out.indices), _p(out.schedule), _p(out.packed), _p(out.meta),
                                     _p(out.meta_hw), _p(workspace), _stream(W.device)), "tw_prune_compress")
        return out
    sz = tw_sizes(dt, tvw, M, K, k)
    dev = W.device
    nt = (M + 127) // 128
    offsets = torch.empty(nt + 1, dtype=torch.int32, device=dev)
    indices = torch.empty(max(1, sz["indices_count"]), dtype=torch.int32, device=dev)
    schedule = torch.empty(4 * max(1, nt), dtype=torch.int32, device=dev)
    packed = torch.empty(max(8, sz["packed_bytes"] // 2), dtype=W.dtype, device=dev)
    meta = torch.empty(max(16, sz["meta_bytes"]), dtype=torch.uint8, device=dev) if tvw else None
    meta_hw = torch.empty(max(16, sz["meta_hw_bytes"]), dtype=torch.uint8, device=dev) if tvw else None
    if workspace is None:
        workspace = torch.empty(max(16, sz["workspace_bytes"]), dtype=torch.uint8, device=dev)
    _check(lib.tw_prune_compress(dt, int(tvw), _p(W), M, K, W.stride(0), _kp(k), _p(offsets), _p(indices),
                                 _p(schedule), _p(packed), _p(meta), _p(meta_hw), _p(workspace), _stream(dev)),
           "tw_prune_compress")
    return TileWise(dt, tvw, M, K, k, offsets, indices[:sz["indices_count"]], schedule[:4 * nt],
                    packed[:sz["packed_bytes"] // 2],
                    None if meta is None else meta[:sz["meta_bytes"]],
                    None if meta_hw is None else meta_hw[:sz["meta_hw_bytes"]])


def tw_prune_compress_noalloc(W: torch.Tensor, keep, tvw: bool) -> TileWise:
    """tw_prune_compress without a workspace: for callers that cannot allocate
    device memory inside the call. The library keeps the score scratch in a fixed
    device array (8 MiB, shared by all calls on a device; overlapping calls race).
    The output tensors here are still allocated by this Python helper."""
    dt = _DT[W.dtype]
    M, K = W.shape
    assert W.stride(1) == 1
    k = _keep_arr(keep)
    sz = tw_sizes(dt, tvw, M, K, k)
    dev = W.device
    nt = (M + 127) // 128
    offsets = torch.empty(nt + 1, dtype=torch.int32, device=dev)
    indices = torch.empty(max(1, sz["indices_count"]), dtype=torch.int32, device=dev)
    schedule = torch.empty(4 * max(1, nt), dtype=torch.int32, device=dev)
    packed = torch.empty(max(8, sz["packed_bytes"] // 2), dtype=W.dtype, device=dev)
    meta = torch.empty(max(16, sz["meta_bytes"]), dtype=torch.uint8, device=dev) if tvw else None
    meta_hw = torch.empty(max(16, sz["meta_hw_bytes"]), dtype=torch.uint8, device=dev) if tvw else None
    _check(lib.tw_prune_compress_noalloc(dt, int(tvw), _p(W), M, K, W.stride(0), _kp(k), _p(offsets), _p(indices),
                                         _p(schedule), _p(packed), _p(meta), _p(meta_hw), _stream(dev)),
           "tw_prune_compress_noalloc")
    return TileWise(dt, tvw, M, K, k, offsets, indices[:sz["indices_count"]], schedule[:4 * nt],
                    packed[:sz["packed_bytes"] // 2],
                    None if meta is None else meta[:sz["meta_bytes"]],
                    None if meta_hw is None else meta_hw[:sz["meta_hw_bytes"]])


def tvw_gemm(form: TileWise, X: torch.Tensor, out: torch.Tensor | None = None, out_dtype: torch.dtype | None = None,
             alpha: float = 1.0, bias: torch.Tensor | None = None, act: str = "none", y_scale: float = 1.0):
    """Y = W_tw . X[idx] per tile (TW), or its 2:4 form (TVW); with the fused
    epilogue when bias / act / y_scale / alpha / an e4m3 output are given."""
    N = X.shape[1]
    if out is None:
        out = torch.empty((form.M, N), dtype=out_dtype or X.dtype, device=X.device)
    ep = _epilogue(bias, act, y_scale, form.M)
    tail = (_kp(form.keep), _p(form.offsets), _p(form.indices), _p(form.schedule), _p(form.packed),
            _p(form.meta_hw), _p(X), X.stride(0), _p(out), out.stride(0))
    if ep is None and out.dtype == X.dtype and alpha == 1.0:
        _check(lib.tvw_gemm(form.dt, int(form.tvw), form.M, N, form.K, *tail, _stream(X.device)), "tvw_gemm")
    else:
        _check(lib.tvw_gemm_ep(form.dt, _DT[out.dtype], int(form.tvw), form.M, N, form.K, *tail, alpha,
                               None if ep is None else C.byref(ep), _stream(X.device)), "tvw_gemm_ep")
    return out


# ---------------------------------------------------------------- block-wise
@dataclass
class BlockWise:
    """A block-wise compressed weight (128 x 64 blocks kept per 128-row tile)."""
    dt: int
    M: int
    K: int
    keep: np.ndarray          # kept blocks per tile
    offsets: torch.Tensor     # in blocks
    indices: torch.Tensor     # kept block indices
    schedule: torch.Tensor
    packed: torch.Tensor


def bw_sizes(dt: int, M: int, K: int, keep_blocks) -> dict:
    k = _keep_arr(keep_blocks)
    out = [_sz() for _ in range(3)]
    _check(lib.bw_sizes(dt, M, K, _kp(k), *[C.byref(o) for o in out]), "bw_sizes")
    return dict(zip(("packed_bytes", "indices_count", "workspace_bytes"), (o.value for o in out)))


def bw_prune_compress(W: torch.Tensor, keep_blocks, workspace: torch.Tensor | None = None,
                      out: BlockWise | None = None) -> BlockWise:
    """Block-wise prune + pack. `out`, a result of an earlier call with the same
    shape, type and kept block counts, is overwritten in place (no allocation)."""
    dt = _DT[W.dtype]
    M, K = W.shape
    assert W.stride(1) == 1
    k = _keep_arr(keep_blocks)
    if out is not None:
        if (out.dt, out.M, out.K) != (dt, M, K) or not np.array_equal(out.keep, k):
            raise ValueError("bw_prune_compress: out was made for another weight shape or kept counts")
        if workspace is None:
            raise ValueError("bw_prune_compress: out= needs a workspace")
        _check(lib.bw_prune_compress(dt, _p(W), M, K, W.stride(0), _kp(out.keep), _p(out.offsets), _p(out.indices),
                                     _p(out.schedule), _p(out.packed), _p(workspace), _stream(W.device)),
               "bw_prune_compress")
        return out
    sz = bw_sizes(dt, M, K, k)
    dev = W.device
    nt = (M + 127) // 128
    offsets = torch.empty(nt + 1, dtype=torch.int32, device=dev)
    indices = torch.empty(max(1, sz["indices_count"]), dtype=torch.int32, device=dev)
    schedule = torch.empty(4 * max(1, nt), dtype=torch.int32, device=dev)
    packed = torch.empty(max(8, sz["packed_bytes"] // 2), dtype=W.dtype, device=dev)
    if workspace is None:
        workspace = torch.empty(max(16, sz["workspace_bytes"]), dtype=torch.uint8, device=dev)
    _check(lib.bw_prune_compress(dt, _p(W), M, K, W.stride(0), _kp(k), _p(offsets), _p(indices), _p(schedule),
                                 _p(packed), _p(workspace), _stream(dev)), "bw_prune_compress")
    return BlockWise(dt, M, K, k, offsets, indices[:sz["indices_count"]], schedule[:4 * nt],
                     packed[:sz["packed_bytes"] // 2])


def bw_gemm(form: BlockWise, X: torch.Tensor, out: torch.Tensor | None = None, out_dtype: torch.dtype | None = None,
            alpha: float = 1.0, bias: torch.Tensor | None = None, act: str = "none", y_scale: float = 1.0):
    """Y = W_bw . X (each tile: its kept blocks against their X panels); with the
    fused epilogue when bias / act / y_scale / alpha / another output type are given."""
    N = X.shape[1]
    if out is None:
        out = torch.empty((form.M, N), dtype=out_dtype or X.dtype, device=X.device)
    ep = _epilogue(bias, act, y_scale, form.M)
    tail = (_kp(form.keep), _p(form.offsets), _p(form.indices), _p(form.schedule), _p(form.packed), _p(X),
            X.stride(0), _p(out), out.stride(0))
    if ep is None and out.dtype == X.dtype and alpha == 1.0:
        _check(lib.bw_gemm(form.dt, form.M, N, form.K, *tail, _stream(X.device)), "bw_gemm")
    else:
        _check(lib.bw_gemm_ep(form.dt, _DT[out.dtype], form.M, N, form.K, *tail, alpha,
                              None if ep is None else C.byref(ep), _stream(X.device)), "bw_gemm_ep")
    return out


# ---------------------------------------------------------------- element-wise
@dataclass
class ElementWise:
    """An element-wise (unstructured) sparse weight in CSR form (k kept per row)."""
    dt: int
    M: int
    K: int
    k: int
    row_ptr: torch.Tensor
    col_idx: torch.Tensor
    vals: torch.Tensor
    col_buf: torch.Tensor | None = None   # the allocations behind col_idx / vals (at least one element,
    val_buf: torch.Tensor | None = None   # so that an empty CSR still passes valid pointers)


def ew_sizes(dt: int, M: int, K: int, k: int) -> dict:
    out = [_sz() for _ in range(3)]
    _check(lib.ew_sizes(dt, M, K, k, *[C.byref(o) for o in out]), "ew_sizes")
    return dict(zip(("vals_bytes", "indices_count", "workspace_bytes"), (o.value for o in out)))


def ew_prune_compress(W: torch.Tensor, k: int, workspace: torch.Tensor | None = None,
                      out: ElementWise | None = None) -> ElementWise:
    """Element-wise prune to CSR (k kept per row). `out`, a result of an earlier call
    with the same shape, type and k, is overwritten in place (no allocation)."""
    dt = _DT[W.dtype]
    M, K = W.shape
    assert W.stride(1) == 1
    if out is not None:
        if (out.dt, out.M, out.K, out.k) != (dt, M, K, k):
            raise ValueError("ew_prune_compress: out was made for another weight shape or k")
        if workspace is None:
            raise ValueError("ew_prune_compress: out= needs a workspace")
        _check(lib.ew_prune_compress(dt, _p(W), M, K, W.stride(0), k, _p(out.row_ptr), _p(out.col_buf),
                                     _p(out.val_buf), _p(workspace), _stream(W.device)), "ew_prune_compress")
        return out
    sz = ew_sizes(dt, M, K, k)
    dev = W.device
    row_ptr = torch.empty(M + 1, dtype=torch.int32, device=dev)
    col_idx = torch.empty(max(1, sz["indices_count"]), dtype=torch.int32, device=dev)
    vals = torch.empty(max(1, sz["indices_count"]), dtype=W.dtype, device=dev)
    if workspace is None:
        workspace = torch.empty(max(16, sz["workspace_bytes"]), dtype=torch.uint8, device=dev)
    _check(lib.ew_prune_compress(dt, _p(W), M, K, W.stride(0), k, _p(row_ptr), _p(col_idx), _p(vals), _p(workspace),
                                 _stream(dev)), "ew_prune_compress")
    n = sz["indices_count"]
    return ElementWise(dt, M, K, k, row_ptr, col_idx[:n], vals[:n], col_idx, vals)


def ew_spmm(form: ElementWise, X: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """Y = W_ew . X on the CUDA cores (fp32 accumulation, one rounding to X's type)."""
    N = X.shape[1]
    if out is None:
        out = torch.empty((form.M, N), dtype=X.dtype, device=X.device)
    cols = form.col_buf if form.col_buf is not None else form.col_idx
    vals = form.val_buf if form.val_buf is not None else form.vals
    _check(lib.ew_spmm(form.dt, form.M, N, form.K, _p(form.row_ptr), _p(cols), _p(vals), _p(X),
                       X.stride(0), _p(out), out.stride(0), _stream(X.device)), "ew_spmm")
    return out


# ---------------------------------------------------------------- 3x3 convolution
def conv3x3(filt, X: torch.Tensor, out: torch.Tensor | None = None, alpha: float = 1.0) -> torch.Tensor:
    """3x3 convolution (stride 1, zero padding 1) of NHWC activations X (Nb, H, W, Cin).
    `filt` is an Sp24 (the 2:4 form of the Cout x 9 Cin flattened filter), a
    BlockWise (the tile-wise filter: bw_prune_compress of the flattened filter, whose
    64-column blocks are (tap, 64-channel) groups), or the dense flattened filter
    tensor. Returns Y as Cout x (Nb H W)."""
    Nb, H, W, Cin = X.shape
    assert X.is_contiguous()
    dt = _DT[X.dtype]
    Cout = filt.M if isinstance(filt, (Sp24, BlockWise)) else filt.shape[0]
    if out is None:
        out = torch.empty((Cout, Nb * H * W), dtype=X.dtype, device=X.device)
    if isinstance(filt, BlockWise):
        assert filt.K == 9 * Cin and filt.dt == dt
        _check(lib.tw_conv3x3(dt, _DT[out.dtype], Cout, Cin, Nb, H, W, _kp(filt.keep), _p(filt.offsets),
                              _p(filt.indices), _p(filt.schedule), _p(filt.packed), _p(X), _p(out), out.stride(0),
                              alpha, _stream(X.device)), "tw_conv3x3")
        return out
    if isinstance(filt, Sp24):
        assert filt.K == 9 * Cin and filt.dt == dt
        _check(lib.sp24_conv3x3(dt, _DT[out.dtype], Cout, Cin, Nb, H, W, _p(filt.values), _p(filt.meta_hw), _p(X),
                                _p(out), out.stride(0), alpha, _stream(X.device)), "sp24_conv3x3")
    else:
        assert filt.shape[1] == 9 * Cin and filt.stride(1) == 1
        _check(lib.dense_conv3x3(dt, _DT[out.dtype], Cout, Cin, Nb, H, W, _p(filt), filt.stride(0), _p(X), _p(out),
                                 out.stride(0), alpha, _stream(X.device)), "dense_conv3x3")
    return out
