"""Helpers shared by the GPU parity tests: device transfer of stored bits and
the bound check against the oracle."""
import numpy as np
import pytest
import torch

from structured_sparse_dnn_gb300 import inputs as I

DT_CODE = {"f16": 0, "bf16": 1, "e4m3": 2}
REL = {"f16": 1e-2, "bf16": 1e-2, "e4m3": 6e-2}   # elementwise bound factors (fp16/bf16, fp8)
CANARY = 0x5A


def lib():
    """The binding; fails loudly (no skip) when the library is missing on a GPU machine."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from structured_sparse_dnn_gb300 import build
    build.build()
    from structured_sparse_dnn_gb300 import ssdnn
    return ssdnn


def dev_tensor(bits: np.ndarray, dt: str) -> torch.Tensor:
    return I.torch_view(bits, dt).cuda()


def dev_padded(bits: np.ndarray, dt: str, align_bytes: int = 16) -> torch.Tensor:
    """A device view of the matrix whose row pitch is rounded up to align_bytes."""
    rows, cols = bits.shape
    eb = I.ELEM_BYTES[dt]
    ld = -(-cols * eb // align_bytes) * align_bytes // eb
    full = np.zeros((rows, ld), dtype=bits.dtype)
    full[:, :cols] = bits
    return dev_tensor(full, dt)[:, :cols]


def bits_of(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.element_size() == 1:
        return t.view(torch.uint8).numpy().copy()
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def rand_bits(seed: int, shape, dt: str, sigma: float = 1.0) -> np.ndarray:
    bits, _ = I.normal_matrix(seed, shape[0], shape[1], sigma, dt)
    return bits


def guarded_output(M: int, N: int, dtype, pad_cols: int = 8, pad_rows: int = 2):
    """An M x N output view inside a larger buffer filled with a canary byte; the
    view has leading dimension N + pad_cols. Returns (view, buffer)."""
    ld = N + pad_cols
    buf = torch.empty((M + pad_rows, ld), dtype=dtype, device="cuda")
    buf.view(torch.uint8).fill_(CANARY)
    return buf[:M, :N], buf


def canary_intact(buf: torch.Tensor, M: int, N: int) -> bool:
    b = buf.view(torch.uint8).cpu().numpy().reshape(buf.shape[0], -1)
    eb = buf.element_size()
    return bool((b[:M, N * eb:] == CANARY).all() and (b[M:] == CANARY).all())
