"""Seeded synthetic inputs shared by the CUDA path and the CPU oracle.

This module only draws random numbers and stores them in the element types the
workloads use. It holds none of the sparse-GEMM arithmetic (no pruning, no
compression, no tile selection, no products): both sides consume the exact
bytes produced here.

Recipe (stated once, used everywhere):
  * splitmix64 stream: state_i = seed + (i + 1) * 0x9E3779B97F4A7C15 (mod 2**64),
    output = the splitmix64 finaliser of state_i (Steele, Lea, Flood, "Fast
    splittable pseudorandom number generators", OOPSLA 2014).
  * uniform u in [0, 1): the top 24 bits of an output times 2**-24.
  * normal: Box-Muller in fp64 on consecutive uniform pairs (u1, u2):
    r = sqrt(-2 ln(1 - u1)), z0 = r cos(2 pi u2), z1 = r sin(2 pi u2).
  * z * sigma is rounded to fp32 (RNE), then to the storage type (RNE): fp16
    and bf16 by the standard casts; e4m3 after dividing by a per-tensor scale
    s = amax / 448 (s = 1 when amax = 0), clamping to +-448 and casting.

Workload shapes follow the five layer shapes the method is evaluated on (a toy
2:4 layer, BERT-base FFN up/down, a ResNet-50 1x1 convolution, a 4096-square
tile-wise layer and an LLM FFN in fp8).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed: int, n: int, start: int = 0) -> np.ndarray:
    """n outputs of the splitmix64 stream for `seed`, beginning at index `start`."""
    out = np.empty(n, dtype=np.uint64)
    chunk = 1 << 20
    z = np.empty(min(n, chunk), dtype=np.uint64)
    t = np.empty_like(z)
    s0 = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
    for c0 in range(0, n, chunk):
        m = min(chunk, n - c0)
        zz, tt = z[:m], t[:m]
        zz[:] = np.arange(start + c0 + 1, start + c0 + m + 1, dtype=np.uint64)
        np.multiply(zz, _GOLDEN, out=zz)
        np.add(zz, s0, out=zz)
        np.right_shift(zz, np.uint64(30), out=tt)
        np.bitwise_xor(zz, tt, out=zz)
        np.multiply(zz, _M1, out=zz)
        np.right_shift(zz, np.uint64(27), out=tt)
        np.bitwise_xor(zz, tt, out=zz)
        np.multiply(zz, _M2, out=zz)
        np.right_shift(zz, np.uint64(31), out=tt)
        np.bitwise_xor(zz, tt, out=out[c0:c0 + m])
    return out


def uniform(seed: int, n: int) -> np.ndarray:
    """n fp64 uniforms in [0, 1) with 24-bit resolution."""
    z = splitmix64(seed, n)
    np.right_shift(z, np.uint64(40), out=z)
    u = z.astype(np.float64)
    u *= 2.0 ** -24
    return u


def normal(seed: int, n: int) -> np.ndarray:
    """n fp64 standard normals (Box-Muller over consecutive uniform pairs)."""
    m = (n + 1) // 2
    u = uniform(seed, 2 * m).reshape(m, 2)
    r = np.negative(u[:, 0])
    np.log1p(r, out=r)
    r *= -2.0
    np.sqrt(r, out=r)
    th = u[:, 1] * (2.0 * math.pi)
    z = np.empty((m, 2), dtype=np.float64)
    np.cos(th, out=z[:, 0])
    np.sin(th, out=z[:, 1])
    z[:, 0] *= r
    z[:, 1] *= r
    return z.reshape(-1)[:n]


# Storage types. Bits are kept as unsigned integers so that both sides see the
# exact same bytes; torch tensors of the matching dtype are views of them.
DTYPES = ("f16", "bf16", "e4m3")
ELEM_BYTES = {"f16": 2, "bf16": 2, "e4m3": 1}
TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}
BITS_DTYPE = {"f16": np.uint16, "bf16": np.uint16, "e4m3": np.uint8}


def to_storage(v: np.ndarray, dt: str) -> tuple[np.ndarray, float]:
    """Round fp64 values to fp32 then to `dt`; returns (bits, scale).

    scale is 1 for fp16/bf16; for e4m3 it is the per-tensor scale s such that
    the stored code q approximates v / s.
    """
    f32 = np.ascontiguousarray(v, dtype=np.float32)
    t = torch.from_numpy(f32)
    scale = 1.0
    if dt == "f16":
        bits = f32.astype(np.float16).view(np.uint16)
    elif dt == "bf16":
        bits = t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    elif dt == "e4m3":
        amax = float(np.max(np.abs(f32))) if f32.size else 0.0
        scale = float(np.float32(amax) / np.float32(448.0)) if amax > 0 else 1.0
        q = torch.clamp(t / torch.tensor(scale, dtype=torch.float32), -448.0, 448.0)
        bits = q.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    else:
        raise ValueError(dt)
    return np.ascontiguousarray(bits).copy(), scale


def normal_matrix(seed: int, rows: int, cols: int, sigma: float, dt: str,
                  relu: bool = False) -> tuple[np.ndarray, float]:
    z = normal(seed, rows * cols) * sigma
    if relu:
        z = np.maximum(z, 0.0)
    bits, scale = to_storage(z.reshape(rows, cols), dt)
    return bits.reshape(rows, cols), scale


def keep_counts(seed: int, tiles: int, K: int, lo: float = 0.15, hi: float = 0.35,
                quantum: int = 64) -> np.ndarray:
    """Per-tile kept K counts: u_t = lo + (hi - lo) * U[0,1), one draw per tile
    in tile order; L_t = quantum * round_half_even(u_t * K / quantum), clamped to
    [quantum, K]."""
    u = lo + (hi - lo) * uniform(seed, tiles)
    L = quantum * np.rint(u * K / quantum).astype(np.int64)
    return np.clip(L, quantum, K).astype(np.int32)


@dataclass(frozen=True)
class Workload:
    name: str
    dt: str           # input storage type of W and X
    out_dt: str       # Y type
    M: int
    K: int
    N: int
    sigma_w: float
    relu_x: bool = False
    tile_wise: bool = False
    seed: int = 0

    def make(self):
        """Returns dict with W bits (M x K), X bits (K x N), scales and, for
        tile-wise layers, keep counts per 128-row tile."""
        W, sw = normal_matrix(1000 + self.seed, self.M, self.K, self.sigma_w, self.dt)
        X, sx = normal_matrix(2000 + self.seed, self.K, self.N, 1.0, self.dt, relu=self.relu_x)
        out = {"W": W, "X": X, "s_w": sw, "s_x": sx, "alpha": float(np.float32(sw) * np.float32(sx))}
        if self.tile_wise:
            out["keep"] = keep_counts(3000 + self.seed, (self.M + 127) // 128, self.K)
        return out


WORKLOADS = {
    "toy_fp16": Workload("toy_fp16", "f16", "f16", 256, 256, 128, 1.0, seed=1),
    "bert_ffn_up_bf16": Workload("bert_ffn_up_bf16", "bf16", "bf16", 3072, 768, 1024, 0.02, seed=2),
    "bert_ffn_down_bf16": Workload("bert_ffn_down_bf16", "bf16", "bf16", 768, 3072, 1024, 0.02, seed=12),
    "resnet50_1x1_fp16": Workload("resnet50_1x1_fp16", "f16", "f16", 256, 1024, 6272,
                                  math.sqrt(2.0 / 1024.0), relu_x=True, seed=3),
    "tile_wise_4096_bf16": Workload("tile_wise_4096_bf16", "bf16", "bf16", 4096, 4096, 4096, 0.02,
                                    tile_wise=True, seed=4),
    "llm_ffn_e4m3": Workload("llm_ffn_e4m3", "e4m3", "bf16", 14336, 4096, 8192, 0.02, seed=5),
    # The same LLM FFN shape stored in bf16: the shape on which the 2:4-sparse
    # bf16 tensor-core rate is measured.
    "llm_ffn_bf16": Workload("llm_ffn_bf16", "bf16", "bf16", 14336, 4096, 8192, 0.02, seed=15),
}


def torch_view(bits: np.ndarray, dt: str) -> torch.Tensor:
    """A torch tensor of storage type `dt` viewing (a copy of) the given bits."""
    b = np.ascontiguousarray(bits)
    if dt == "e4m3":
        return torch.from_numpy(b.view(np.uint8).copy()).view(torch.float8_e4m3fn)
    return torch.from_numpy(b.view(np.int16).copy()).view(TORCH_DTYPE[dt])
