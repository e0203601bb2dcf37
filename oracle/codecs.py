"""Element-type codecs written from the format definitions.

  fp16 : IEEE 754 binary16 (1 sign, 5 exponent bits with bias 15, 10 fraction bits).
  bf16 : the top half of IEEE binary32 (1 sign, 8 exponent bits with bias 127,
         7 fraction bits).
  e4m3 : OCP 8-bit floating point E4M3 (1 sign, 4 exponent bits with bias 7,
         3 fraction bits); no infinities, S.1111.111 is NaN, largest finite 448.

Decoding is exact in fp64. Encoding rounds an fp64 value to the nearest
representable value, ties to even (the output rounding of the GEMM).
"""
from __future__ import annotations

import numpy as np

# (precision in significant bits, smallest subnormal exponent, largest finite)
_FORMATS = {
    "f16": (11, -24, 65504.0),
    "bf16": (8, -133, float.fromhex("0x1.fep127")),
    "e4m3": (4, -9, 448.0),
}


def _decode_generic(bits: np.ndarray, ebits: int, fbits: int, bias: int,
                    ieee_special: bool) -> np.ndarray:
    b = bits.astype(np.int64)
    sign = (b >> (ebits + fbits)) & 1
    e = (b >> fbits) & ((1 << ebits) - 1)
    f = b & ((1 << fbits) - 1)
    emax = (1 << ebits) - 1
    mag = np.where(e == 0,
                   np.ldexp(f.astype(np.float64), 1 - bias - fbits),
                   np.ldexp((f + (1 << fbits)).astype(np.float64), e - bias - fbits))
    if ieee_special:
        mag = np.where(e == emax, np.where(f == 0, np.inf, np.nan), mag)
    else:  # OCP E4M3: only S.1111.111 is special (NaN); exponent 15 is otherwise finite
        mag = np.where((e == emax) & (f == (1 << fbits) - 1), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def decode(bits: np.ndarray, dt: str) -> np.ndarray:
    """Exact fp64 values of the stored bits of type dt."""
    if dt == "f16":
        return _decode_generic(bits, 5, 10, 15, True)
    if dt == "bf16":
        return _decode_generic(bits, 8, 7, 127, True)
    if dt == "e4m3":
        return _decode_generic(bits, 4, 3, 7, False)
    raise ValueError(dt)


def round_to(x: np.ndarray, dt: str) -> np.ndarray:
    """Round fp64 x to the nearest value representable in dt (ties to even).

    Values beyond the largest finite magnitude become +-inf for fp16/bf16 and
    saturate to +-448 for e4m3. The result is an fp64 array whose entries are
    exactly representable in dt.
    """
    p, qmin_exp, maxval = _FORMATS[dt]
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    fin = np.isfinite(x) & (x != 0)
    xf = x[fin]
    _, e = np.frexp(xf)                      # |xf| = m * 2**e, 0.5 <= m < 1
    q_exp = np.maximum(e - p, qmin_exp)      # weight of the last kept bit
    q = np.ldexp(1.0, q_exp)
    r = np.rint(xf / q) * q                  # np.rint rounds half to even; xf/q is exact
    big = np.abs(r) > maxval
    if dt == "e4m3":
        r = np.where(big, np.copysign(maxval, r), r)
    else:
        r = np.where(big, np.copysign(np.inf, r), r)
    out[fin] = r
    return out


def encode(x: np.ndarray, dt: str) -> np.ndarray:
    """Bits of round_to(x, dt). NaN maps to the canonical quiet NaN of dt."""
    r = round_to(x, dt)
    if dt == "f16":
        return r.astype(np.float16).view(np.uint16)          # exact: r is representable
    if dt == "bf16":
        f = r.astype(np.float32).view(np.uint32)              # exact: r is representable
        bits = (f >> np.uint32(16)).astype(np.uint16)
        return np.where(np.isnan(r), np.uint16(0x7FC0), bits).astype(np.uint16)
    if dt == "e4m3":
        # r holds representable values only: look each magnitude up among the 127
        # finite non-negative codes (ascending in value), then set the sign bit
        pos = np.arange(127, dtype=np.uint8)                  # 0x00 .. 0x7E
        vals = decode(pos, "e4m3")
        mag = np.abs(r)
        idx = np.clip(np.searchsorted(vals, np.where(np.isnan(mag), 0.0, mag)), 0, 126)
        code = pos[idx]
        assert np.all((vals[idx] == mag) | np.isnan(mag)), "value not representable in e4m3"
        code = np.where(np.signbit(r), code | np.uint8(0x80), code).astype(np.uint8)
        return np.where(np.isnan(r), np.uint8(0x7F), code).astype(np.uint8)
    raise ValueError(dt)
