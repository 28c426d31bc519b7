"""Exact decoding of the KV storage formats to float64 (oracle side).

The KV cache may be stored as fp32, bf16 or fp8 e4m3 with a per-kv-head scale
("Deploying FlashRec", precision table: fp8_e4m3 KV cache).  Decoding is done
from the bit patterns with the textbook formulas, independent of any torch or
CUDA conversion routine:

* bf16: the upper 16 bits of an IEEE binary32 value.
* e4m3 (OCP FP8 "E4M3FN"): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
  exponent 0 encodes subnormals m/8 * 2^-6; S.1111.111 is NaN; no infinities.
"""
import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64 (exact)."""
    u32 = bits.astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def e4m3_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """uint8 e4m3fn bit patterns -> float64 (exact; NaN for 0x7f / 0xff)."""
    b = bits.astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    normal = sign * (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = sign * (m / 8.0) * 2.0 ** -6
    out = np.where(e == 0, sub, normal)
    return np.where((e == 0xF) & ((b & 0x7) == 0x7), np.nan, out)


def to_f64(arr, kv_dtype: int, scale=None) -> np.ndarray:
    """Decode a KV array (numpy view of its raw storage) to float64.

    ``kv_dtype``: 0 = fp32, 1 = bf16 (uint16 bits), 2 = e4m3 (uint8 bits).
    ``scale``: per-kv-head float array applied along axis -2 for e4m3.
    """
    if kv_dtype == 0:
        return np.asarray(arr, dtype=np.float32).astype(np.float64)
    if kv_dtype == 1:
        return bf16_bits_to_f64(np.asarray(arr, dtype=np.uint16))
    x = e4m3_bits_to_f64(np.asarray(arr, dtype=np.uint8))
    if scale is not None:
        x = x * np.asarray(scale, dtype=np.float32).astype(np.float64)[:, None]
    return x
