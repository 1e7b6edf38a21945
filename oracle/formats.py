"""Storage-format decoders written from the formats' bit-level definitions.

TEST INFRASTRUCTURE ONLY: nothing in the product path imports this package.

* bf16: 1 sign bit, 8 exponent bits (bias 127), 7 mantissa bits; exponent 0 is
  subnormal (m / 2^7 * 2^-126), exponent 255 is inf (m = 0) or NaN.
* fp8 e4m3fn (the "fn" variant: finite, no infinities): 1 sign bit, 4 exponent
  bits (bias 7), 3 mantissa bits; exponent 0 is subnormal (m / 8 * 2^-6); the
  two codes 0x7F / 0xFF are NaN; the largest finite magnitude is 1.75 * 2^8 = 448.
  The pages store the latent KV cache "fp8" with a per-tensor scale
  ("[ROCm][Spec Decode] Add Aiter MLA decode support non-causal draft block",
  section "Three pieces"; "[ROCm] Dspark MLA module", Details); the e4m3fn
  variant is this build's reading of that word.

Both decoders return float64 and are pinned in tests against torch's own casts.
"""
from __future__ import annotations

import numpy as np


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits).astype(np.uint32)
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    exp = ((b >> 7) & 0xFF).astype(np.int64)
    man = (b & 0x7F).astype(np.float64)
    normal = sign * (1.0 + man / 128.0) * np.exp2((exp - 127).astype(np.float64))
    sub = sign * (man / 128.0) * 2.0 ** -126
    special = np.where(man == 0, sign * np.inf, np.nan)
    out = np.where(exp == 0, sub, np.where(exp == 255, special, normal))
    return out.astype(np.float64)


def decode_e4m3fn(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits).astype(np.uint32)
    sign = np.where((b >> 7) & 1, -1.0, 1.0)
    exp = ((b >> 3) & 0xF).astype(np.int64)
    man = (b & 0x7).astype(np.float64)
    normal = sign * (1.0 + man / 8.0) * np.exp2((exp - 7).astype(np.float64))
    sub = sign * (man / 8.0) * 2.0 ** -6
    out = np.where(exp == 0, sub, normal)
    out = np.where((b & 0x7F) == 0x7F, np.nan, out)
    return out.astype(np.float64)


def decode_kv(bits: np.ndarray, kv_dtype: str) -> np.ndarray:
    if kv_dtype == "bf16":
        return decode_bf16(bits)
    if kv_dtype == "fp8":
        return decode_e4m3fn(bits)
    raise ValueError(f"unknown kv dtype {kv_dtype!r}")
