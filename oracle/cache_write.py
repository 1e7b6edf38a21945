"""KV-cache write (the step before the decode), written out in plain NumPy.

TEST INFRASTRUCTURE ONLY: nothing in the product path imports this package.

The decode path writes each new token's latent row into the page-size-1 pool
before attending over it: the 512 latent columns kv_c and the 64 RoPE columns
k_pe are concatenated into one 576-wide row at the token's slot, stored as bf16
or as fp8 with the per-tensor KV scale ("[ROCm] Dspark MLA module", Details: the
decode KV-cache write goes through concat_and_cache_mla; bf16 / fp8 caches with
a stacked k scale).  The same page reports the step reinterpreting an fp32 k_pe
as bf16 because nothing checked its dtype (review comment after the Test plan),
so here every input carries an explicit dtype and is converted, never
reinterpreted.

Definition, for token n with slot = slot_mapping[n]:
  skip the token when slot < 0 (padding) or slot >= num_slots;
  row = concat(kv_c[n, 0:512], k_pe[n, 0:64]) as float32 values
        (bf16 inputs widen exactly; fp32 inputs are taken as they are);
  bf16 pool: pool[slot] = bf16 round-to-nearest-even of row;
  fp8 pool:  inv = fp32(1 / fp32(kv_scale)), y = fp32(row * inv) (each product
             rounded to float32), pool[slot] = e4m3fn(y) rounded to nearest,
             ties to even, magnitudes above 448 saturated to +-448, NaN -> 0x7F.
A slot named by two tokens of one call is outside the contract (the oracle lets
the later token win).  The fp8 reading (scale applied as a float32 product with
the float32 reciprocal, saturation instead of NaN) is this build's reading: the
pages name the scale, not its arithmetic.
"""
from __future__ import annotations

import numpy as np

D_C, D_PE, D_QK = 512, 64, 576
E4M3_MAX = 448.0


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact: bf16 is the upper half of float32)."""
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_rne(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits, round to nearest, ties to even; NaN -> quiet NaN."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    keep = u >> 16                          # upper 16 bits (truncation)
    rest = u & 0xFFFF                       # discarded lower 16 bits
    up = (rest > 0x8000) | ((rest == 0x8000) & ((keep & 1) == 1))
    out = (keep + up.astype(np.uint64)) & 0xFFFF
    nan = np.isnan(np.ascontiguousarray(x, dtype=np.float32))
    out = np.where(nan, (keep | 0x40) & 0xFFFF, out)
    return out.astype(np.uint16)


def encode_e4m3fn_satfinite(y: np.ndarray) -> np.ndarray:
    """float values -> e4m3fn codes: nearest, ties to even, |y| > 448 -> +-448.

    e4m3fn: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 holds the
    subnormals m/8 * 2^-6 (step 2^-9); 0x7F / 0xFF are NaN, so the largest finite
    magnitude is 1.75 * 2^8 = 448 (code 0x7E).
    """
    y = np.asarray(y, dtype=np.float64)
    sign = np.signbit(y).astype(np.uint32) << 7
    big = ~(np.abs(y) < E4M3_MAX)                     # >= 448, inf or NaN: handled last
    a = np.where(big, 1.0, np.abs(y))
    code = np.zeros(a.shape, dtype=np.uint32)
    sub = a < 2.0 ** -6
    # subnormal range: multiples of 2^-9; rounding up to 8 units lands exactly on
    # the smallest normal, whose code (exponent 1, mantissa 0) is also 8
    code = np.where(sub, np.round(a / 2.0 ** -9).astype(np.int64), code)
    # normal range: a = f * 2^E with f in [0.5, 1)  ->  floor(log2 a) = E - 1
    _, E = np.frexp(np.where(sub, 1.0, a))
    e = (E - 1).astype(np.int64)                      # in [-6, 8] below 448
    q = np.round(np.where(sub, 8.0, a) / np.exp2((e - 3).astype(np.float64)))  # in [8, 16]
    carry = q >= 16
    e = np.where(carry, e + 1, e)
    q = np.where(carry, 8, q).astype(np.int64)
    normal_code = ((e + 7) << 3) | (q - 8)
    code = np.where(sub, code, normal_code).astype(np.int64)
    code = np.where(big, 0x7E, code)                  # saturate (448 itself is 0x7E)
    code = np.where(np.isnan(y), 0x7F, code | sign)
    return code.astype(np.uint8)


def scale_for_fp8(row_f32: np.ndarray, kv_scale: float) -> np.ndarray:
    """float32 row * float32(1 / float32(kv_scale)), each product rounded to float32."""
    inv = np.float32(1.0) / np.float32(kv_scale)
    return (np.asarray(row_f32, dtype=np.float32) * inv).astype(np.float32)


def cache_write(pool: np.ndarray, kv_c: np.ndarray, k_pe: np.ndarray, slot_mapping: np.ndarray,
                kv_dtype: str, kv_scale: float = 1.0) -> np.ndarray:
    """Return a copy of `pool` (uint16 bf16 bits or uint8 e4m3fn codes, [slots, 576])
    with the tokens written.  kv_c [n, 512] and k_pe [n, 64] are float32 arrays
    holding the input values (bf16 inputs widened with bf16_bits_to_f32)."""
    out = np.array(pool, copy=True)
    num_slots = out.shape[0]
    for n, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if slot < 0 or slot >= num_slots:
            continue
        row = np.concatenate([np.asarray(kv_c[n], np.float32), np.asarray(k_pe[n], np.float32)])
        if kv_dtype == "bf16":
            out[slot] = f32_to_bf16_rne(row)
        elif kv_dtype == "fp8":
            out[slot] = encode_e4m3fn_satfinite(scale_for_fp8(row, kv_scale))
        else:
            raise ValueError(f"unknown kv dtype {kv_dtype!r}")
    return out
