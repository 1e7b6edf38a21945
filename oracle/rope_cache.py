"""Fused decode RoPE + q concat + KV-cache write, written out in plain NumPy.

TEST INFRASTRUCTURE ONLY: nothing in the product path imports this package.

After the absorb, the decode applies the rotary embedding to the 64 RoPE columns
of q and k, concatenates q's 512 absorbed latent columns with its rotated RoPE
columns into the 576-wide q the decode reads, and writes kv_c with the rotated
k_pe into the cache ("[ROCm] Dspark MLA module": fused_qk_rope_concat_and_cache_mla,
decode RoPE + cache after absorb, left there as a follow-up; the same page's
review comment shows the rotated k_pe coming out in float32 and being read as
bf16).  The rotary tables are an input (the pages' models build them with YaRN
scaling; the fused step only applies them).

Definition, token n at position p = positions[n] (clamped to [0, max_pos)),
c = cos_sin[p, 0:32], s = cos_sin[p, 32:64] (float32), for a 64-wide x in
float32 (bf16 inputs widen exactly):
  neox style (rotate halves):   a = x[0:32], b = x[32:64]
      y[0:32]  = a*c - b*s,   y[32:64] = b*c + a*s
  interleaved style (pairs):    a = x[0::2], b = x[1::2]
      y[0::2]  = a*c - b*s,   y[1::2]  = b*c + a*s
  every product and every sum rounded to float32 on its own (no fused
  multiply-add), so the result is one exact float32 per element.
  q_out[n, h] = (q_nope[n, h, 0:512], bf16(rope(q_pe[n, h])))   bf16 [576]
  pool[slot_mapping[n]] = cache row of (kv_c[n], rope(k_pe[n]))  as in cache_write.py
Which rotation style a model uses is its own choice; both are offered.
"""
from __future__ import annotations

import numpy as np

from .cache_write import bf16_bits_to_f32, cache_write, f32_to_bf16_rne

NEOX, INTERLEAVED = 0, 1


def rope_f32(x: np.ndarray, cos: np.ndarray, sin: np.ndarray, style: int) -> np.ndarray:
    """x [..., 64] float32, cos/sin [..., 32] float32 -> rotated float32 [..., 64]."""
    x = np.asarray(x, dtype=np.float32)
    c = np.asarray(cos, dtype=np.float32)
    s = np.asarray(sin, dtype=np.float32)
    if style == NEOX:
        a, b = x[..., :32], x[..., 32:]
    elif style == INTERLEAVED:
        a, b = x[..., 0::2], x[..., 1::2]
    else:
        raise ValueError(f"unknown rope style {style}")
    ac = (a * c).astype(np.float32)
    bs = (b * s).astype(np.float32)
    bc = (b * c).astype(np.float32)
    as_ = (a * s).astype(np.float32)
    ya = (ac - bs).astype(np.float32)
    yb = (bc + as_).astype(np.float32)
    y = np.empty_like(x)
    if style == NEOX:
        y[..., :32], y[..., 32:] = ya, yb
    else:
        y[..., 0::2], y[..., 1::2] = ya, yb
    return y


def rope_q_cache(q_nope_bits: np.ndarray, q_pe_bits: np.ndarray, kv_c_bits: np.ndarray, k_pe_bits: np.ndarray,
                 positions: np.ndarray, cos_sin: np.ndarray, style: int, slot_mapping: np.ndarray,
                 pool: np.ndarray, kv_dtype: str, kv_scale: float = 1.0):
    """bf16 bit inputs: q_nope [n, H, 512], q_pe [n, H, 64], kv_c [n, 512], k_pe [n, 64];
    positions int [n]; cos_sin float32 [max_pos, 64].  Returns (q_out bits uint16
    [n, H, 576], new pool)."""
    max_pos = cos_sin.shape[0]
    p = np.clip(np.asarray(positions, dtype=np.int64), 0, max_pos - 1)
    cos, sin = cos_sin[p, :32].astype(np.float32), cos_sin[p, 32:].astype(np.float32)
    qr = rope_f32(bf16_bits_to_f32(q_pe_bits), cos[:, None, :], sin[:, None, :], style)
    q_out = np.concatenate([np.asarray(q_nope_bits, np.uint16), f32_to_bf16_rne(qr)], axis=-1)
    kr = rope_f32(bf16_bits_to_f32(k_pe_bits), cos, sin, style)
    new_pool = cache_write(pool, bf16_bits_to_f32(kv_c_bits), kr, slot_mapping, kv_dtype, kv_scale)
    return q_out, new_pool
