"""Float64 CPU oracle for MLA paged decode with a multi-token query block.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import it; it shares no code with the CUDA path.

What it computes (the plain definition; the GPU method reaches the same result
up to rounding order):

For request b with local KV length L_b, query tokens T_b and head h:
  k_i     = dec(pool[kv_indices[kv_indptr[b] + i]]) * kappa        i in [0, L_b)
            (kappa = kv_scale for an fp8 pool, 1 for bf16)
  s_i     = sigma * <q[t, h, 0:576], k_i[0:576]>                    sigma = softmax_scale
  V_t     = { i : not causal  or  g_b(i) <= Lg_b - T_b + t },  g_b(i) = base_b + i * stride
            (g_b(i) = kv_pos[kv_indptr[b] + i] when per-entry positions are given;
             with a window W > 0, causal rows also need g_b(i) > Lg_b - T_b + t - W)
  LSE     = ln sum_{i in V_t} exp(s_i)                              (natural log)
  O       = sum_{i in V_t} exp(s_i - LSE) * k_i[0:512]
  empty V_t:  O = 0, LSE = -inf

Sources on the pages:
  * absorbed-latent decode: one 576-wide latent row per KV entry (512 latent +
    64 RoPE) serves every head, and the output lives in the 512-wide latent
    space -- "[ROCm] Dspark MLA module", Details (absorb BMM, MLAAttention,
    concat_and_cache_mla writes kv_c and k_pe);
  * a page-size-1 flat index list per request (kv_indptr / kv_indices) --
    "[ROCm][Spec Decode] Add Aiter MLA decode support non-causal draft block",
    Purpose;
  * non-causal draft block: every token of the block sees the whole committed KV
    -- same page, Purpose;
  * causal mask on global positions over a round-robin context-parallel shard,
    with the global lengths carried by g_kv_indptr and an LSE output --
    "Speculative decode + DCP on gfx1250", Problem;
  * per-tensor fp8 scale -- "[ROCm][Spec Decode] ...", section "Three pieces".
  * index lists other than the whole committed KV: one plan per layer type --
    a sliding window (SWA), a window plus top-k selected entries (CSA), a
    window plus one compressed entry per 128 tokens (HCA) -- over the same
    decode ("[DSV4] Tuned ASM FP8 decode with split plans; HCA on aiter's
    persistent V4-NM kernel", Summary part 1).  Such lists are not a run of
    positions base + i*stride, so each entry can carry its global position
    (kv_pos), and the sliding window is a lower bound on visible positions.
The exact causal limit (token t of a T-token block sees global positions up to
Lg - T + t), the window reading (positions in (limit - W, limit]), the 576/512
widths and the natural-log LSE are this build's readings where the pages are
silent.

Computation uses max subtraction and processes query rows in chunks so memory
stays bounded; the chunking is exact (each row is independent).
"""
from __future__ import annotations

import math
from typing import Optional, Tuple

import numpy as np

from .formats import decode_bf16, decode_kv

D_QK = 576
D_V = 512


def visible_mask(L: int, T: int, t_of_row: np.ndarray, causal: bool, base: int, stride: int,
                 Lg: int, pos: Optional[np.ndarray] = None, window: int = 0) -> np.ndarray:
    """Boolean [rows, L]: entry i is visible to the row's token t.

    Non-causal: all L entries.  Causal: the entry's global position (pos[i] when
    given, else base + i*stride) must not exceed limit = Lg - T + t, and with a
    window W > 0 must also exceed limit - W.
    """
    if not causal:
        return np.ones((t_of_row.shape[0], L), dtype=bool)
    g = (np.asarray(pos, dtype=np.int64) if pos is not None
         else base + stride * np.arange(L, dtype=np.int64))
    limit = (Lg - T + t_of_row.astype(np.int64))[:, None]
    vis = g[None, :] <= limit
    if window > 0:
        vis &= g[None, :] > limit - window
    return vis


def attend_rows(qrows: np.ndarray, K: np.ndarray, vis: np.ndarray,
                sigma: float) -> Tuple[np.ndarray, np.ndarray]:
    """Masked softmax attention of float64 query rows over float64 KV rows.

    qrows [R, 576], K [L, 576], vis [R, L] -> O [R, 512], LSE [R].
    """
    R = qrows.shape[0]
    if K.shape[0] == 0:
        return np.zeros((R, D_V)), np.full(R, -np.inf)
    s = sigma * (qrows @ K.T)
    s = np.where(vis, s, -np.inf)
    m = s.max(axis=1)
    has = np.isfinite(m)
    m_safe = np.where(has, m, 0.0)
    e = np.exp(s - m_safe[:, None])
    e = np.where(vis, e, 0.0)
    l = e.sum(axis=1)
    with np.errstate(divide="ignore"):
        lse = np.where(has, m_safe + np.log(np.where(has, l, 1.0)), -np.inf)
    o = (e @ K[:, :D_V]) / np.where(has, l, 1.0)[:, None]
    o[~has] = 0.0
    return o, lse


def mla_decode(q_bits: np.ndarray, kv_bits: np.ndarray, kv_dtype: str,
               kv_indptr: np.ndarray, kv_indices: np.ndarray, qo_indptr: np.ndarray,
               causal: bool, softmax_scale: float, kv_scale: float = 1.0,
               pos_base: int = 0, pos_stride: int = 1,
               pos_base_per_req: Optional[np.ndarray] = None,
               g_kv_indptr: Optional[np.ndarray] = None,
               requests=None, row_chunk: int = 64, kv_pos: Optional[np.ndarray] = None,
               window: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """Reference MLA decode.  Returns O float64 [total_q, H, 512] and LSE float64 [total_q, H].

    ``requests`` restricts the work to a subset of request indices (rows of the
    other requests are left as NaN), which the tests and the CPU baseline use to
    sample large workloads.
    """
    total_q, H, dq = q_bits.shape
    assert dq == D_QK and kv_bits.shape[1] == D_QK
    kappa = float(kv_scale) if kv_dtype == "fp8" else 1.0
    B = kv_indptr.shape[0] - 1
    O = np.full((total_q, H, D_V), np.nan)
    LSE = np.full((total_q, H), np.nan)
    reqs = range(B) if requests is None else requests
    for b in reqs:
        k0, k1 = int(kv_indptr[b]), int(kv_indptr[b + 1])
        q0, q1 = int(qo_indptr[b]), int(qo_indptr[b + 1])
        L, T = k1 - k0, q1 - q0
        if T <= 0:
            continue
        K = decode_kv(kv_bits[kv_indices[k0:k1]], kv_dtype) * kappa
        base = int(pos_base_per_req[b]) if pos_base_per_req is not None else int(pos_base)
        Lg = int(g_kv_indptr[b + 1] - g_kv_indptr[b]) if g_kv_indptr is not None else L
        qrows = decode_bf16(q_bits[q0:q1]).reshape(T * H, D_QK)
        t_of_row = np.arange(T * H) // H
        o_b = np.empty((T * H, D_V))
        lse_b = np.empty(T * H)
        for r0 in range(0, T * H, row_chunk):
            r1 = min(T * H, r0 + row_chunk)
            vis = visible_mask(L, T, t_of_row[r0:r1], causal, base, pos_stride, Lg,
                               None if kv_pos is None else kv_pos[k0:k1], window)
            o_b[r0:r1], lse_b[r0:r1] = attend_rows(qrows[r0:r1], K, vis, softmax_scale)
        O[q0:q1] = o_b.reshape(T, H, D_V)
        LSE[q0:q1] = lse_b.reshape(T, H)
    return O, LSE


def mla_decode_workload(w, **kw) -> Tuple[np.ndarray, np.ndarray]:
    """Convenience wrapper over a ``mla_inputs.Workload``."""
    return mla_decode(w.q_bits, w.kv_bits, w.kv_dtype, w.kv_indptr, w.kv_indices, w.qo_indptr,
                      w.causal, w.softmax_scale, w.kv_scale, w.pos_base, w.pos_stride,
                      w.pos_base_per_req, w.g_kv_indptr, kv_pos=w.kv_pos, window=w.window, **kw)


def merge_states(o_parts: np.ndarray, lse_parts: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Combine partial attention states over disjoint KV subsets.

    o_parts [n, rows, dv] (each normalised over its own subset), lse_parts [n, rows]:
      M   = max_s lse_s
      LSE = M + ln sum_s exp(lse_s - M)
      O   = sum_s exp(lse_s - LSE) * O_s
    A state with lse = -inf (empty subset) contributes nothing; if every state is
    empty the result is O = 0, LSE = -inf.  This is the split-and-merge the pages
    describe for long rows ("[DSV4] Tuned ASM FP8 decode ...", Summary part 2,
    in-kernel split and merge) and the per-shard LSE combine that round-robin
    context parallelism needs ("Speculative decode + DCP on gfx1250", Problem).
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    M = lse_parts.max(axis=0)
    has = np.isfinite(M)
    M_safe = np.where(has, M, 0.0)
    w = np.where(np.isfinite(lse_parts), np.exp(lse_parts - M_safe[None]), 0.0)
    tot = w.sum(axis=0)
    with np.errstate(divide="ignore"):
        lse = np.where(has, M_safe + np.log(np.where(has, tot, 1.0)), -np.inf)
    coef = w / np.where(has, tot, 1.0)[None]
    o = np.einsum("sr,srd->rd", coef, np.where(np.isfinite(lse_parts)[..., None], o_parts, 0.0))
    o[~has] = 0.0
    return o, lse


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 (ties to even), returned as float64.

    Used by tests to model the kernel's bf16 output rounding when a tolerance is
    derived; never to produce an expected value.
    """
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounding = 0x7FFF + ((u >> 16) & 1)
    r = ((u + rounding) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def ln(x: float) -> float:
    return math.log(x)
