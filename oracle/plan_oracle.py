"""Work/split plan specification, written out in plain Python integers.

TEST INFRASTRUCTURE ONLY.  The CUDA library implements the same specification on
its own (host planner in C++ and a device planner kernel); tests require both to
produce this module's plan bit for bit.

The pages fix the ideas, not the numbers:
  * a split count per row and a split table that depends only on the row count
    and configuration, built on the host next to the CSR so that CUDA-graph
    capture and replay agree ("[DSV4] Tuned ASM FP8 decode with split plans; HCA
    on aiter's persistent V4-NM kernel", Summary part 1, which also uses a
    16-row uniform split table);
  * a persistent kernel that plans the split from the real per-row KV lengths on
    every call ("[DSV4] ...", Summary part 2).
The constants and the tie-break rules below are this build's choices.  ROWS and
BLOCK_N are the library's (256 query rows per work item, 128 KV entries per tile);
every function also takes them as keyword arguments, so plans worked out by hand
for other values stay checkable.

Specification (all integers, 64-bit intermediates):
  For request b:  T_b = qo_indptr[b+1]-qo_indptr[b],  L_b = kv_indptr[b+1]-kv_indptr[b]
    G_b = ceil(H*T_b / ROWS)          query-row groups (0 when T_b = 0)
    N_b = ceil(L_b / BLOCK_N)         DYNAMIC, HOST: from the real length
          ceil(cap / BLOCK_N)         STATIC: from the capacity kv_len_cap
  total  = sum_b G_b * N_b
  target = max(MIN_TILES, ceil(total / W))             W = num_workers
  S_b    = min(MAX_SPLITS, max(1, ceil(N_b / target)))
  group_base[b]   = sum_{b'<b} G_b'
  partial_base[b] = sum_{b'<b, S_b'>1} S_b' * G_b'   (-1 when S_b = 1)
  items, enumerated with b outer, then s in [0,S_b), then g in [0,G_b):
    partial_slot = partial_base[b] + s*G_b + g  (or -1 when S_b = 1)
    tiles [t0,t1) = [floor(s*N_b/S_b), floor((s+1)*N_b/S_b))
    cost = (t1 - t0) + 1
  items are sorted by min(cost, 65535) descending; ties keep enumeration order.
  At run time the kernel recomputes each split's tile range from the actual L_b
  with the planned S_b, so a STATIC plan stays valid as lengths change.

Buffer layout (int32, little endian):
  header[16] = MAGIC, VERSION, B, H, max_q_len, W, mode, n_items, n_partials,
               n_groups, cap_lo, cap_hi, ROWS, BLOCK_N, items_capacity, 0
  S[B], group_base[B+1], partial_base[B], items[items_capacity][4] = (b, s, g, slot)
  items_capacity = W + B * ceil(H*max_q_len/ROWS) bounds n_items for any lengths,
  because sum_b S_b*G_b <= sum_b G_b*(N_b/target + 1) <= W + sum_b G_b.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

MAGIC = 0x4D4C4150
VERSION = 1
ROWS = 256
BLOCK_N = 128
MAX_SPLITS = 16
MIN_TILES = 4
COST_CLAMP = 65535
STATIC = 0
DYNAMIC = 1
HOST = 2            # built on the host from the real lengths, used as is
HEADER_INTS = 16


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


def items_capacity(batch: int, num_heads: int, max_q_len: int, num_workers: int, rows: int = ROWS) -> int:
    return num_workers + batch * cdiv(num_heads * max_q_len, rows)


def plan_ints(batch: int, num_heads: int, max_q_len: int, num_workers: int, rows: int = ROWS) -> int:
    cap = items_capacity(batch, num_heads, max_q_len, num_workers, rows)
    return HEADER_INTS + batch + (batch + 1) + batch + 4 * cap


def build_plan(batch: int, num_heads: int, max_q_len: int, num_workers: int, kv_len_cap: int,
               mode: int, kv_indptr: Optional[np.ndarray], qo_indptr: np.ndarray, *,
               rows: int = ROWS, block_n: int = BLOCK_N) -> np.ndarray:
    """Return the plan buffer as an int32 array (raises ValueError on invalid input)."""
    if batch < 0 or num_heads < 1 or max_q_len < 0 or num_workers < 1 or mode not in (STATIC, DYNAMIC, HOST):
        raise ValueError("invalid plan parameters")
    if mode == STATIC and kv_len_cap < 0:
        raise ValueError("negative kv_len_cap")
    T = [int(qo_indptr[b + 1]) - int(qo_indptr[b]) for b in range(batch)]
    if any(t < 0 or t > max_q_len for t in T):
        raise ValueError("q length outside [0, max_q_len]")
    if mode in (DYNAMIC, HOST):
        L = [int(kv_indptr[b + 1]) - int(kv_indptr[b]) for b in range(batch)]
        if any(x < 0 for x in L):
            raise ValueError("decreasing kv_indptr")
        N = [cdiv(x, block_n) for x in L]
    else:
        N = [cdiv(int(kv_len_cap), block_n)] * batch
    G = [cdiv(num_heads * t, rows) for t in T]
    total = sum(g * n for g, n in zip(G, N))
    target = max(MIN_TILES, cdiv(total, num_workers))
    S = [min(MAX_SPLITS, max(1, cdiv(n, target))) for n in N]

    group_base = [0] * (batch + 1)
    for b in range(batch):
        group_base[b + 1] = group_base[b] + G[b]
    partial_base = []
    run = 0
    for b in range(batch):
        if S[b] > 1:
            partial_base.append(run)
            run += S[b] * G[b]
        else:
            partial_base.append(-1)
    n_partials = run

    items = []
    for b in range(batch):
        for s in range(S[b]):
            t0 = (s * N[b]) // S[b]
            t1 = ((s + 1) * N[b]) // S[b]
            cost = (t1 - t0) + 1
            for g in range(G[b]):
                slot = partial_base[b] + s * G[b] + g if S[b] > 1 else -1
                items.append((min(cost, COST_CLAMP), len(items), (b, s, g, slot)))
    cap = items_capacity(batch, num_heads, max_q_len, num_workers, rows)
    if len(items) > cap or cap > 65535:
        raise ValueError("item capacity exceeded")
    items.sort(key=lambda it: (-it[0], it[1]))

    out = np.zeros(plan_ints(batch, num_heads, max_q_len, num_workers, rows), dtype=np.int64)
    cap64 = int(kv_len_cap) if mode == STATIC else 0
    hdr = [MAGIC, VERSION, batch, num_heads, max_q_len, num_workers, mode, len(items), n_partials,
           group_base[batch], cap64 & 0xFFFFFFFF, (cap64 >> 32) & 0xFFFFFFFF, rows, block_n, cap, 0]
    out[:HEADER_INTS] = hdr
    o = HEADER_INTS
    out[o:o + batch] = S
    o += batch
    out[o:o + batch + 1] = group_base
    o += batch + 1
    out[o:o + batch] = partial_base
    o += batch
    for k, (_, _, rec) in enumerate(items):
        out[o + 4 * k: o + 4 * k + 4] = rec
    return (out & 0xFFFFFFFF).astype(np.uint32).view(np.int32)


def parse_plan(buf: np.ndarray) -> dict:
    """Split a plan buffer into named fields (for tests)."""
    buf = np.asarray(buf, dtype=np.int32)
    B = int(buf[2])
    cap = int(buf[14])
    o = HEADER_INTS
    S = buf[o:o + B]
    o += B
    gb = buf[o:o + B + 1]
    o += B + 1
    pb = buf[o:o + B]
    o += B
    items = buf[o:o + 4 * cap].reshape(cap, 4)[: int(buf[7])]
    return dict(magic=int(buf[0]), version=int(buf[1]), batch=B, num_heads=int(buf[3]),
                max_q_len=int(buf[4]), num_workers=int(buf[5]), mode=int(buf[6]),
                n_items=int(buf[7]), n_partials=int(buf[8]), n_groups=int(buf[9]),
                splits=S, group_base=gb, partial_base=pb, items=items, capacity=cap)


def split_tile_range(s: int, S_b: int, L_b: int, block_n: int = BLOCK_N):
    """Entry range [e0, e1) of split s of S_b over a request of real length L_b."""
    N = cdiv(L_b, block_n)
    t0 = (s * N) // S_b
    t1 = ((s + 1) * N) // S_b
    return block_n * t0, min(block_n * t1, L_b)
