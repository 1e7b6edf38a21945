"""Seeded synthetic inputs for MLA paged decode.

This module is shared by the float64 oracle tests, the GPU parity tests and the
benchmark.  It only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Every tensor is produced on the host with
``numpy.random.default_rng(seed)`` and then rounded to its storage type with
torch's own casts (bf16 round-to-nearest-even, fp8 e4m3fn), so the oracle and
the CUDA path see the very same bytes.

Workload shapes follow the pages:
  * draft blocks of 7-8 tokens over an 8k committed context
    ("[ROCm][Spec Decode] Add Aiter MLA decode support non-causal draft block",
    Purpose and Test Plan);
  * 128 local heads with an fp8 cache ("[DSV4] Tuned ASM FP8 decode with split
    plans; HCA on aiter's persistent V4-NM kernel", Summary part 2);
  * 64 / 96 gathered heads and round-robin context-parallel shards
    ("Speculative decode + DCP on gfx1250", Problem).
Each latent KV entry is 576 wide: 512 latent + 64 RoPE.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

D_QK = 576
D_V = 512
SEED_BASE = 20261202
SOFTMAX_SCALE = 1.0 / math.sqrt(192.0)
FP8_KV_SCALE = 0.05
FP8_E4M3_MAX = 448.0


@dataclasses.dataclass
class Workload:
    """One decode call's inputs, as raw storage bits plus index metadata."""

    name: str
    num_heads: int
    q_bits: np.ndarray            # uint16 [total_q, H, 576], bf16 bit patterns
    kv_bits: np.ndarray           # uint16 (bf16) or uint8 (fp8 e4m3fn) [num_slots, 576]
    kv_dtype: str                 # "bf16" | "fp8"
    kv_indptr: np.ndarray         # int32 [B+1]
    kv_indices: np.ndarray        # int32 [nnz]
    qo_indptr: np.ndarray         # int32 [B+1]
    causal: bool
    softmax_scale: float
    kv_scale: float = 1.0
    pos_base: int = 0
    pos_stride: int = 1
    pos_base_per_req: Optional[np.ndarray] = None   # int32 [B]
    g_kv_indptr: Optional[np.ndarray] = None        # int32 [B+1]
    kv_pos: Optional[np.ndarray] = None             # int32 [nnz] global position of each entry
    window: int = 0                                 # sliding window (causal only), 0 = none
    meta: dict = dataclasses.field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.kv_indptr.shape[0] - 1)

    @property
    def num_slots(self) -> int:
        return int(self.kv_bits.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.qo_indptr[-1])

    def kv_lens(self) -> np.ndarray:
        return np.diff(self.kv_indptr.astype(np.int64))

    def q_lens(self) -> np.ndarray:
        return np.diff(self.qo_indptr.astype(np.int64))


# ----------------------------------------------------------------------------
# storage casts (torch does the rounding; we only move bits around)
# ----------------------------------------------------------------------------

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def to_fp8_bits(x: np.ndarray, scale: float) -> np.ndarray:
    """Stored byte = e4m3fn(x / scale); values are clipped to +-448 first."""
    import torch
    y = np.clip(np.asarray(x, dtype=np.float32) / np.float32(scale), -FP8_E4M3_MAX, FP8_E4M3_MAX)
    t = torch.from_numpy(np.ascontiguousarray(y))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _normal_bits(rng: np.random.Generator, shape, kv_dtype: str, kv_scale: float,
                 chunk_rows: int = 1 << 16) -> np.ndarray:
    """N(0,1) rows cast to storage bits, generated chunk by chunk to bound memory."""
    rows, width = shape
    out = np.empty((rows, width), dtype=np.uint16 if kv_dtype == "bf16" else np.uint8)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = rng.standard_normal((r1 - r0, width), dtype=np.float32)
        out[r0:r1] = to_bf16_bits(x) if kv_dtype == "bf16" else to_fp8_bits(x, kv_scale)
    return out


def _pow2_at_least(n: int) -> int:
    p = 1
    while p < n:
        p <<= 1
    return p


def _indptr(lens) -> np.ndarray:
    out = np.zeros(len(lens) + 1, dtype=np.int64)
    out[1:] = np.cumsum(np.asarray(lens, dtype=np.int64))
    assert out[-1] < 2 ** 31
    return out.astype(np.int32)


def make_workload(name: str, *, batch: int, num_heads: int, q_lens, kv_lens,
                  kv_dtype: str, causal: bool, seed: int, num_slots: Optional[int] = None,
                  softmax_scale: float = SOFTMAX_SCALE, kv_scale: Optional[float] = None,
                  identical_q_rows: bool = False, draw_pool: bool = True) -> Workload:
    """Generic generator: random q, random pool, kv_indices = seeded permutation prefix.

    ``draw_pool=False`` leaves the pool undrawn (an all-zero read-only view of the
    right shape): for extra draws of lengths and indices that reuse another
    workload's pool."""
    rng = np.random.default_rng(seed)
    q_lens = np.asarray(q_lens, dtype=np.int64)
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    assert q_lens.shape == (batch,) and kv_lens.shape == (batch,)
    nnz = int(kv_lens.sum())
    if num_slots is None:
        num_slots = max(1, _pow2_at_least(nnz))
    assert num_slots >= nnz
    if kv_scale is None:
        kv_scale = FP8_KV_SCALE if kv_dtype == "fp8" else 1.0
    perm = rng.permutation(num_slots).astype(np.int32)
    kv_indices = perm[:nnz].copy()
    total_q = int(q_lens.sum())
    if identical_q_rows:
        one = rng.standard_normal((1, 1, D_QK), dtype=np.float32)
        qf = np.broadcast_to(one, (total_q, num_heads, D_QK)).copy()
    else:
        qf = rng.standard_normal((total_q, num_heads, D_QK), dtype=np.float32)
    q_bits = to_bf16_bits(qf)
    if draw_pool:
        kv_bits = _normal_bits(rng, (num_slots, D_QK), kv_dtype, kv_scale)
    else:
        kv_bits = np.broadcast_to(np.zeros((1, D_QK), dtype=np.uint16 if kv_dtype == "bf16" else np.uint8),
                                  (num_slots, D_QK))
    return Workload(name=name, num_heads=num_heads, q_bits=q_bits, kv_bits=kv_bits,
                    kv_dtype=kv_dtype, kv_indptr=_indptr(kv_lens), kv_indices=kv_indices,
                    qo_indptr=_indptr(q_lens), causal=causal, softmax_scale=softmax_scale,
                    kv_scale=float(kv_scale))


# ----------------------------------------------------------------------------
# the five workloads (plus scaled-down variants for fast parity runs)
# ----------------------------------------------------------------------------

def tiny_causal_bf16() -> Workload:
    """Batch 2, 16 heads, T=2, KV lengths 37 and 100 in a 256-slot pool, causal, bf16.

    kv_indices: a seeded permutation of the 256 slots; request 0 takes the first
    37, request 1 the next 100.
    """
    return make_workload("tiny_causal_bf16", batch=2, num_heads=16, q_lens=[2, 2],
                         kv_lens=[37, 100], kv_dtype="bf16", causal=True,
                         seed=SEED_BASE + 0, num_slots=256)


def draft_block_bf16(scale: float = 1.0, seed: Optional[int] = None) -> Workload:
    """Non-causal draft block: batch 8, T=8, 64 heads, 8192 committed KV, bf16.

    The pool has 131072 slots; the 65536 used ones are the prefix of a seeded
    permutation.  ``scale`` < 1 shrinks the context and pool for quick parity runs.
    """
    L = max(1, int(round(8192 * scale)))
    slots = 131072 if scale == 1.0 else _pow2_at_least(8 * L) * 2
    w = make_workload("draft_block_bf16" + ("" if scale == 1.0 else f"_x{scale:g}"),
                      batch=8, num_heads=64, q_lens=[8] * 8, kv_lens=[L] * 8,
                      kv_dtype="bf16", causal=False,
                      seed=SEED_BASE + 1 if seed is None else seed, num_slots=slots)
    return w


def verify_fp8(scale: float = 1.0, seed: Optional[int] = None) -> Workload:
    """Causal verify pass: batch 32, T=8, 128 heads, fp8 KV (scale 0.05), L ~ U[1024, 16384]."""
    rng = np.random.default_rng(SEED_BASE + 2 if seed is None else seed)
    lo, hi = max(1, int(1024 * scale)), max(2, int(16384 * scale))
    lens = rng.integers(lo, hi, size=32, endpoint=True)
    w = make_workload("verify_fp8" + ("" if scale == 1.0 else f"_x{scale:g}"),
                      batch=32, num_heads=128, q_lens=[8] * 32, kv_lens=lens,
                      kv_dtype="fp8", causal=True, seed=int(rng.integers(1 << 31)))
    w.meta["kv_len_cap"] = hi
    return w


def long_skewed_fp8(replay: int = 0, scale: float = 1.0, num_slots: Optional[int] = None,
                    batch: int = 64, draw_pool: bool = True) -> Workload:
    """Batch 64, T in {1,2,4}, 128 heads, fp8, L = floor(exp(U[ln 256, ln 131072])), causal.

    ``replay`` selects a fresh draw of lengths, T and indices (graph replays with
    changed lengths).  ``num_slots`` fixes the pool capacity across replays.
    """
    rng = np.random.default_rng(SEED_BASE + 3 + 1000 * replay)
    lo, hi = 256 * scale, 131072 * scale
    lens = np.floor(np.exp(rng.uniform(math.log(lo), math.log(hi), size=batch))).astype(np.int64)
    lens = np.maximum(lens, 1)
    qls = rng.choice(np.array([1, 2, 4]), size=batch)
    w = make_workload("long_skewed_fp8" + ("" if scale == 1.0 else f"_x{scale:g}") + f"_r{replay}",
                      batch=batch, num_heads=128, q_lens=qls, kv_lens=lens, kv_dtype="fp8",
                      causal=True, seed=int(rng.integers(1 << 31)), num_slots=num_slots,
                      draw_pool=draw_pool)
    return w


def long_skewed_pool_slots(replays: int, scale: float = 1.0, batch: int = 64) -> int:
    """Pool capacity covering every replay's total KV length."""
    need = 0
    for r in range(replays):
        rng = np.random.default_rng(SEED_BASE + 3 + 1000 * r)
        lo, hi = 256 * scale, 131072 * scale
        lens = np.floor(np.exp(rng.uniform(math.log(lo), math.log(hi), size=batch))).astype(np.int64)
        need = max(need, int(np.maximum(lens, 1).sum()))
    return _pow2_at_least(need)


@dataclasses.dataclass
class ShardedWorkload:
    """Round-robin context-parallel shards of one unsharded causal workload."""

    full: Workload            # the unsharded problem (positions 0..Lg-1)
    shards: Workload          # (shard, request) flattened shard-major into one batched call
    num_shards: int


def cp_shards_bf16(scale: float = 1.0, num_shards: int = 8) -> ShardedWorkload:
    """Global KV 32768 split round-robin into 8 shards; batch 16, T=8, 96 heads, bf16, causal.

    Shard r holds the global positions r, r+8, r+16, ...; its local entry i is
    global position r + 8 i.  All shards run as one batched call over
    (shard, request) pairs, shard-major, with pos_base_per_req = r, stride 8 and
    g_kv_indptr carrying the global length.
    """
    Lg = max(num_shards, int(32768 * scale))
    B, T, H = 16, 8, 96
    full = make_workload("cp_full_bf16" + ("" if scale == 1.0 else f"_x{scale:g}"),
                         batch=B, num_heads=H, q_lens=[T] * B, kv_lens=[Lg] * B,
                         kv_dtype="bf16", causal=True, seed=SEED_BASE + 4,
                         num_slots=_pow2_at_least(B * Lg))
    idx = [full.kv_indices[full.kv_indptr[b]:full.kv_indptr[b + 1]] for b in range(B)]
    sh_idx, sh_lens, base, g_lens = [], [], [], []
    for r in range(num_shards):
        for b in range(B):
            part = idx[b][r::num_shards]
            sh_idx.append(part)
            sh_lens.append(part.shape[0])
            base.append(r)
            g_lens.append(Lg)
    q_bits = np.concatenate([full.q_bits] * num_shards, axis=0)
    shards = Workload(name=full.name.replace("cp_full", "cp_shards"), num_heads=H,
                      q_bits=q_bits, kv_bits=full.kv_bits, kv_dtype="bf16",
                      kv_indptr=_indptr(sh_lens), kv_indices=np.concatenate(sh_idx).astype(np.int32),
                      qo_indptr=_indptr([T] * (B * num_shards)), causal=True,
                      softmax_scale=full.softmax_scale, kv_scale=1.0, pos_base=0,
                      pos_stride=num_shards, pos_base_per_req=np.asarray(base, dtype=np.int32),
                      g_kv_indptr=_indptr(g_lens))
    return ShardedWorkload(full=full, shards=shards, num_shards=num_shards)


def flatten_block(w: Workload) -> Workload:
    """The flattened form of a non-causal block: one single-token request per query token,
    each reading its request's whole committed KV list."""
    assert not w.causal
    idx: List[np.ndarray] = []
    lens = []
    for b in range(w.batch):
        seg = w.kv_indices[w.kv_indptr[b]:w.kv_indptr[b + 1]]
        for _ in range(int(w.qo_indptr[b + 1] - w.qo_indptr[b])):
            idx.append(seg)
            lens.append(seg.shape[0])
    return dataclasses.replace(
        w, name=w.name + "_flat", kv_indptr=_indptr(lens),
        kv_indices=np.concatenate(idx).astype(np.int32) if idx else np.zeros(0, np.int32),
        qo_indptr=_indptr([1] * len(lens)))


CONFIG_NAMES = ["tiny_causal_bf16", "draft_block_bf16", "verify_fp8", "long_skewed_fp8", "cp_shards_bf16"]
def sparse_variant(kind: str, *, batch: int, num_heads: int, q_lens, global_lens, window: int = 128,
                   topk: int = 2048, ratio: int = 128, kv_dtype: str = "fp8", seed: int = SEED_BASE + 7,
                   num_slots: Optional[int] = None) -> Workload:
    """Index lists of the DSV4 layer types over a page-size-1 pool, every entry with
    its global position (kv_pos), causal on global positions (g_kv_indptr = the
    requests' real lengths Lg).  Token t of a T-token block sits at Lg - T + t.
      swa: the positions a T-token block can see through a sliding window W,
           [Lg - T - W + 1, Lg); the decode applies the window (window = W).
      csa: the window's positions plus `topk` distinct positions drawn (seeded,
           uniformly) from the older ones, sorted; no window bound.
      hca: one compressed entry per complete block of `ratio` positions before the
           window (its position is the block's last), then the window's
           positions; no window bound.
    Pool rows are N(0,1) latent rows (compressed entries are just more rows)."""
    rng = np.random.default_rng(seed)
    q_lens = np.asarray(q_lens, dtype=np.int64)
    Lg = np.asarray(global_lens, dtype=np.int64)
    pos_lists = []
    for b in range(batch):
        T, L = int(q_lens[b]), int(Lg[b])
        w0 = max(0, L - T - window + 1)
        win = np.arange(w0, L, dtype=np.int64)
        if kind == "swa":
            pos = win
        elif kind == "csa":
            k = min(topk, w0)
            pos = np.sort(np.concatenate([rng.choice(w0, size=k, replace=False), win]))
        elif kind == "hca":
            nblk = w0 // ratio
            pos = np.concatenate([np.arange(nblk, dtype=np.int64) * ratio + ratio - 1, win])
        else:
            raise ValueError(kind)
        pos_lists.append(pos)
    lens = np.array([len(p) for p in pos_lists], dtype=np.int64)
    nnz = int(lens.sum())
    if num_slots is None:
        num_slots = max(1, _pow2_at_least(nnz))
    kv_scale = FP8_KV_SCALE if kv_dtype == "fp8" else 1.0
    kv_indices = rng.permutation(num_slots)[:nnz].astype(np.int32)
    total_q = int(q_lens.sum())
    q_bits = to_bf16_bits(rng.standard_normal((total_q, num_heads, D_QK), dtype=np.float32))
    kv_bits = _normal_bits(rng, (num_slots, D_QK), kv_dtype, kv_scale)
    return Workload(name=f"{kind}_{kv_dtype}", num_heads=num_heads, q_bits=q_bits, kv_bits=kv_bits,
                    kv_dtype=kv_dtype, kv_indptr=_indptr(lens), kv_indices=kv_indices,
                    qo_indptr=_indptr(q_lens), causal=True, softmax_scale=SOFTMAX_SCALE,
                    kv_scale=float(kv_scale), g_kv_indptr=_indptr(Lg),
                    kv_pos=np.concatenate(pos_lists).astype(np.int32) if nnz else np.zeros(0, np.int32),
                    window=window if kind == "swa" else 0)


@dataclasses.dataclass
class RopeInputs:
    """Inputs of the fused decode RoPE + q concat + cache write (bf16 bit patterns)."""
    q_nope_bits: np.ndarray      # uint16 [n, H, 512] absorbed latent q
    q_pe_bits: np.ndarray        # uint16 [n, H, 64] RoPE columns of q, not yet rotated
    kv_c_bits: np.ndarray        # uint16 [n, 512]
    k_pe_bits: np.ndarray        # uint16 [n, 64], not yet rotated
    positions: np.ndarray        # int32 [n]
    cos_sin: np.ndarray          # float32 [max_pos, 64]: cos of the 32 angles, then their sin
    slot_mapping: np.ndarray     # int32 [n]
    num_slots: int


def rope_inputs(num_tokens: int, num_heads: int, max_pos: int = 131072, num_slots: Optional[int] = None,
                seed: int = SEED_BASE + 9, rope_base: float = 10000.0) -> RopeInputs:
    """Seeded activations N(0,1), positions uniform in [0, max_pos), slots a seeded
    permutation prefix, and a rotary table for 32 angles p * base^(-2i/64) (the
    plain RoPE table; models with scaled tables pass their own)."""
    rng = np.random.default_rng(seed)
    n, H = num_tokens, num_heads
    if num_slots is None:
        num_slots = max(16, _pow2_at_least(n))
    f = lambda *shape: to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))  # noqa: E731
    inv_freq = rope_base ** (-np.arange(0, 64, 2, dtype=np.float64) / 64.0)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    cos_sin = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
    return RopeInputs(q_nope_bits=f(n, H, 512), q_pe_bits=f(n, H, 64), kv_c_bits=f(n, 512), k_pe_bits=f(n, 64),
                      positions=rng.integers(0, max_pos, size=n).astype(np.int32), cos_sin=cos_sin,
                      slot_mapping=rng.permutation(num_slots)[:n].astype(np.int32), num_slots=num_slots)


@dataclasses.dataclass
class BmmInputs:
    """One absorb BMM: activations x (bf16 bits [n, H, K]) times a per-head weight
    stored as [H, K, N] (bf16 bits, or fp8 e4m3fn codes with a per-tensor scale)."""
    x_bits: np.ndarray
    w_bits: np.ndarray
    w_dtype: str
    w_scale: float


def bmm_inputs(num_tokens: int, num_heads: int, k: int, n: int, w_dtype: str = "fp8",
               seed: int = SEED_BASE + 11, x_std: float = 1.0) -> BmmInputs:
    """Seeded x ~ N(0, x_std^2) and weights ~ N(0, 1/k) (unit-scale outputs, the
    usual initialisation of a projection); an fp8 weight is stored per tensor as
    e4m3fn(w / s) with s = max|w| / 448.  Absorb: k=128, n=512 (W_UK); un-absorb:
    k=512, n=128 (W_UV)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((num_tokens, num_heads, k), dtype=np.float32) * np.float32(x_std)
    w = rng.standard_normal((num_heads, k, n), dtype=np.float32) * np.float32(1.0 / math.sqrt(k))
    if w_dtype == "bf16":
        return BmmInputs(to_bf16_bits(x), to_bf16_bits(w), "bf16", 1.0)
    scale = float(np.float32(np.abs(w).max() / 448.0))
    return BmmInputs(to_bf16_bits(x), to_fp8_bits(w, scale), "fp8", scale)


# decode over the DSV4 layer types' index lists (per-entry positions)
SPARSE_CONFIG_NAMES = ["csa_topk_fp8", "hca_fp8"]
# the KV-cache write that precedes the decode (a separate call, measured on its own)
EXTRA_CONFIG_NAMES = ["cache_write_fp8", "cache_write_bf16", "rope_cache_fp8", "absorb_bmm_fp8"]


@dataclasses.dataclass
class CacheWriteInputs:
    """New tokens' activations and their slots.  kv_c / k_pe are float32 arrays of
    the input values; with bf16 inputs they hold bf16-representable values and
    kv_c_bits / k_pe_bits hold the bf16 patterns."""
    kv_c: np.ndarray
    k_pe: np.ndarray
    kv_c_bits: Optional[np.ndarray]
    k_pe_bits: Optional[np.ndarray]
    slot_mapping: np.ndarray
    num_slots: int
    kv_scale: float


def cache_write_inputs(num_tokens: int, num_slots: int, *, kv_c_dtype: str = "bf16", k_pe_dtype: str = "bf16",
                       seed: int = SEED_BASE + 6, padding: float = 0.0, out_of_range: float = 0.0,
                       spread: bool = False) -> CacheWriteInputs:
    """Seeded inputs: values N(0,1) (with spread=True a mix of magnitudes from 1e-5 to
    40, so fp8 at kv_scale 0.05 sees subnormals and saturation), slots a seeded
    permutation prefix of the pool, a fraction replaced by -1 (padding) or by
    slots past the end."""
    rng = np.random.default_rng(seed)
    assert num_tokens <= num_slots
    def draw(shape, dtype):
        x = rng.standard_normal(shape).astype(np.float32)
        if spread:
            x *= rng.choice(np.array([1e-5, 1e-3, 0.05, 1.0, 10.0, 40.0], np.float32), size=shape)
        if dtype == "bf16":
            bits = to_bf16_bits(x)
            return (bits.astype(np.uint32) << 16).view(np.float32), bits
        return x, None
    kv_c, kv_c_bits = draw((num_tokens, 512), kv_c_dtype)
    k_pe, k_pe_bits = draw((num_tokens, 64), k_pe_dtype)
    slots = rng.permutation(num_slots)[:num_tokens].astype(np.int32)
    u = rng.random(num_tokens)
    slots[u < padding] = -1
    slots[(u >= padding) & (u < padding + out_of_range)] = num_slots + rng.integers(0, 1000)
    return CacheWriteInputs(kv_c=kv_c, k_pe=k_pe, kv_c_bits=kv_c_bits, k_pe_bits=k_pe_bits,
                            slot_mapping=slots, num_slots=num_slots, kv_scale=FP8_KV_SCALE)


# ----------------------------------------------------------------------------
# device upload (plain copies of the same bytes)
# ----------------------------------------------------------------------------

def to_device(w: Workload, device="cuda") -> dict:
    """Copy a workload's bytes to the device as the tensors the C ABI takes."""
    import torch
    dev = torch.device(device)

    def i32(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    q = torch.from_numpy(w.q_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    if w.kv_dtype == "bf16":
        kv = torch.from_numpy(w.kv_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        kv = torch.from_numpy(w.kv_bits).to(dev).view(torch.float8_e4m3fn)
    return dict(q=q, kv_pool=kv, kv_dtype=0 if w.kv_dtype == "bf16" else 1,
                kv_indptr=i32(w.kv_indptr), kv_indices=i32(w.kv_indices), qo_indptr=i32(w.qo_indptr),
                causal=w.causal, softmax_scale=w.softmax_scale, kv_scale=w.kv_scale,
                pos_base=w.pos_base, pos_stride=w.pos_stride,
                pos_base_per_req=i32(w.pos_base_per_req), g_kv_indptr=i32(w.g_kv_indptr),
                kv_pos=i32(w.kv_pos), window=int(w.window))
