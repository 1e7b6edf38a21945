"""Pins for the oracle's per-entry positions (kv_pos) and sliding window.

Index lists of the DSV4 layer types (sliding window, window + top-k, window +
compressed entries) are decoded with each entry's global position.  These pins
tie that part of the oracle to things other than itself:
  * a pure-Python brute force that reads the positions and the window straight
    from the definition (direct exp, math.fsum);
  * closed forms: window 1 leaves one visible entry (O = v, LSE = s); a zero
    query gives the mean over, and the log of the count of, the window;
  * invariants: the sliding window given as its own index list with positions
    equals the whole committed KV with the window applied; explicit positions
    base + i*stride equal the implicit ones; a window longer than the context
    changes nothing;
  * a planted off-by-one in the window bound fails a pin.
"""
import dataclasses
import math

import numpy as np
import pytest

import mla_inputs as mi
from oracle import formats, mla_oracle as mo


def _brute(w):
    H = w.num_heads
    kappa = w.kv_scale if w.kv_dtype == "fp8" else 1.0
    O = np.zeros((w.total_q, H, mi.D_V))
    LSE = np.zeros((w.total_q, H))
    for b in range(w.batch):
        k0, k1 = int(w.kv_indptr[b]), int(w.kv_indptr[b + 1])
        q0, q1 = int(w.qo_indptr[b]), int(w.qo_indptr[b + 1])
        T = q1 - q0
        Lg = int(w.g_kv_indptr[b + 1] - w.g_kv_indptr[b]) if w.g_kv_indptr is not None else k1 - k0
        for t in range(T):
            lim = Lg - T + t
            for h in range(H):
                q = formats.decode_bf16(w.q_bits[q0 + t, h])
                es, rows = [], []
                for j in range(k0, k1):
                    g = int(w.kv_pos[j]) if w.kv_pos is not None else w.pos_base + (j - k0) * w.pos_stride
                    if w.causal and (g > lim or (w.window > 0 and g <= lim - w.window)):
                        continue
                    k = formats.decode_kv(w.kv_bits[w.kv_indices[j]], w.kv_dtype) * kappa
                    es.append(math.exp(w.softmax_scale * math.fsum(float(a) * float(c) for a, c in zip(q, k))))
                    rows.append(k)
                if not es:
                    LSE[q0 + t, h] = -math.inf
                    continue
                tot = math.fsum(es)
                LSE[q0 + t, h] = math.log(tot)
                O[q0 + t, h] = [math.fsum(e * r[d] for e, r in zip(es, rows)) / tot for d in range(mi.D_V)]
    return O, LSE


@pytest.mark.parametrize("kind", ["swa", "csa", "hca"])
def test_brute_force_layer_types(kind):
    w = mi.sparse_variant(kind, batch=2, num_heads=1, q_lens=[2, 1], global_lens=[300, 90], window=16,
                          topk=12, ratio=32, kv_dtype="bf16", seed=3)
    O, L = mo.mla_decode_workload(w)
    Ob, Lb = _brute(w)
    assert np.allclose(L, Lb, rtol=1e-12, atol=1e-12)
    assert np.allclose(O, Ob, rtol=1e-10, atol=1e-12)


def test_window_one_leaves_the_entry_at_the_limit():
    """W = 1: token t sees only position Lg - T + t: O = v, LSE = s."""
    w = mi.make_workload("w1", batch=1, num_heads=3, q_lens=[3], kv_lens=[20], kv_dtype="fp8",
                         causal=True, seed=21, num_slots=32)
    w = dataclasses.replace(w, window=1)
    O, L = mo.mla_decode_workload(w)
    for t in range(3):
        i = 20 - 3 + t
        k = formats.decode_e4m3fn(w.kv_bits[w.kv_indices[i]]) * w.kv_scale
        for h in range(3):
            q = formats.decode_bf16(w.q_bits[t, h])
            assert abs(L[t, h] - w.softmax_scale * float(np.dot(q, k))) < 1e-12
            assert np.allclose(O[t, h], k[:512], atol=1e-14)


def test_zero_query_averages_the_window():
    """q = 0 with window W: O = mean of the W newest visible rows, LSE = ln W."""
    W = 7
    w = mi.make_workload("zw", batch=2, num_heads=2, q_lens=[3, 2], kv_lens=[40, 5], kv_dtype="bf16",
                         causal=True, seed=22, num_slots=64)
    w = dataclasses.replace(w, window=W)
    w.q_bits[:] = 0
    O, L = mo.mla_decode_workload(w)
    for b in range(2):
        k0, k1 = int(w.kv_indptr[b]), int(w.kv_indptr[b + 1])
        q0, q1 = int(w.qo_indptr[b]), int(w.qo_indptr[b + 1])
        T, n = q1 - q0, k1 - k0
        V = formats.decode_bf16(w.kv_bits[w.kv_indices[k0:k1]])[:, :512]
        for t in range(T):
            lim = n - T + t
            lo = max(0, lim - W + 1)
            assert abs(L[q0 + t, 0] - math.log(lim - lo + 1)) < 1e-13
            assert np.allclose(O[q0 + t], V[lo:lim + 1].mean(axis=0)[None], atol=1e-12)


def test_window_list_equals_whole_list_with_window():
    """The sliding window as its own index list (with positions and the real
    lengths) equals the whole committed KV decoded with the window applied."""
    full = mi.make_workload("full", batch=3, num_heads=2, q_lens=[1, 3, 2], kv_lens=[200, 150, 33],
                            kv_dtype="fp8", causal=True, seed=8, num_slots=512)
    W = 40
    full = dataclasses.replace(full, window=W)
    O1, L1 = mo.mla_decode_workload(full)
    idx, pos, lens = [], [], []
    for b in range(3):
        k0, k1 = int(full.kv_indptr[b]), int(full.kv_indptr[b + 1])
        T = int(full.qo_indptr[b + 1] - full.qo_indptr[b])
        n = k1 - k0
        w0 = max(0, n - T - W + 1)
        idx.append(full.kv_indices[k0 + w0:k1])
        pos.append(np.arange(w0, n))
        lens.append(n - w0)
    win = dataclasses.replace(full, kv_indices=np.concatenate(idx).astype(np.int32),
                              kv_indptr=np.concatenate([[0], np.cumsum(lens)]).astype(np.int32),
                              kv_pos=np.concatenate(pos).astype(np.int32),
                              g_kv_indptr=full.kv_indptr.copy())
    O2, L2 = mo.mla_decode_workload(win)
    assert np.allclose(L1, L2, atol=1e-12) and np.allclose(O1, O2, atol=1e-12)


def test_explicit_positions_equal_implicit_ones():
    sw = mi.cp_shards_bf16(scale=1 / 1024)
    w = sw.shards
    pos = []
    for b in range(w.batch):
        n = int(w.kv_indptr[b + 1] - w.kv_indptr[b])
        pos.append(int(w.pos_base_per_req[b]) + w.pos_stride * np.arange(n))
    O1, L1 = mo.mla_decode_workload(w, requests=range(0, w.batch, 5))
    w2 = dataclasses.replace(w, kv_pos=np.concatenate(pos).astype(np.int32), pos_base_per_req=None, pos_base=10 ** 6)
    O2, L2 = mo.mla_decode_workload(w2, requests=range(0, w.batch, 5))
    m = ~np.isnan(L1[:, 0])
    assert np.array_equal(L1[m], L2[m]) and np.array_equal(O1[m], O2[m])


def test_long_window_changes_nothing():
    w = mi.make_workload("lw", batch=2, num_heads=2, q_lens=[2, 4], kv_lens=[60, 9], kv_dtype="bf16",
                         causal=True, seed=25, num_slots=128)
    O1, L1 = mo.mla_decode_workload(w)
    O2, L2 = mo.mla_decode_workload(dataclasses.replace(w, window=61))
    assert np.array_equal(L1, L2) and np.array_equal(O1, O2)
    O3, _ = mo.mla_decode_workload(dataclasses.replace(w, window=5))
    assert not np.allclose(O1, O3)                         # a short window does matter


def test_planted_off_by_one_window_fails(monkeypatch):
    orig = mo.visible_mask

    def wrong(L, T, t_of_row, causal, base, stride, Lg, pos=None, window=0):
        return orig(L, T, t_of_row, causal, base, stride, Lg, pos, window + 1 if window else 0)

    monkeypatch.setattr(mo, "visible_mask", wrong)
    with pytest.raises(AssertionError):
        test_window_one_leaves_the_entry_at_the_limit()
