"""Pins for the float64 oracle: checks against things other than the oracle itself.

Each test ties the oracle to a library routine, a closed form, a brute-force
evaluation or an invariant the pages fix, so a plausible slip anywhere in it (a
dropped term, a wrong sign or index, an off-by-one in the causal limit, a
transposed operand) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import mla_inputs as mi
from oracle import formats, mla_oracle as mo, plan_oracle as po

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- formats

def test_e4m3fn_decoder_exhaustive_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = formats.decode_e4m3fn(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(ours[m], ref[m])
    assert np.nanmax(ours) == 448.0 and np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])
    assert ours[0x01] == 2.0 ** -9  # smallest subnormal


def test_bf16_decoder_exhaustive_vs_torch():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = formats.decode_bf16(codes)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(ours[m], ref[m])


def test_bf16_round_matches_torch():
    x = np.random.default_rng(1).standard_normal(10000) * 10
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(mo.bf16_round(x), ref)


# ---------------------------------------------------------------- brute force

def _brute_force(w):
    """Direct exp (no max subtraction) and math.fsum sums, pure-Python loops."""
    H = w.num_heads
    kappa = w.kv_scale if w.kv_dtype == "fp8" else 1.0
    O = np.zeros((w.total_q, H, mi.D_V))
    LSE = np.zeros((w.total_q, H))
    for b in range(w.batch):
        k0, k1 = int(w.kv_indptr[b]), int(w.kv_indptr[b + 1])
        q0, q1 = int(w.qo_indptr[b]), int(w.qo_indptr[b + 1])
        T = q1 - q0
        K = [list(formats.decode_kv(w.kv_bits[w.kv_indices[j]], w.kv_dtype) * kappa)
             for j in range(k0, k1)]
        Lg = (int(w.g_kv_indptr[b + 1] - w.g_kv_indptr[b]) if w.g_kv_indptr is not None
              else k1 - k0)
        base = int(w.pos_base_per_req[b]) if w.pos_base_per_req is not None else w.pos_base
        for t in range(T):
            for h in range(H):
                q = list(formats.decode_bf16(w.q_bits[q0 + t, h]))
                es, vis_rows = [], []
                for i, k in enumerate(K):
                    gpos = base + i * w.pos_stride
                    if w.causal and gpos > Lg - T + t:
                        continue
                    s = w.softmax_scale * math.fsum(a * c for a, c in zip(q, k))
                    es.append(math.exp(s))
                    vis_rows.append(k)
                if not es:
                    LSE[q0 + t, h] = -math.inf
                    continue
                tot = math.fsum(es)
                LSE[q0 + t, h] = math.log(tot)
                for d in range(mi.D_V):
                    O[q0 + t, h, d] = math.fsum(e * k[d] for e, k in zip(es, vis_rows)) / tot
    return O, LSE


def _shrink(w, heads=2):
    """Keep only the first `heads` heads (brute force cost)."""
    import dataclasses
    return dataclasses.replace(w, num_heads=heads, q_bits=np.ascontiguousarray(w.q_bits[:, :heads]))


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_brute_force_tiny(kv_dtype):
    w = mi.make_workload("bf", batch=2, num_heads=3, q_lens=[2, 3], kv_lens=[7, 19],
                         kv_dtype=kv_dtype, causal=True, seed=5, num_slots=64)
    O, L = mo.mla_decode_workload(w)
    Ob, Lb = _brute_force(w)
    assert np.allclose(L, Lb, rtol=1e-12, atol=1e-12)
    assert np.allclose(O, Ob, rtol=1e-10, atol=1e-12)


def test_brute_force_config1_two_heads():
    w = _shrink(mi.tiny_causal_bf16(), heads=2)
    O, L = mo.mla_decode_workload(w)
    Ob, Lb = _brute_force(w)
    assert np.allclose(L, Lb, rtol=1e-12, atol=1e-12)
    assert np.allclose(O, Ob, rtol=1e-10, atol=1e-12)


def test_brute_force_cp_positions():
    """Global-position mask with a base and a stride, checked by brute force."""
    sw = mi.cp_shards_bf16(scale=1 / 2048)   # Lg = 16, shards of 2
    w = _shrink(sw.shards, heads=1)
    O, L = mo.mla_decode_workload(w, requests=range(0, w.batch, 7))
    Ob, Lb = _brute_force(w)
    m = ~np.isnan(L[:, 0])
    assert m.any()
    assert np.allclose(L[m], Lb[m], rtol=1e-12, atol=1e-12)
    assert np.allclose(O[m], Ob[m], rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- closed forms

def _bits(x):
    return mi.to_bf16_bits(np.asarray(x, dtype=np.float32))


def test_zero_query_gives_mean_and_log_count():
    """q = 0: every visible logit is 0, so O = mean of the visible V rows, LSE = ln |V_t|.
    With the causal limit Lg - T + t, token t sees L - T + t + 1 entries."""
    w = mi.make_workload("z", batch=2, num_heads=4, q_lens=[3, 5], kv_lens=[10, 40],
                         kv_dtype="bf16", causal=True, seed=9, num_slots=64)
    w.q_bits[:] = 0
    O, L = mo.mla_decode_workload(w)
    for b in range(2):
        k0, k1 = w.kv_indptr[b], w.kv_indptr[b + 1]
        q0, q1 = w.qo_indptr[b], w.qo_indptr[b + 1]
        T, Lb = q1 - q0, k1 - k0
        V = formats.decode_bf16(w.kv_bits[w.kv_indices[k0:k1]])[:, :512]
        for t in range(T):
            n = Lb - T + t + 1
            assert np.allclose(L[q0 + t], math.log(n), atol=1e-13)
            assert np.allclose(O[q0 + t], V[:n].mean(axis=0)[None], atol=1e-12)


def test_identical_kv_rows():
    """All KV rows equal to k: O = k[:512], LSE = s + ln |V_t|."""
    w = mi.make_workload("ik", batch=1, num_heads=2, q_lens=[4], kv_lens=[13],
                         kv_dtype="bf16", causal=True, seed=11, num_slots=16)
    w.kv_bits[:] = w.kv_bits[w.kv_indices[0]][None]
    O, L = mo.mla_decode_workload(w)
    k = formats.decode_bf16(w.kv_bits[0])
    for t in range(4):
        for h in range(2):
            q = formats.decode_bf16(w.q_bits[t, h])
            s = w.softmax_scale * float(np.dot(q, k))
            assert abs(L[t, h] - (s + math.log(13 - 4 + t + 1))) < 1e-11
            assert np.allclose(O[t, h], k[:512], atol=1e-12)


def test_single_visible_entry():
    """Causal, L = T: token 0 sees exactly one entry: O = v_0, LSE = s_0."""
    w = mi.make_workload("one", batch=1, num_heads=3, q_lens=[5], kv_lens=[5],
                         kv_dtype="fp8", causal=True, seed=13, num_slots=8)
    O, L = mo.mla_decode_workload(w)
    k = formats.decode_e4m3fn(w.kv_bits[w.kv_indices[0]]) * w.kv_scale
    for h in range(3):
        q = formats.decode_bf16(w.q_bits[0, h])
        assert abs(L[0, h] - w.softmax_scale * float(np.dot(q, k))) < 1e-12
        assert np.allclose(O[0, h], k[:512], atol=1e-14)


def test_empty_rows():
    w = mi.make_workload("e", batch=3, num_heads=2, q_lens=[2, 0, 1], kv_lens=[0, 5, 3],
                         kv_dtype="bf16", causal=False, seed=3, num_slots=16)
    O, L = mo.mla_decode_workload(w)
    assert np.all(np.isneginf(L[0:2])) and np.all(O[0:2] == 0)
    assert np.all(np.isfinite(L[2]))


# ---------------------------------------------------------------- invariants

def test_causal_T1_equals_noncausal():
    w = mi.make_workload("t1", batch=3, num_heads=4, q_lens=[1, 1, 1], kv_lens=[5, 64, 130],
                         kv_dtype="fp8", causal=True, seed=17, num_slots=256)
    import dataclasses
    O1, L1 = mo.mla_decode_workload(w)
    O2, L2 = mo.mla_decode_workload(dataclasses.replace(w, causal=False))
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_last_causal_token_sees_everything():
    import dataclasses
    w = mi.make_workload("lt", batch=2, num_heads=4, q_lens=[4, 8], kv_lens=[33, 70],
                         kv_dtype="bf16", causal=True, seed=19, num_slots=128)
    O1, L1 = mo.mla_decode_workload(w)
    O2, L2 = mo.mla_decode_workload(dataclasses.replace(w, causal=False))
    for b in range(2):
        last = w.qo_indptr[b + 1] - 1
        assert np.array_equal(O1[last], O2[last])
        first = w.qo_indptr[b]
        assert not np.allclose(L1[first], L2[first])


def test_noncausal_block_equals_flattened_rows():
    """A non-causal T-token block equals T single-token rows over the same KV
    ("[ROCm][Spec Decode] Add Aiter MLA decode support non-causal draft block", Purpose)."""
    w = mi.draft_block_bf16(scale=1 / 64)
    O1, L1 = mo.mla_decode_workload(w)
    O2, L2 = mo.mla_decode_workload(mi.flatten_block(w))
    assert np.allclose(O1, O2, atol=1e-13) and np.allclose(L1, L2, atol=1e-13)


def test_split_and_merge_equals_unsplit():
    import dataclasses
    w = mi.make_workload("sm", batch=2, num_heads=4, q_lens=[3, 2], kv_lens=[100, 257],
                         kv_dtype="bf16", causal=False, seed=23, num_slots=512)
    O, L = mo.mla_decode_workload(w)
    rng = np.random.default_rng(0)
    for b in range(2):
        k0, k1 = int(w.kv_indptr[b]), int(w.kv_indptr[b + 1])
        cuts = np.sort(rng.choice(np.arange(1, k1 - k0), size=4, replace=False))
        bounds = [0, *cuts.tolist(), k1 - k0]
        parts_o, parts_l = [], []
        q0, q1 = int(w.qo_indptr[b]), int(w.qo_indptr[b + 1])
        for a, c in zip(bounds[:-1], bounds[1:]):
            sub = dataclasses.replace(
                w, kv_indptr=np.array([0, c - a], np.int32),
                kv_indices=w.kv_indices[k0 + a:k0 + c], qo_indptr=np.array([0, q1 - q0], np.int32),
                q_bits=w.q_bits[q0:q1])
            o, l = mo.mla_decode_workload(sub)
            parts_o.append(o.reshape(-1, 512))
            parts_l.append(l.reshape(-1))
        # an empty part must not change anything
        parts_o.append(np.zeros_like(parts_o[0]))
        parts_l.append(np.full_like(parts_l[0], -np.inf))
        om, lm = mo.merge_states(np.stack(parts_o), np.stack(parts_l))
        assert np.allclose(om, O[q0:q1].reshape(-1, 512), atol=1e-12)
        assert np.allclose(lm, L[q0:q1].reshape(-1), atol=1e-12)


def test_cp_round_robin_shards_merge_to_unsharded():
    """Round-robin shards merged by LSE equal the unsharded result
    ("Speculative decode + DCP on gfx1250", Problem)."""
    sw = mi.cp_shards_bf16(scale=1 / 256)   # Lg = 128 -> 8 shards of 16
    Of, Lf = mo.mla_decode_workload(sw.full)
    Os, Ls = mo.mla_decode_workload(sw.shards)
    R = sw.full.total_q * sw.full.num_heads
    om, lm = mo.merge_states(Os.reshape(sw.num_shards, R, 512), Ls.reshape(sw.num_shards, R))
    assert np.allclose(om, Of.reshape(R, 512), atol=1e-12)
    assert np.allclose(lm, Lf.reshape(R), atol=1e-12)


def test_mask_is_live():
    """Causal and non-causal results differ by far more than the GPU tolerance
    (the pages saw 6e-2 to 9e-2 between a masked and an unmasked block,
    "[ROCm][Spec Decode] ...", Test Result)."""
    import dataclasses
    w = mi.verify_fp8(scale=1 / 32)
    w2 = dataclasses.replace(w, causal=False)
    O1, _ = mo.mla_decode_workload(w, requests=[0, 1])
    O2, _ = mo.mla_decode_workload(w2, requests=[0, 1])
    m = ~np.isnan(O1)
    assert np.abs(O1[m] - O2[m]).max() > 0.1


def test_identical_query_rows_identical_outputs():
    w = mi.make_workload("id", batch=2, num_heads=4, q_lens=[4, 4], kv_lens=[50, 50],
                         kv_dtype="fp8", causal=False, seed=29, num_slots=128,
                         identical_q_rows=True)
    O, L = mo.mla_decode_workload(w)
    for b in range(2):
        blk = O[w.qo_indptr[b]:w.qo_indptr[b + 1]].reshape(-1, 512)
        assert np.all(blk == blk[0][None])


# ---------------------------------------------------------------- merge closed forms

def test_merge_closed_forms():
    o = np.random.default_rng(2).standard_normal((2, 5, 8))
    lse = np.array([[0.3] * 5, [0.3] * 5])
    om, lm = mo.merge_states(o, lse)
    assert np.allclose(om, o.mean(axis=0)) and np.allclose(lm, 0.3 + math.log(2))
    om, lm = mo.merge_states(o[:1], lse[:1])
    assert np.array_equal(om, o[0]) and np.array_equal(lm, lse[0])
    om, lm = mo.merge_states(o, np.full((2, 5), -np.inf))
    assert np.all(om == 0) and np.all(np.isneginf(lm))
    # weights e^a : e^b
    lse2 = np.array([[0.0] * 5, [math.log(3.0)] * 5])
    om, lm = mo.merge_states(o, lse2)
    assert np.allclose(om, 0.25 * o[0] + 0.75 * o[1]) and np.allclose(lm, math.log(4.0))


# ---------------------------------------------------------------- plan spec

def _check_plan_case(c):
    buf = po.build_plan(c["batch"], c["num_heads"], c["max_q_len"], c["num_workers"],
                        c["kv_len_cap"], c["mode"],
                        None if c["kv_indptr"] is None else np.array(c["kv_indptr"]),
                        np.array(c["qo_indptr"]), rows=c["rows"], block_n=c["block_n"])
    p = po.parse_plan(buf)
    assert p["magic"] == po.MAGIC and p["version"] == po.VERSION
    assert list(p["splits"]) == c["splits"]
    assert list(p["group_base"]) == c["group_base"]
    assert list(p["partial_base"]) == c["partial_base"]
    assert p["n_partials"] == c["n_partials"]
    if "items" in c:
        assert p["items"].tolist() == c["items"]
    else:
        assert p["n_items"] == c["items_count"]
        assert p["items"][:4].tolist() == c["first_items"]
        assert p["items"][-1].tolist() == c["last_item"]


def test_plan_worked_examples():
    cases = json.load(open(os.path.join(GOLDEN, "plan_worked_examples.json")))["cases"]
    for c in cases:
        _check_plan_case(c)


@pytest.mark.parametrize("seed", range(20))
def test_plan_properties(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(0, 40))
    H = int(rng.choice([1, 16, 64, 96, 128]))
    maxT = int(rng.integers(1, 9))
    W = int(rng.integers(1, 300))
    mode = int(rng.integers(0, 2))
    T = rng.integers(0, maxT + 1, size=B)
    L = np.floor(np.exp(rng.uniform(0, math.log(200000), size=B))).astype(np.int64)
    L[rng.random(B) < 0.1] = 0
    cap = int(rng.integers(0, 100000))
    kvp = np.concatenate([[0], np.cumsum(L)]).astype(np.int64)
    qop = np.concatenate([[0], np.cumsum(T)]).astype(np.int64)
    p = po.parse_plan(po.build_plan(B, H, maxT, W, cap, mode, kvp, qop))
    assert p["n_items"] <= W + int(sum(po.cdiv(H * t, po.ROWS) for t in T))
    S = p["splits"]
    assert np.all((S >= 1) & (S <= po.MAX_SPLITS))
    # every (b, g) is covered by exactly S_b items, one per split
    seen = {}
    for b, s, g, slot in p["items"].tolist():
        seen.setdefault((b, g), []).append(s)
        if S[b] > 1:
            G_b = p["group_base"][b + 1] - p["group_base"][b]
            assert slot == p["partial_base"][b] + s * G_b + g
        else:
            assert slot == -1
    for b in range(B):
        G = po.cdiv(H * int(T[b]), po.ROWS)
        for g in range(G):
            assert sorted(seen[(b, g)]) == list(range(S[b]))
    slots = [x for x in p["items"][:, 3].tolist() if x >= 0]
    assert sorted(slots) == list(range(p["n_partials"]))
    # the splits of a real length tile [0, L) with no gap or overlap
    for b in range(B):
        e = 0
        for s in range(S[b]):
            a, c = po.split_tile_range(s, int(S[b]), int(L[b]))
            assert a == e and c >= a
            e = c
        assert e == int(L[b])


def test_split_ranges_of_the_256_row_worked_example():
    """Hand-worked: 4000 entries in 128-entry tiles (32 tiles) split in two."""
    assert po.split_tile_range(0, 2, 4000, block_n=128) == (0, 2048)
    assert po.split_tile_range(1, 2, 4000, block_n=128) == (2048, 4000)
    assert po.split_tile_range(0, 1, 1000, block_n=128) == (0, 1000)


def test_plan_rejects_bad_input():
    with pytest.raises(ValueError):
        po.build_plan(2, 16, 2, 4, 0, po.DYNAMIC, np.array([0, 5, 3]), np.array([0, 1, 2]))
    with pytest.raises(ValueError):
        po.build_plan(2, 16, 1, 4, 0, po.DYNAMIC, np.array([0, 5, 9]), np.array([0, 2, 3]))
    with pytest.raises(ValueError):
        po.build_plan(2, 16, 2, 0, 0, po.DYNAMIC, np.array([0, 5, 9]), np.array([0, 1, 2]))


# ---------------------------------------------------------------- planted mistakes

def test_pins_catch_an_off_by_one_causal_limit(monkeypatch):
    """Plant an off-by-one in the oracle's mask; the closed-form pin must fail."""
    orig = mo.visible_mask

    def wrong(L, T, t_of_row, causal, base, stride, Lg, pos=None, window=0):
        return orig(L, T, t_of_row, causal, base, stride, Lg - 1, pos, window)

    monkeypatch.setattr(mo, "visible_mask", wrong)
    with pytest.raises(AssertionError):
        test_zero_query_gives_mean_and_log_count()


def test_pins_catch_a_dropped_rope_part(monkeypatch):
    """Plant a QK over the 512 latent dims only; the brute-force pin must fail."""
    orig = mo.attend_rows

    def wrong(qrows, K, vis, sigma):
        K2 = K.copy()
        K2[:, 512:] = 0
        return orig(qrows, K2, vis, sigma)

    monkeypatch.setattr(mo, "attend_rows", wrong)
    with pytest.raises(AssertionError):
        test_brute_force_tiny("bf16")


def test_pins_catch_a_missing_kv_scale(monkeypatch):
    orig = formats.decode_kv
    monkeypatch.setattr(mo, "decode_kv", lambda bits, dt: orig(bits, dt) / (20.0 if dt == "fp8" else 1))
    with pytest.raises(AssertionError):
        test_single_visible_entry()
