"""Host arithmetic of the benchmark (CPU only): the units and bytes behind the
reported throughput and roofline.

* visible (row, entry) pairs: the benchmark's closed-form count (searchsorted over
  positions) against a brute-force count of the oracle's own visibility mask, for
  non-causal, causal, round-robin-shard and index-list (positions + window) workloads;
* algorithmic bytes of every kernel, recomputed from the tensors' shapes;
* the ncu traffic record is reported only while the kernel source it was taken from
  is unchanged.
"""
import hashlib
import json
import os

import numpy as np
import pytest

import bench
import mla_inputs as mi
from oracle import mla_oracle as mo


def _brute_pairs(w):
    tot = 0
    for b in range(w.batch):
        k0, k1 = int(w.kv_indptr[b]), int(w.kv_indptr[b + 1])
        q0, q1 = int(w.qo_indptr[b]), int(w.qo_indptr[b + 1])
        L, T = k1 - k0, q1 - q0
        if T == 0:
            continue
        base = int(w.pos_base_per_req[b]) if w.pos_base_per_req is not None else w.pos_base
        Lg = int(w.g_kv_indptr[b + 1] - w.g_kv_indptr[b]) if w.g_kv_indptr is not None else L
        vis = mo.visible_mask(L, T, np.arange(T), w.causal, base, w.pos_stride, Lg,
                              None if w.kv_pos is None else w.kv_pos[k0:k1], w.window)
        tot += int(vis.sum())
    return tot * w.num_heads


@pytest.mark.parametrize("make", [
    lambda: mi.tiny_causal_bf16(),
    lambda: mi.make_workload("nc", batch=3, num_heads=5, q_lens=[1, 7, 8], kv_lens=[9, 1, 300],
                             kv_dtype="fp8", causal=False, seed=1),
    lambda: mi.make_workload("c", batch=3, num_heads=5, q_lens=[1, 7, 8], kv_lens=[9, 3, 300],
                             kv_dtype="bf16", causal=True, seed=2),
    lambda: mi.cp_shards_bf16(scale=1 / 64).shards,
    lambda: mi.sparse_variant("swa", batch=3, num_heads=4, q_lens=[2, 2, 2], global_lens=[100, 700, 5000],
                              window=128, seed=3),
    lambda: mi.sparse_variant("csa", batch=3, num_heads=4, q_lens=[2, 2, 2], global_lens=[100, 700, 5000],
                              window=128, seed=4),
    lambda: mi.sparse_variant("hca", batch=3, num_heads=4, q_lens=[2, 2, 2], global_lens=[100, 700, 5000],
                              window=128, seed=5),
], ids=["tiny", "noncausal", "causal", "cp_shards", "swa", "csa", "hca"])
def test_visible_pairs_match_the_oracle_mask(make):
    w = make()
    assert bench.visible_pairs(w) == _brute_pairs(w)


def test_algorithmic_bytes_from_shapes():
    w = mi.make_workload("c", batch=2, num_heads=3, q_lens=[2, 1], kv_lens=[5, 4],
                         kv_dtype="fp8", causal=True, seed=9)
    q_bytes = 3 * 3 * 576 * 2                # 3 tokens x 3 heads of bf16 q
    o_bytes = 3 * 3 * (512 * 2 + 4)          # bf16 O and fp32 LSE per row
    kv_bytes = 9 * 576 * 1 + 9 * 4           # fp8 rows once, one int32 index each
    assert bench.algorithmic_bytes(w) == q_bytes + o_bytes + kv_bytes
    assert bench.cache_write_bytes(10, True) == 10 * (1152 + 576 + 4)
    assert bench.cache_write_bytes(10, False) == 10 * (1152 + 1152 + 4)
    # q_nope (512) + q_pe (64) in and q (576) out in bf16 per head; kv_c + k_pe in;
    # one fp8 row out; slot + position (int32 + int64); one fp32 cos/sin row
    assert bench.rope_cache_bytes(3, 2) == 3 * (2 * (512 * 2 + 64 * 2 + 576 * 2) + 576 * 2 + 576 + 4 + 4 + 64 * 4)
    # x (bf16) in, fp8 weight once, bf16 result out
    assert bench.absorb_bytes(256, 128, 128, 512) == 256 * 128 * 128 * 2 + 128 * 128 * 512 + 256 * 128 * 512 * 2
    assert bench.absorb_bytes(256, 128, 128, 512) == bench.absorb_bytes(256, 128, 512, 128) == 50331648


def test_ncu_traffic_only_for_the_profiled_code(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// profiled version\nint a = 1;  // one\n")
    (tmp_path / "profiles").mkdir()
    code = hashlib.sha256("int a = 1;".encode()).hexdigest()[:16]
    assert bench.kernel_code_hash(str(src)) == code
    rec = {"kernel_source": "kernel.cu", "kernel_code_sha256_16": code,
           "workloads": {"w": {"dram_bytes": 1234}}}
    (tmp_path / "profiles" / "rec.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic("w", "rec.json") == 1234
    assert bench.ncu_traffic("other", "rec.json") is None
    src.write_text("// a comment edited\n\nint a = 1;   // still one\n")
    assert bench.ncu_traffic("w", "rec.json") == 1234        # comments do not change the kernel
    src.write_text("int a = 2;\n")
    assert bench.ncu_traffic("w", "rec.json") is None


def test_committed_records_name_existing_sources():
    for name in os.listdir(os.path.join(bench.ROOT, "profiles")):
        if name.endswith(".json"):
            d = json.load(open(os.path.join(bench.ROOT, "profiles", name)))
            assert os.path.exists(os.path.join(bench.ROOT, d["kernel_source"])), name
            assert len(d["kernel_code_sha256_16"]) == 16 and d["workloads"], name
            # the committed kernel is the profiled one
            assert bench.kernel_code_hash(os.path.join(bench.ROOT, d["kernel_source"])) == d["kernel_code_sha256_16"], name
