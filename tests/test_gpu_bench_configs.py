"""Parity at full size in the launch configuration the benchmark times.

Each decode workload is built exactly as `bench.py` builds it (same workload
function and seed, plan mode, KV capacity and worker count), run once through the C
ABI, and checked on whole sampled requests against the float64 oracle; the tiny
workload is checked in full.  For the context-parallel workload the per-shard states
are merged as the benchmark merges them (bf16 shard outputs) and the merged result is
checked against the oracle of the unsharded problem.
"""
import numpy as np
import pytest

import bench
import mla_inputs as mi
from oracle import mla_oracle as mo
from tests import harness as hz

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped there
    pytest.skip("needs a GPU", allow_module_level=True)

import token_mla_paged_gb300 as m  # noqa: E402


def _bench_run(config: str):
    w, extra = bench.build_workload(config)
    if config == "long_skewed_fp8":
        w = mi.long_skewed_fp8(replay=0, num_slots=mi.long_skewed_pool_slots(bench.REPLAYS_LONG))
    torch.cuda.set_device(0)
    algo = m.MLA_ALGO_TENSOR
    workers = bench.decode_workers(config, w, algo, 0)
    maxq = int(w.q_lens().max())
    runner = m.DecodeRunner(w.batch, w.num_heads, maxq, mode=extra["mode"], num_workers=workers,
                            kv_len_cap=extra["cap"])
    if extra["mode"] == m.MLA_PLAN_STATIC:
        runner.set_host_plan(None, w.qo_indptr)
    elif extra["mode"] == m.MLA_PLAN_HOST:
        runner.set_host_plan(w.kv_indptr, w.qo_indptr)
    dev = mi.to_device(w)
    o = torch.full((w.total_q, w.num_heads, 512), float("nan"), device="cuda", dtype=torch.bfloat16)
    lse = torch.full((w.total_q, w.num_heads), float("nan"), device="cuda", dtype=torch.float32)
    runner.forward(o=o, lse=lse, algo=algo, **dev)
    torch.cuda.synchronize()
    assert hz.device_error(runner) == (0, 0)
    return w, extra, o, lse


@pytest.mark.parametrize("config", ["draft_block_bf16", "verify_fp8", "long_skewed_fp8", "csa_topk_fp8",
                                    "hca_fp8", "tiny_causal_bf16"])
def test_bench_workload_matches_oracle(config):
    w, _, o, lse = _bench_run(config)
    reqs = None if config == "tiny_causal_bf16" else hz.sample_requests(w, 3, seed=11)
    Oref, Lref = mo.mla_decode_workload(w, requests=reqs)
    rows = None if reqs is None else hz.rows_of(w, reqs)
    hz.assert_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), Oref, Lref, w.kv_dtype,
                    rows=rows, what=config)


def test_bench_cp_shards_merged_matches_unsharded_oracle():
    w, extra, o, lse = _bench_run("cp_shards_bf16")
    sw = extra["shards"]
    R = sw.full.total_q * sw.full.num_heads
    om = torch.empty(R, 512, dtype=torch.bfloat16, device="cuda")
    lm = torch.empty(R, dtype=torch.float32, device="cuda")
    m.mla_merge_states(o.view(sw.num_shards, R, 512), lse.view(sw.num_shards, R), om, lm)
    torch.cuda.synchronize()
    reqs = hz.sample_requests(sw.full, 2, seed=5)
    Oref, Lref = mo.mla_decode_workload(sw.full, requests=reqs)
    H = sw.full.num_heads
    O = om.view(sw.full.total_q, H, 512).double().cpu().numpy()
    L = lm.view(sw.full.total_q, H).double().cpu().numpy()
    hz.assert_close(O, L, Oref, Lref, "bf16", rows=hz.rows_of(sw.full, reqs), what="cp_shards merged")
