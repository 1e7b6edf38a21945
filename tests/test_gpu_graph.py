"""CUDA-graph capture and replay with changing lengths (the re-planning path).

The persistent kernel re-plans the split from the real per-row KV lengths at every
call, so a graph captured once stays correct while the KV grows ("[DSV4] Tuned ASM
FP8 decode with split plans; HCA on aiter's persistent V4-NM kernel", Summary
part 2).  The graph holds [device planner, decode]; between replays the
index lists and query block are rewritten in place in buffers sized for capacity.
"""
import numpy as np
import pytest

import mla_inputs as mi
from oracle import mla_oracle as mo
from tests import harness as hz

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import token_mla_paged_gb300 as m  # noqa: E402


def _capacity_buffers(B, H, max_T, num_slots):
    max_nnz = num_slots            # every replay's index list fits the pool
    max_q = B * max_T
    dev = dict(
        q=torch.zeros(max_q, H, 576, dtype=torch.bfloat16, device="cuda"),
        kv_indptr=torch.zeros(B + 1, dtype=torch.int32, device="cuda"),
        kv_indices=torch.zeros(max_nnz, dtype=torch.int32, device="cuda"),
        qo_indptr=torch.zeros(B + 1, dtype=torch.int32, device="cuda"),
    )
    o = torch.zeros(max_q, H, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(max_q, H, dtype=torch.float32, device="cuda")
    return dev, o, lse


def _load(dev, w):
    dev["q"][: w.total_q].copy_(torch.from_numpy(w.q_bits.view(np.int16)).view(torch.bfloat16))
    dev["kv_indptr"].copy_(torch.from_numpy(w.kv_indptr))
    dev["kv_indices"][: w.kv_indices.shape[0]].copy_(torch.from_numpy(w.kv_indices))
    dev["qo_indptr"].copy_(torch.from_numpy(w.qo_indptr))


@pytest.mark.parametrize("algo", [m.MLA_ALGO_TENSOR, m.MLA_ALGO_CUDA_CORE], ids=["tensor", "cuda_core"])
@pytest.mark.parametrize("scale", [1 / 64, 1.0], ids=["small", "full"])
def test_graph_replay_with_changing_lengths(algo, scale):
    if algo == m.MLA_ALGO_CUDA_CORE and scale == 1.0:
        pytest.skip("full-size replays checked on the tensor kernel")
    replays = 5
    slots = mi.long_skewed_pool_slots(replays, scale=scale)
    # each replay brings fresh lengths, T, indices and cache contents (pool sized for
    # all); the workloads are drawn one at a time to bound host memory
    w0 = mi.long_skewed_fp8(replay=0, scale=scale, num_slots=slots)
    B, H = w0.batch, w0.num_heads
    dev, o, lse = _capacity_buffers(B, H, 4, slots)
    pool = torch.zeros(slots, 576, dtype=torch.uint8, device="cuda")
    runner = m.DecodeRunner(B, H, 4, mode=m.MLA_PLAN_DYNAMIC, num_workers=76)
    kw = dict(kv_pool=pool.view(torch.float8_e4m3fn), kv_dtype=m.MLA_KV_FP8_E4M3, causal=True,
              softmax_scale=w0.softmax_scale, kv_scale=w0.kv_scale)
    _load(dev, w0)
    pool.copy_(torch.from_numpy(w0.kv_bits))
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        runner.forward(o=o, lse=lse, algo=algo, **dev, **kw)       # warm-up outside capture
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        runner.forward(o=o, lse=lse, algo=algo, **dev, **kw)
    outs = []
    for r in range(replays):
        w = w0 if r == 0 else mi.long_skewed_fp8(replay=r, scale=scale, num_slots=slots)
        _load(dev, w)
        pool.copy_(torch.from_numpy(w.kv_bits))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert m.mla_get_device_error(runner.workspace) == (0, 0)
        O = o[: w.total_q].double().cpu().numpy()
        L = lse[: w.total_q].double().cpu().numpy()
        reqs = None if scale < 1 else hz.sample_requests(w, 3, seed=r)
        Oref, Lref = mo.mla_decode_workload(w, requests=reqs)
        rows = None if reqs is None else hz.rows_of(w, reqs)
        hz.assert_close(O, L, Oref, Lref, "fp8", rows=rows, what=f"replay {r}")
        outs.append((O.copy(), L.copy()))
    # replaying the last lengths again gives bitwise the same result
    graph.replay()
    torch.cuda.synchronize()
    assert np.array_equal(o[: w.total_q].double().cpu().numpy(), outs[-1][0])
    assert np.array_equal(lse[: w.total_q].double().cpu().numpy(), outs[-1][1])
