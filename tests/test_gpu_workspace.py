"""Workspace state across calls.

No call clears the workspace: it is zero-filled once when allocated, and every
call that completes leaves its queue words (header words 2-3) and split-merge
counters (from byte 256 on, as many words as header word 4 says) at zero again.
After a fault, reading the error zeroes what the faulted call may have left set.
The fault here is planted on the host (the error word and dirty counters written
into the workspace), so no kernel is made to fail.
"""
import numpy as np
import pytest

import mla_inputs as mi
from oracle import mla_oracle as mo
from tests import harness as hz

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped there
    pytest.skip("needs a GPU", allow_module_level=True)

import token_mla_paged_gb300 as m  # noqa: E402

H_NPARTIALS = 8          # plan header word: number of split partials
WS_COUNTER_WORDS = 4     # workspace header word: counter words of the last call
COUNTERS_WORD0 = 64      # the counters start at byte 256


def _state(runner):
    ws = runner.workspace.cpu().numpy()
    n = int(ws[WS_COUNTER_WORDS])
    return ws[2:4].copy(), ws[COUNTERS_WORD0:COUNTERS_WORD0 + n].copy(), n


@pytest.mark.parametrize("algo", [m.MLA_ALGO_CUDA_CORE, m.MLA_ALGO_TENSOR], ids=["cuda_core", "tensor"])
def test_calls_leave_the_state_at_zero(algo):
    """Three calls of a split plan on one workspace, nothing cleared in between:
    each matches the oracle and leaves the queue words and counters at zero."""
    w = mi.verify_fp8(scale=1 / 16)
    dev = mi.to_device(w)
    Oref, Lref = mo.mla_decode_workload(w)
    runner = None
    for _ in range(3):
        O, L, runner = hz.run(w, algo=algo, mode=1, num_workers=608, runner=runner, dev=dev)
        assert hz.device_error(runner) == (0, 0)
        hz.assert_close(O, L, Oref, Lref, w.kv_dtype, what=w.name)
        assert int(runner.plan_d[H_NPARTIALS]) > 0, "the plan must split for this test to mean anything"
        queue, counters, n = _state(runner)
        g_max = -(-w.num_heads * int(w.q_lens().max()) // 256)
        assert n == 2 * w.batch * g_max
        assert not queue.any() and not counters.any()


def test_reading_a_fault_clears_the_state():
    w = mi.tiny_causal_bf16()
    dev = mi.to_device(w)
    O, L, runner = hz.run(w, algo=m.MLA_ALGO_TENSOR, dev=dev)
    n = int(runner.workspace[WS_COUNTER_WORDS])
    assert n > 0
    # what a call stopped by a fault may leave behind
    runner.workspace[2:4] = 7
    runner.workspace[COUNTERS_WORD0:COUNTERS_WORD0 + n] = 3
    runner.workspace[0] = 5
    runner.workspace[1] = 99
    assert m.mla_get_device_error(runner.workspace) == (5, 99)
    ws = runner.workspace.cpu().numpy()
    assert not ws[:COUNTERS_WORD0 + n].any()
    O2, L2, _ = hz.run(w, algo=m.MLA_ALGO_TENSOR, runner=runner, dev=dev)
    Oref, Lref = mo.mla_decode_workload(w)
    hz.assert_close(O2, L2, Oref, Lref, w.kv_dtype, what=w.name)


@pytest.mark.parametrize("algo", [m.MLA_ALGO_CUDA_CORE, m.MLA_ALGO_TENSOR], ids=["cuda_core", "tensor"])
def test_back_to_back_calls_with_changing_lengths(algo):
    """Six DYNAMIC calls queued on one stream with no synchronisation between them,
    on one plan buffer and workspace, each with other lengths, T and indices: the
    planner of a call may start while the previous call's decode still runs (an
    overlapped launch) and must not rewrite the plan before that decode is done.
    Every call's output matches the oracle."""
    slots = mi.long_skewed_pool_slots(3, scale=1 / 64)
    ws = [mi.long_skewed_fp8(replay=r, scale=1 / 64, num_slots=slots) for r in range(3)]
    devs = [mi.to_device(w) for w in ws]
    maxq = max(int(w.q_lens().max()) for w in ws)
    runner = m.DecodeRunner(ws[0].batch, ws[0].num_heads, maxq, mode=m.MLA_PLAN_DYNAMIC, num_workers=76)
    outs = []
    for k in range(6):
        w, dev = ws[k % 3], devs[k % 3]
        o = torch.full((w.total_q, w.num_heads, 512), float("nan"), device="cuda", dtype=torch.bfloat16)
        lse = torch.full((w.total_q, w.num_heads), float("nan"), device="cuda", dtype=torch.float32)
        runner.forward(o=o, lse=lse, algo=algo, **dev)
        outs.append((k % 3, o, lse))
    torch.cuda.synchronize()
    assert hz.device_error(runner) == (0, 0)
    refs = [mo.mla_decode_workload(w) for w in ws]
    for r, o, lse in outs:
        hz.assert_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), *refs[r], "fp8",
                        what=f"call of draw {r}")
    queue, counters, _ = _state(runner)
    assert not queue.any() and not counters.any()
