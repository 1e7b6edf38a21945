"""The device failure path: a bounded barrier wait that runs out.

Every barrier wait in the tensor-core decode kernel gives up after a limit and
records MLA_DEV_WAIT_TIMEOUT (with the wait's site) in the workspace error word;
the kernel then raises an abort flag in every CTA of its cluster, frees its TMEM
and leaves, so the context stays usable.  The test hook MLA_TEST_STALL_CYCLES=n
makes every warp wait, before any copy or MMA is issued, on a barrier nothing
signals, with a limit of n cycles -- the wait runs out with nothing in flight.
The test checks the recorded error and that the next call, without the hook, is
correct against the oracle.
"""
import os

import pytest

import mla_inputs as mi
from oracle import mla_oracle as mo
from tests import harness as hz

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import token_mla_paged_gb300 as m  # noqa: E402


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_wait_timeout_is_recorded_and_the_context_survives(kv_dtype):
    w = mi.make_workload("stall", batch=3, num_heads=64, q_lens=[4, 2, 3], kv_lens=[700, 150, 1200],
                         kv_dtype=kv_dtype, causal=True, seed=91, num_slots=4096)
    dev = mi.to_device(w)
    os.environ["MLA_TEST_STALL_CYCLES"] = "20000"
    try:
        _, _, runner = hz.run(w, algo=m.MLA_ALGO_TENSOR, dev=dev, num_workers=8)
    finally:
        del os.environ["MLA_TEST_STALL_CYCLES"]
    code, info = hz.device_error(runner)
    assert (code, info) == (5, 99)
    assert hz.device_error(runner) == (0, 0)          # read and cleared
    O, L, _ = hz.run(w, algo=m.MLA_ALGO_TENSOR, dev=dev, runner=runner)
    assert hz.device_error(runner) == (0, 0)
    Oref, Lref = mo.mla_decode_workload(w)
    hz.assert_close(O, L, Oref, Lref, kv_dtype, what="call after the timeout")
