"""The allocation-free forward entry point (mla_decode_fwd_noalloc).

Some callers of this library cannot allocate device memory themselves: a
framework or runtime that owns the device allocator and hands the kernel only
its input and output tensors.  For them the library keeps its plan buffer and
workspace in one static device array.  This test calls that entry point through
the C ABI and checks its output against the float64 oracle and against the
regular entry point (which uses a caller-allocated plan and workspace) on the
same inputs, within the parity tolerance of the other GPU tests, on two calls in
a row (the second call sees the first call's leftovers in the shared array).

The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import mla_inputs as mi
from oracle import mla_oracle as mo

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import token_mla_paged_gb300 as m  # noqa: E402
from tests import harness as hz  # noqa: E402


def _args(dev, w, o, lse, params):
    a = m.FwdArgs()
    a.q = dev["q"].data_ptr()
    a.kv_pool = dev["kv_pool"].data_ptr()
    a.num_slots = int(dev["kv_pool"].shape[0])
    a.kv_dtype = dev["kv_dtype"]
    a.out_dtype = m.MLA_OUT_BF16
    a.kv_indptr = dev["kv_indptr"].data_ptr()
    a.kv_indices = dev["kv_indices"].data_ptr()
    a.qo_indptr = dev["qo_indptr"].data_ptr()
    a.causal = 1 if w.causal else 0
    a.pos_base = w.pos_base
    a.pos_stride = w.pos_stride
    a.algo = m.MLA_ALGO_TENSOR
    a.pos_base_per_req = None
    a.g_kv_indptr = None
    a.softmax_scale = w.softmax_scale
    a.kv_scale = w.kv_scale
    a.o = o.data_ptr()
    a.lse = lse.data_ptr()
    a.params = ctypes.pointer(params)
    a.plan_d = None
    a.plan_bytes = 0
    a.workspace_d = None
    a.ws_bytes = 0
    return a


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_noalloc_matches_regular_entry_point(kv_dtype):
    lib = m.library()
    # several row groups, causal, with split-merged rows (few workers -> splits)
    w = mi.make_workload("noalloc", batch=3, num_heads=64, q_lens=[4, 2, 3], kv_lens=[3000, 150, 1200],
                         kv_dtype=kv_dtype, causal=True, seed=71, num_slots=8192)
    dev = mi.to_device(w)
    H = w.num_heads
    # regular entry point: caller-owned plan and workspace
    O_ref, L_ref, _ = hz.run(w, algo=m.MLA_ALGO_TENSOR, mode=m.MLA_PLAN_DYNAMIC, num_workers=24, dev=dev)
    O_or, L_or = mo.mla_decode_workload(w)
    hz.assert_close(O_ref, L_ref, O_or, L_or, kv_dtype, what="regular entry point")
    params = m.plan_params(w.batch, H, int(w.q_lens().max()), 24, 0, m.MLA_PLAN_DYNAMIC)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        o = torch.full((w.total_q, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((w.total_q, H), float("nan"), dtype=torch.float32, device="cuda")
        st = lib.mla_decode_fwd_noalloc(ctypes.byref(_args(dev, w, o, lse, params)), stream)
        assert st == 0, m.mla_status_string(st)
        torch.cuda.synchronize()
        O = o.double().cpu().numpy()
        L = lse.double().cpu().numpy()
        hz.assert_close(O, L, O_or, L_or, kv_dtype, what=f"noalloc call {call} vs oracle")
        hz.assert_close(O, L, O_ref, L_ref, kv_dtype, what=f"noalloc call {call} vs regular entry point")


def test_noalloc_rejects_static_mode_and_oversized_problems():
    lib = m.library()
    w = mi.tiny_causal_bf16()
    dev = mi.to_device(w)
    o = torch.empty(w.total_q, w.num_heads, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.total_q, w.num_heads, dtype=torch.float32, device="cuda")
    static = m.plan_params(w.batch, w.num_heads, 2, 8, 128, m.MLA_PLAN_STATIC)
    assert lib.mla_decode_fwd_noalloc(ctypes.byref(_args(dev, w, o, lse, static)), None) == 2
    huge = m.plan_params(w.batch, w.num_heads, 2, 5000, 0, m.MLA_PLAN_DYNAMIC)   # 5000 partial slots
    assert lib.mla_decode_fwd_noalloc(ctypes.byref(_args(dev, w, o, lse, huge)), None) == 3
