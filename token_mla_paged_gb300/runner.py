"""Buffer plumbing around the C ABI: allocates the plan and workspace with torch
and issues the calls.  No attention arithmetic happens here."""
from __future__ import annotations

from typing import Optional

import numpy as np

from . import (MLA_ALGO_TENSOR, MLA_PLAN_DYNAMIC, MLA_PLAN_HOST, MLA_PLAN_STATIC, mla_decode_fwd,
               mla_decode_plan, mla_decode_plan_size, mla_decode_workers, plan_params)


def default_workers(device=None, algo: int = MLA_ALGO_TENSOR) -> int:
    """Work items the decode kernel runs at once on the device: the plan splits
    long rows to give about this many items."""
    import torch
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        return mla_decode_workers(algo)


def default_workers_for(algo: int, batch: int, num_heads: int, max_q_len: int, device=None) -> int:
    """Plan workers for a shape: the tensor kernel runs one work item per
    four-SM cluster, the CUDA-core kernel one per SM."""
    return default_workers(device, algo)


class DecodeRunner:
    """Owns one plan buffer and one workspace sized for `params`.

    STATIC mode: call ``set_host_plan`` once (outside any graph) with the host
    qo_indptr (kv_indptr unused); the plan is uploaded and then only read.
    HOST mode: call ``set_host_plan`` with host copies of kv_indptr / qo_indptr
    whenever the lengths change; the plan is built from the real lengths.
    DYNAMIC mode: every ``forward`` re-plans on the device.
    """

    def __init__(self, batch: int, num_heads: int, max_q_len: int, *, mode: int = MLA_PLAN_DYNAMIC,
                 num_workers: Optional[int] = None, kv_len_cap: int = 0, device="cuda"):
        import torch
        self.device = torch.device(device)
        if num_workers is None:
            num_workers = default_workers(self.device)
        self.params = plan_params(batch, num_heads, max_q_len, num_workers, kv_len_cap, mode)
        plan_bytes, ws_bytes = mla_decode_plan_size(self.params)
        self.plan_d = torch.zeros(plan_bytes // 4, dtype=torch.int32, device=self.device)
        self.workspace = torch.zeros((ws_bytes + 3) // 4, dtype=torch.int32, device=self.device)
        self.host_plan: Optional[np.ndarray] = None

    def set_host_plan(self, kv_indptr_h: Optional[np.ndarray], qo_indptr_h: np.ndarray) -> np.ndarray:
        import torch
        assert self.params.mode in (MLA_PLAN_STATIC, MLA_PLAN_HOST)
        plan = mla_decode_plan(self.params, kv_indptr_h, qo_indptr_h)
        self.plan_d.copy_(torch.from_numpy(plan))
        self.host_plan = plan
        return plan

    def forward(self, *, q, kv_pool, kv_dtype: int, kv_indptr, kv_indices, qo_indptr, causal: bool,
                softmax_scale: float, kv_scale: float, o, lse, pos_base: int = 0,
                pos_stride: int = 1, pos_base_per_req=None, g_kv_indptr=None,
                algo: int = MLA_ALGO_TENSOR, kv_pos=None, window: int = 0, stream=None) -> None:
        mla_decode_fwd(q=q, kv_pool=kv_pool, kv_dtype=kv_dtype, kv_indptr=kv_indptr,
                       kv_indices=kv_indices, qo_indptr=qo_indptr, causal=causal,
                       softmax_scale=softmax_scale, kv_scale=kv_scale, o=o, lse=lse,
                       params=self.params, plan_d=self.plan_d, workspace_d=self.workspace,
                       pos_base=pos_base, pos_stride=pos_stride, pos_base_per_req=pos_base_per_req,
                       g_kv_indptr=g_kv_indptr, algo=algo, kv_pos=kv_pos, window=window,
                       stream=stream)
