"""The context-parallel exchange on a GPU: `cp_merge` under a one-rank NCCL group.

With one rank the all-gather returns the local state and the merge of a single
state is that state: O unchanged (bf16 in, bf16 out, weight exactly 1) and the LSE
unchanged; an empty row (LSE = -inf) comes out O = 0, LSE = -inf.  The gather layout
and rank order with two ranks are tested on host tensors in
`test_distributed_cpu.py`; the merge arithmetic with several states in
`test_gpu_parity.py`.
"""
import socket

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped there
    pytest.skip("needs a GPU", allow_module_level=True)

import torch.distributed as dist  # noqa: E402

import token_mla_paged_gb300 as m  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_cp_merge_one_rank_is_identity():
    if not dist.is_nccl_available():
        pytest.skip("no NCCL in this torch build")
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0, world_size=1)
    try:
        g = torch.Generator(device="cuda").manual_seed(5)
        rows, H = 24, 16
        o = torch.randn(rows, H, 512, device="cuda", generator=g).to(torch.bfloat16)
        lse = torch.randn(rows, H, device="cuda", generator=g)
        lse[3, 5] = float("-inf")
        o[3, 5] = 0
        out = torch.empty_like(o)
        lse_out = torch.empty_like(lse)
        m.cp_merge(o, lse, out, lse_out)
        torch.cuda.synchronize()
        assert torch.equal(out, o)
        a, b = lse_out.cpu().numpy(), lse.cpu().numpy()
        assert np.array_equal(np.isneginf(a), np.isneginf(b))
        fin = np.isfinite(b)
        assert np.abs(a[fin] - b[fin]).max() <= 1e-6
    finally:
        dist.destroy_process_group()
