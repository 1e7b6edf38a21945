"""GPU test helpers: run a workload through the C ABI and compare with the oracle."""
from __future__ import annotations

import numpy as np

import mla_inputs as mi

TOL = {"bf16": (1e-2, 1e-2), "fp8": (3e-2, 3e-2)}   # (atol, rtol) on O
LSE_TOL = 2e-3


def run(w: mi.Workload, *, algo: int, mode: int = 1, num_workers=None, kv_len_cap: int = 0,
        out_fp32: bool = False, runner=None, dev=None, o=None, lse=None):
    """One forward call; returns (O float64 [total_q,H,512], LSE float64 [total_q,H], runner)."""
    import torch
    import token_mla_paged_gb300 as m
    if dev is None:
        dev = mi.to_device(w)
    H = w.num_heads
    if runner is None:
        maxq = int(max(1, w.q_lens().max(initial=0)))
        runner = m.DecodeRunner(w.batch, H, maxq, mode=mode, num_workers=num_workers,
                                kv_len_cap=kv_len_cap)
        if mode == m.MLA_PLAN_STATIC:
            runner.set_host_plan(None, w.qo_indptr)
        elif mode == m.MLA_PLAN_HOST:
            runner.set_host_plan(w.kv_indptr, w.qo_indptr)
    if o is None:
        o = torch.full((w.total_q, H, 512), float("nan"), device="cuda",
                       dtype=torch.float32 if out_fp32 else torch.bfloat16)
        lse = torch.full((w.total_q, H), float("nan"), device="cuda", dtype=torch.float32)
    runner.forward(o=o, lse=lse, algo=algo, **dev)
    torch.cuda.synchronize()
    return o.double().cpu().numpy(), lse.double().cpu().numpy(), runner


def device_error(runner):
    import token_mla_paged_gb300 as m
    return m.mla_get_device_error(runner.workspace)


def assert_close(O, L, Oref, Lref, kv_dtype: str, rows=None, what=""):
    """Elementwise |o - o*| <= atol + rtol |o*|; |lse - lse*| <= 2e-3; empty rows exact."""
    atol, rtol = TOL[kv_dtype]
    if rows is not None:
        O, L, Oref, Lref = O[rows], L[rows], Oref[rows], Lref[rows]
    assert not np.isnan(Lref).any(), "reference rows missing"
    empty = np.isneginf(Lref)
    assert np.array_equal(np.isneginf(L), empty), f"{what}: empty-row pattern differs"
    assert np.all(O[empty] == 0), f"{what}: empty rows must be zero"
    full = ~empty
    dl = np.abs(L[full] - Lref[full])
    assert dl.size == 0 or dl.max() <= LSE_TOL, f"{what}: LSE err {dl.max():.3e}"
    err = np.abs(O[full] - Oref[full])
    bound = atol + rtol * np.abs(Oref[full])
    worst = (err - bound).max() if err.size else -1
    assert worst <= 0, (f"{what}: O err max {err.max():.3e} exceeds tolerance "
                        f"(atol {atol}, rtol {rtol})")
    return float(err.max()) if err.size else 0.0, float(dl.max()) if dl.size else 0.0


def sample_requests(w: mi.Workload, k: int, seed: int = 0):
    """A few requests to check with the oracle: the longest, the shortest, random others."""
    lens = w.kv_lens()
    rng = np.random.default_rng(seed)
    pick = {int(np.argmax(lens)), int(np.argmin(lens))}
    while len(pick) < min(k, w.batch):
        pick.add(int(rng.integers(w.batch)))
    return sorted(pick)


def rows_of(w: mi.Workload, reqs):
    return np.concatenate([np.arange(w.qo_indptr[b], w.qo_indptr[b + 1]) for b in reqs])
