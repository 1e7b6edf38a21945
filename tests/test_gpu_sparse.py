"""GPU parity for index lists with per-entry positions and a sliding window.

The DSV4 layer types ("[DSV4] Tuned ASM FP8 decode with split plans; HCA on
aiter's persistent V4-NM kernel", Summary part 1) run the same decode over
different index lists: a sliding window (SWA), a window plus top-k selected
older entries (CSA), a window plus one compressed entry per 128 tokens (HCA).
Each entry carries its global position (kv_pos); SWA also applies the window.
Both kernels are compared with the oracle, element by element, at sizes the
oracle finishes in seconds (several tiles, ragged tails, T up to 3) and on
sampled requests at a full size; the whole-KV list with a window (positions
base + i*stride, no kv_pos) is checked too.
"""
import dataclasses

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

ALGOS = [m.MLA_ALGO_TENSOR, m.MLA_ALGO_CUDA_CORE]


def _check(w, algo, reqs=None, mode=m.MLA_PLAN_DYNAMIC, num_workers=76):
    O, L, runner = hz.run(w, algo=algo, mode=mode, num_workers=num_workers)
    assert hz.device_error(runner) == (0, 0)
    Oref, Lref = mo.mla_decode_workload(w, requests=reqs)
    rows = None if reqs is None else hz.rows_of(w, reqs)
    hz.assert_close(O, L, Oref, Lref, w.kv_dtype, rows=rows, what=w.name)


@pytest.mark.parametrize("algo", ALGOS, ids=["tensor", "cuda_core"])
@pytest.mark.parametrize("kind", ["swa", "csa", "hca"])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_layer_types_small(kind, kv_dtype, algo):
    w = mi.sparse_variant(kind, batch=5, num_heads=64, q_lens=[1, 2, 3, 1, 2],
                          global_lens=[3000, 700, 150, 9000, 64], window=128, topk=300, ratio=128,
                          kv_dtype=kv_dtype, seed=41)
    _check(w, algo, num_workers=24)


@pytest.mark.parametrize("algo", ALGOS, ids=["tensor", "cuda_core"])
def test_whole_list_with_window(algo):
    """Implicit positions (base + i*stride) with a sliding window: tiles before the
    window are visited but masked."""
    w = mi.make_workload("win", batch=3, num_heads=128, q_lens=[2, 1, 3], kv_lens=[1500, 90, 700],
                         kv_dtype="fp8", causal=True, seed=43, num_slots=4096)
    _check(dataclasses.replace(w, window=100), algo, num_workers=24)


def test_window_list_matches_whole_list_on_the_gpu():
    """The same visible sets given two ways give the same result within tolerance."""
    full = mi.make_workload("full", batch=4, num_heads=64, q_lens=[1, 2, 3, 2], kv_lens=[2000, 500, 130, 4000],
                            kv_dtype="bf16", causal=True, seed=47, num_slots=8192)
    W = 96
    wfull = dataclasses.replace(full, window=W)
    idx, pos, lens = [], [], []
    for b in range(full.batch):
        k0, k1 = int(full.kv_indptr[b]), int(full.kv_indptr[b + 1])
        T = int(full.qo_indptr[b + 1] - full.qo_indptr[b])
        n = k1 - k0
        w0 = max(0, n - T - W + 1)
        idx.append(full.kv_indices[k0 + w0:k1])
        pos.append(np.arange(w0, n))
        lens.append(n - w0)
    wwin = dataclasses.replace(wfull, kv_indices=np.concatenate(idx).astype(np.int32),
                               kv_indptr=np.concatenate([[0], np.cumsum(lens)]).astype(np.int32),
                               kv_pos=np.concatenate(pos).astype(np.int32), g_kv_indptr=full.kv_indptr.copy())
    O1, L1, _ = hz.run(wfull, algo=m.MLA_ALGO_TENSOR, num_workers=24)
    O2, L2, _ = hz.run(wwin, algo=m.MLA_ALGO_TENSOR, num_workers=24)
    hz.assert_close(O2, L2, O1, L1, "bf16")


def test_csa_full_size_sampled():
    """A verify-sized CSA batch: 32 requests, T=2, 128 heads, fp8, contexts up to 64k,
    window 128 + top-2048 per request; a few whole requests checked."""
    rng = np.random.default_rng(3)
    Lg = rng.integers(4096, 65536, size=32)
    w = mi.sparse_variant("csa", batch=32, num_heads=128, q_lens=[2] * 32, global_lens=Lg, window=128,
                          topk=2048, kv_dtype="fp8", seed=53)
    _check(w, m.MLA_ALGO_TENSOR, reqs=hz.sample_requests(w, 3, seed=2))


def test_host_plan_with_positions():
    w = mi.sparse_variant("hca", batch=6, num_heads=128, q_lens=[1, 2, 1, 3, 1, 2],
                          global_lens=[20000, 5000, 800, 12000, 300, 64000], kv_dtype="fp8", seed=59)
    _check(w, m.MLA_ALGO_TENSOR, mode=m.MLA_PLAN_HOST)
