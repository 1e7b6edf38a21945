"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Tolerances (elementwise over O, on dequantized inputs): abs 1e-2 + rel 1e-2 for a
bf16 pool, abs 3e-2 + rel 3e-2 for fp8; LSE within 2e-3 absolute; plan and
index work bit-exact.
"""
import dataclasses

import numpy as np
import pytest

import mla_inputs as mi
from oracle import mla_oracle as mo, plan_oracle as po
from tests import harness as hz

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped there
    pytest.skip("needs a GPU", allow_module_level=True)

import token_mla_paged_gb300 as m  # noqa: E402

# Both kernels are always in the matrix: on an sm_103a device a tensor-kernel
# launch failure fails these tests instead of dropping the kernel from them.
ALGOS = [m.MLA_ALGO_CUDA_CORE, m.MLA_ALGO_TENSOR]
ALGO_IDS = {m.MLA_ALGO_CUDA_CORE: "cuda_core", m.MLA_ALGO_TENSOR: "tensor"}


@pytest.fixture(params=ALGOS, ids=lambda a: ALGO_IDS[a])
def algo(request):
    return request.param


def _check(w, algo, mode=1, reqs=None, **kw):
    O, L, runner = hz.run(w, algo=algo, mode=mode, **kw)
    assert hz.device_error(runner) == (0, 0)
    Oref, Lref = mo.mla_decode_workload(w, requests=reqs)
    rows = None if reqs is None else hz.rows_of(w, reqs)
    return hz.assert_close(O, L, Oref, Lref, w.kv_dtype, rows=rows, what=w.name)


# ------------------------------------------------------------------ the five workloads

def test_tiny_causal_bf16(algo):
    _check(mi.tiny_causal_bf16(), algo)


@pytest.mark.parametrize("scale", [1 / 64, 1 / 16 + 1 / 512])
def test_draft_block_bf16_small(algo, scale):
    _check(mi.draft_block_bf16(scale=scale), algo)


def test_draft_block_bf16_full_sampled(algo):
    w = mi.draft_block_bf16()
    _check(w, algo, reqs=[0, 5])


def test_draft_block_equals_flattened_rows(algo):
    """A non-causal T-token block equals T flattened single-token rows over the same KV."""
    w = mi.draft_block_bf16(scale=1 / 32)
    O1, L1, _ = hz.run(w, algo=algo)
    O2, L2, _ = hz.run(mi.flatten_block(w), algo=algo)
    Oref, Lref = mo.mla_decode_workload(w)
    hz.assert_close(O1, L1, Oref, Lref, "bf16")
    hz.assert_close(O2, L2, Oref, Lref, "bf16")


@pytest.mark.parametrize("mode", [0, 1, 2], ids=["static", "dynamic", "host"])
def test_verify_fp8_small(algo, mode):
    w = mi.verify_fp8(scale=1 / 16)
    _check(w, algo, mode=mode, kv_len_cap=w.meta["kv_len_cap"], num_workers=608)


def test_verify_fp8_full_sampled_static(algo):
    w = mi.verify_fp8()
    _check(w, algo, mode=0, reqs=hz.sample_requests(w, 3), kv_len_cap=w.meta["kv_len_cap"],
           num_workers=608)


def test_verify_fp8_full_sampled_host_plan(algo):
    """The host plan built from the real kv_indptr (the plan the benchmark uses)."""
    w = mi.verify_fp8()
    _check(w, algo, mode=2, reqs=hz.sample_requests(w, 3, seed=11), num_workers=76)


def test_host_plan_stays_correct_for_other_lengths():
    """A HOST plan sized for one set of lengths, called with other lengths: the
    split ranges follow the call's lengths, so the result is still exact."""
    import token_mla_paged_gb300 as m
    w0 = mi.verify_fp8(scale=1 / 16, seed=3)
    w1 = mi.verify_fp8(scale=1 / 16, seed=4)
    runner = m.DecodeRunner(w1.batch, w1.num_heads, 8, mode=m.MLA_PLAN_HOST, num_workers=76)
    runner.set_host_plan(w0.kv_indptr, w0.qo_indptr)
    O, L, _ = hz.run(w1, algo=m.MLA_ALGO_TENSOR, runner=runner)
    assert hz.device_error(runner) == (0, 0)
    Oref, Lref = mo.mla_decode_workload(w1)
    hz.assert_close(O, L, Oref, Lref, "fp8")


def test_long_skewed_fp8_small(algo):
    _check(mi.long_skewed_fp8(scale=1 / 64), algo, mode=1)


def test_long_skewed_fp8_full_sampled(algo):
    w = mi.long_skewed_fp8()
    _check(w, algo, mode=1, reqs=hz.sample_requests(w, 3))


def _cp_run(sw, algo, reqs=None, out_fp32=True):
    """The shards as one batched call, then the LSE merge.  Shard outputs are fp32
    or bf16 (the benchmark's choice: half the partial traffic; each shard's O is
    normalised, so its bf16 rounding adds at most 2^-9 of max |O_s| to the merge)."""
    sh = sw.shards
    O, L, runner = hz.run(sh, algo=algo, out_fp32=out_fp32)
    assert hz.device_error(runner) == (0, 0)
    R = sw.full.total_q * sw.full.num_heads
    o_parts = torch.from_numpy(O.reshape(sw.num_shards, R, 512).astype(np.float32)).cuda()
    if not out_fp32:
        o_parts = o_parts.to(torch.bfloat16)     # exact: the values are bf16 already
    l_parts = torch.from_numpy(L.reshape(sw.num_shards, R).astype(np.float32)).cuda()
    om = torch.empty(R, 512, dtype=torch.bfloat16, device="cuda")
    lm = torch.empty(R, dtype=torch.float32, device="cuda")
    m.mla_merge_states(o_parts, l_parts, om, lm)
    torch.cuda.synchronize()
    Of, Lf = mo.mla_decode_workload(sw.full, requests=reqs)
    Om = om.double().cpu().numpy().reshape(sw.full.total_q, sw.full.num_heads, 512)
    Lm = lm.double().cpu().numpy().reshape(sw.full.total_q, sw.full.num_heads)
    rows = None if reqs is None else hz.rows_of(sw.full, reqs)
    hz.assert_close(Om, Lm, Of, Lf, "bf16", rows=rows, what="cp merged")


@pytest.mark.parametrize("out_fp32", [True, False], ids=["fp32_parts", "bf16_parts"])
def test_cp_shards_small(algo, out_fp32):
    _cp_run(mi.cp_shards_bf16(scale=1 / 64), algo, out_fp32=out_fp32)


@pytest.mark.parametrize("out_fp32", [True, False], ids=["fp32_parts", "bf16_parts"])
def test_cp_shards_full_sampled(algo, out_fp32):
    _cp_run(mi.cp_shards_bf16(), algo, reqs=[0, 11], out_fp32=out_fp32)


# ------------------------------------------------------------------ planner

@pytest.mark.parametrize("seed", range(6))
def test_device_plan_bit_exact(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 200))
    H = int(rng.choice([16, 64, 96, 128]))
    maxT = int(rng.integers(1, 9))
    W = int(rng.integers(1, 300))
    T = rng.integers(0, maxT + 1, size=B)
    L = np.floor(np.exp(rng.uniform(0, np.log(200000), size=B))).astype(np.int64)
    L[rng.random(B) < 0.1] = 0
    kvp = np.concatenate([[5], 5 + np.cumsum(L)]).astype(np.int32)   # offset kv_indptr[0]
    qop = np.concatenate([[0], np.cumsum(T)]).astype(np.int32)
    params = m.plan_params(B, H, maxT, W, 0, m.MLA_PLAN_DYNAMIC)
    pb, wb = m.mla_decode_plan_size(params)
    plan = torch.full((pb // 4,), -7, dtype=torch.int32, device="cuda")
    ws = torch.zeros((wb + 3) // 4, dtype=torch.int32, device="cuda")
    m.mla_decode_plan_device(params, torch.from_numpy(kvp).cuda(), torch.from_numpy(qop).cuda(),
                             plan, ws)
    torch.cuda.synchronize()
    ref = po.build_plan(B, H, maxT, W, 0, po.DYNAMIC, kvp, qop)
    assert np.array_equal(plan.cpu().numpy(), ref)
    assert np.array_equal(m.mla_decode_plan(params, kvp, qop), ref)
    assert m.mla_get_device_error(ws) == (0, 0)


# ------------------------------------------------------------------ merge

@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("n,dv", [(5, 512), (12, 512), (3, 96)], ids=["n5", "n12", "dv96"])
def test_merge_states_matches_oracle(dtype, n, dv):
    """Both merge paths: vectorised (dv a multiple of 256, up to 8 or 16 states) and general."""
    rng = np.random.default_rng(4 + n + dv)
    rows = 777
    o = rng.standard_normal((n, rows, dv)).astype(np.float32)
    lse = (rng.standard_normal((n, rows)) * 3).astype(np.float32)
    lse[1, :100] = -np.inf
    lse[:, 200:210] = -np.inf
    ot = torch.from_numpy(o).cuda()
    if dtype == "bf16":
        ot = ot.to(torch.bfloat16)
        o = ot.float().cpu().numpy()
    om = torch.empty(rows, dv, dtype=torch.float32, device="cuda")
    lm = torch.empty(rows, dtype=torch.float32, device="cuda")
    m.mla_merge_states(ot, torch.from_numpy(lse).cuda(), om, lm)
    torch.cuda.synchronize()
    ro, rl = mo.merge_states(o, lse)
    hz.assert_close(om.double().cpu().numpy(), lm.double().cpu().numpy(), ro, rl, "bf16")
    assert np.allclose(om.cpu().numpy(), ro, atol=1e-5)


# ------------------------------------------------------------------ edge cases

def test_edge_cases_empty_and_ragged(algo):
    """T=0 request, L=0 request, single entry, ragged tails, offset kv_indptr."""
    w = mi.make_workload("edge", batch=6, num_heads=24, q_lens=[3, 0, 2, 1, 5, 1],
                         kv_lens=[0, 9, 1, 65, 200, 129], kv_dtype="bf16", causal=True,
                         seed=31, num_slots=512)
    _check(w, algo)
    w2 = dataclasses.replace(w, kv_indptr=w.kv_indptr + 3,
                             kv_indices=np.concatenate([np.array([1, 2, 3], np.int32), w.kv_indices]))
    _check(w2, algo)


def test_many_row_groups_and_splits(algo):
    """H*T > 128 (several row groups) with forced splitting (W large)."""
    w = mi.make_workload("groups", batch=3, num_heads=100, q_lens=[3, 1, 4], kv_lens=[3000, 777, 5000],
                         kv_dtype="fp8", causal=True, seed=37, num_slots=16384)
    _check(w, algo, num_workers=400)


def test_bad_index_sets_error_word(algo):
    w = mi.make_workload("bad", batch=1, num_heads=16, q_lens=[1], kv_lens=[10], kv_dtype="bf16",
                         causal=False, seed=41, num_slots=16)
    w.kv_indices[3] = 99
    O, L, runner = hz.run(w, algo=algo)
    code, info = hz.device_error(runner)
    assert code == 1 and info == 3
    assert np.isfinite(L).all()
    assert hz.device_error(runner) == (0, 0)   # cleared by the read


def test_plan_mismatch_detected(algo):
    w = mi.make_workload("pm", batch=2, num_heads=16, q_lens=[1, 2], kv_lens=[10, 20], kv_dtype="bf16",
                         causal=False, seed=43, num_slots=64)
    runner = m.DecodeRunner(2, 16, 2, mode=m.MLA_PLAN_STATIC, num_workers=8, kv_len_cap=64)
    runner.set_host_plan(None, w.qo_indptr)
    runner.plan_d[2] = 5   # corrupt the batch field
    hz.run(w, algo=algo, runner=runner)
    assert hz.device_error(runner)[0] == 3


def test_identical_query_rows_bitwise(algo):
    w = mi.make_workload("ident", batch=2, num_heads=32, q_lens=[4, 4], kv_lens=[300, 90],
                         kv_dtype="fp8", causal=False, seed=47, num_slots=512, identical_q_rows=True)
    O, L, _ = hz.run(w, algo=algo)
    for b in range(2):
        blk = O[w.qo_indptr[b]:w.qo_indptr[b + 1]].reshape(-1, 512)
        assert np.all(blk == blk[0][None])


def test_repeat_calls_bitwise_identical(algo):
    w = mi.long_skewed_fp8(scale=1 / 32)
    dev = mi.to_device(w)
    O1, L1, r = hz.run(w, algo=algo, dev=dev)
    O2, L2, _ = hz.run(w, algo=algo, dev=dev, runner=r)
    assert np.array_equal(O1, O2, equal_nan=True) and np.array_equal(L1, L2, equal_nan=True)


def test_wrong_mask_fails_tolerance(algo):
    """Mask liveness: running the causal workload without its mask must miss the oracle."""
    w = mi.verify_fp8(scale=1 / 16)
    O, L, _ = hz.run(dataclasses.replace(w, causal=False), algo=algo, num_workers=608)
    Oref, Lref = mo.mla_decode_workload(w, requests=[0, 1])
    with pytest.raises(AssertionError):
        hz.assert_close(O, L, Oref, Lref, "fp8", rows=hz.rows_of(w, [0, 1]))


@pytest.mark.parametrize("heads,t", [(127, 1), (128, 1), (129, 1), (85, 3), (128, 2), (257, 1)],
                         ids=["rows127", "rows128", "rows129", "rows255", "rows256", "rows257"])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_row_counts_around_the_item_halves(algo, heads, t, kv_dtype):
    """Query rows per request just below, at and above a CTA's 128 rows and an item's
    256 (the second CTA of a pair empty, one row, full; a second item of one row),
    with KV long enough for the planner to give every row group 16 splits."""
    w = mi.make_workload(f"halves_{heads}x{t}", batch=2, num_heads=heads, q_lens=[t, t],
                         kv_lens=[16 * 128 * 4 + 77, 300], kv_dtype=kv_dtype, causal=True,
                         seed=53 + heads + t, num_slots=16384)
    runner_w = 4096
    O, L, runner = hz.run(w, algo=algo, num_workers=runner_w)
    assert hz.device_error(runner) == (0, 0)
    # the long request's row groups use the largest split count
    assert int(runner.plan_d[16]) == 16
    Oref, Lref = mo.mla_decode_workload(w)
    hz.assert_close(O, L, Oref, Lref, kv_dtype, what=w.name)


def test_empty_batch_is_a_no_op(algo):
    runner = m.DecodeRunner(0, 16, 1, mode=m.MLA_PLAN_DYNAMIC, num_workers=8)
    z32 = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = torch.zeros(1, 16, 576, dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros(4, 576, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros(1, 16, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 16, dtype=torch.float32, device="cuda")
    runner.forward(q=q, kv_pool=pool, kv_dtype=m.MLA_KV_BF16, kv_indptr=z32, kv_indices=z32,
                   qo_indptr=z32, causal=True, softmax_scale=0.07, kv_scale=1.0, o=o, lse=lse, algo=algo)
    torch.cuda.synchronize()
    assert hz.device_error(runner) == (0, 0)
    assert not o.any() and not lse.any()
