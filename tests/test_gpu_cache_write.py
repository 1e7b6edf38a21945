"""GPU parity of the KV-cache write (mla_cache_write) against oracle/cache_write.py.

Byte work, so the bar is bit-exact: every byte of the pool after the call equals
the oracle's pool, for bf16 and fp32 inputs into bf16 and fp8 pools, with
padding and out-of-range slots, strided input rows (latent and RoPE columns as
views of one fused [n, 576] projection output), and the pages' failure case (an
fp32 k_pe next to a bf16 kv_c: converted, not reinterpreted).  Then the decode
reads a pool written this way and matches the oracle decode of the oracle-written
pool.
"""
import numpy as np
import pytest

import mla_inputs as mi
from oracle import cache_write as cw
from oracle import mla_oracle as mo

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import token_mla_paged_gb300 as m  # noqa: E402
from tests import harness as hz  # noqa: E402

POOL_DT = {"bf16": (np.uint16, torch.int16, m.MLA_KV_BF16), "fp8": (np.uint8, torch.uint8, m.MLA_KV_FP8_E4M3)}


def _dev_act(x_f32, bits, dtype):
    if dtype == "bf16":
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(x_f32).cuda()


def _run(inp, kv_dtype, kv_c_dtype, k_pe_dtype, pool0, fused=False):
    npdt, tdt, code = POOL_DT[kv_dtype]
    pool = torch.from_numpy(pool0.copy().view(np.int16 if npdt == np.uint16 else np.uint8)).cuda()
    kv_c = _dev_act(inp.kv_c, inp.kv_c_bits, kv_c_dtype)
    k_pe = _dev_act(inp.k_pe, inp.k_pe_bits, k_pe_dtype)
    if fused:   # one [n, 576] buffer, latent and RoPE columns as strided views
        assert kv_c.dtype == k_pe.dtype
        buf = torch.cat([kv_c, k_pe], dim=1).contiguous()
        kv_c, k_pe = buf[:, :512], buf[:, 512:]
    slots = torch.from_numpy(inp.slot_mapping).cuda()
    m.mla_cache_write(kv_c, k_pe, slots, pool, code, inp.kv_scale)
    torch.cuda.synchronize()
    return pool.cpu().numpy().view(npdt)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("dts", [("bf16", "bf16"), ("fp32", "fp32"), ("bf16", "fp32")],
                         ids=["bf16-in", "fp32-in", "fp32-k_pe"])
def test_cache_write_bit_exact(kv_dtype, dts):
    kv_c_dtype, k_pe_dtype = dts
    inp = mi.cache_write_inputs(700, 1024, kv_c_dtype=kv_c_dtype, k_pe_dtype=k_pe_dtype,
                                padding=0.1, out_of_range=0.05, spread=True)
    npdt = POOL_DT[kv_dtype][0]
    pool0 = np.random.default_rng(9).integers(0, 120, size=(1024, 576)).astype(npdt)
    got = _run(inp, kv_dtype, kv_c_dtype, k_pe_dtype, pool0)
    want = cw.cache_write(pool0, inp.kv_c, inp.k_pe, inp.slot_mapping, kv_dtype, inp.kv_scale)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_cache_write_strided_views(kv_dtype):
    inp = mi.cache_write_inputs(333, 512, seed=17)
    npdt = POOL_DT[kv_dtype][0]
    pool0 = np.zeros((512, 576), npdt)
    got = _run(inp, kv_dtype, "bf16", "bf16", pool0, fused=True)
    want = cw.cache_write(pool0, inp.kv_c, inp.k_pe, inp.slot_mapping, kv_dtype, inp.kv_scale)
    assert np.array_equal(got, want)


def test_fp32_k_pe_is_converted_not_reinterpreted():
    """The pages' failure: an fp32 k_pe next to a bf16 kv_c.  Converted here; reading
    its bytes as bf16 would have put garbage in the RoPE columns."""
    inp = mi.cache_write_inputs(64, 64, kv_c_dtype="bf16", k_pe_dtype="fp32", seed=23)
    pool0 = np.zeros((64, 576), np.uint16)
    got = _run(inp, "bf16", "bf16", "fp32", pool0)
    rows = got[inp.slot_mapping]
    assert np.array_equal(rows[:, 512:], cw.f32_to_bf16_rne(inp.k_pe))
    reinterpreted = inp.k_pe.view(np.uint16)[:, :64]
    assert not np.array_equal(rows[:, 512:], reinterpreted)


def test_cache_write_full_size_sampled():
    """65536 tokens (the draft block's KV) into a 131072-slot fp8 pool; every written
    row checked on a sample, all untouched slots checked."""
    inp = mi.cache_write_inputs(65536, 131072, seed=29)
    pool0 = np.zeros((131072, 576), np.uint8)
    got = _run(inp, "fp8", "bf16", "bf16", pool0)
    pick = np.random.default_rng(1).choice(65536, 2000, replace=False)
    want = cw.cache_write(np.zeros((131072, 576), np.uint8), inp.kv_c[pick], inp.k_pe[pick],
                          inp.slot_mapping[pick], "fp8", inp.kv_scale)
    sl = inp.slot_mapping[pick]
    assert np.array_equal(got[sl], want[sl])
    untouched = np.setdiff1d(np.arange(131072), inp.slot_mapping)
    assert not got[untouched].any()


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_write_then_decode(kv_dtype):
    """Decode over a pool filled by mla_cache_write equals the oracle decode over the
    oracle-written pool (same bytes, checked first)."""
    base = mi.make_workload("cw_decode", batch=3, num_heads=64, q_lens=[2, 1, 3], kv_lens=[300, 77, 513],
                            kv_dtype=kv_dtype, causal=True, seed=31, num_slots=1024)
    n = int(base.kv_indptr[-1])
    inp = mi.cache_write_inputs(n, 1024, seed=37)
    inp.slot_mapping[:] = base.kv_indices          # write exactly the slots the decode reads
    npdt = POOL_DT[kv_dtype][0]
    pool0 = np.zeros((1024, 576), npdt)
    got = _run(inp, kv_dtype, "bf16", "bf16", pool0)
    want = cw.cache_write(pool0, inp.kv_c, inp.k_pe, inp.slot_mapping, kv_dtype, inp.kv_scale)
    assert np.array_equal(got, want)
    w = mi.Workload(name=base.name, num_heads=base.num_heads, q_bits=base.q_bits, kv_bits=want,
                    kv_dtype=kv_dtype, kv_indptr=base.kv_indptr, kv_indices=base.kv_indices,
                    qo_indptr=base.qo_indptr, causal=True, softmax_scale=base.softmax_scale,
                    kv_scale=inp.kv_scale if kv_dtype == "fp8" else 1.0)
    O, L, runner = hz.run(w, algo=m.MLA_ALGO_TENSOR, mode=m.MLA_PLAN_DYNAMIC, num_workers=24)
    assert hz.device_error(runner) == (0, 0)
    Oref, Lref = mo.mla_decode_workload(w)
    hz.assert_close(O, L, Oref, Lref, kv_dtype)


def test_cache_write_rejects_other_dtypes():
    kv_c = torch.zeros(4, 512, dtype=torch.float16, device="cuda")
    k_pe = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros(8, 576, dtype=torch.int16, device="cuda")
    with pytest.raises(m.MlaError):
        m.mla_cache_write(kv_c, k_pe, torch.arange(4, dtype=torch.int32, device="cuda"), pool, m.MLA_KV_BF16)
