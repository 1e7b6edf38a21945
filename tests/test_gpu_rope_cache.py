"""GPU parity of the fused decode RoPE + q concat + cache write (mla_rope_q_cache)
against oracle/rope_cache.py: bit-exact q rows and pool bytes for both rotation
styles and both pool dtypes, with strided inputs (q's latent and RoPE columns as
views of one [n, H, 576] projection, kv_c / k_pe as views of one [n, 576] row),
padding slots and positions outside the table; then the decode over the q and
pool it produced matches the oracle decode."""
import numpy as np
import pytest

import mla_inputs as mi
from oracle import mla_oracle as mo
from oracle import rope_cache as rc

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import token_mla_paged_gb300 as m  # noqa: E402
from tests import harness as hz  # noqa: E402


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _run(inp, kv_dtype, style, fused_views=False, pool0=None):
    n, H = inp.q_nope_bits.shape[:2]
    if fused_views:
        qa = _bf16(np.concatenate([inp.q_nope_bits, inp.q_pe_bits], axis=-1))
        q_nope, q_pe = qa[..., :512], qa[..., 512:]
        ka = _bf16(np.concatenate([inp.kv_c_bits, inp.k_pe_bits], axis=-1))
        kv_c, k_pe = ka[:, :512], ka[:, 512:]
    else:
        q_nope, q_pe, kv_c, k_pe = (_bf16(inp.q_nope_bits), _bf16(inp.q_pe_bits), _bf16(inp.kv_c_bits),
                                    _bf16(inp.k_pe_bits))
    npdt = np.uint16 if kv_dtype == "bf16" else np.uint8
    if pool0 is None:
        pool0 = np.zeros((inp.num_slots, 576), npdt)
    pool = torch.from_numpy(pool0.copy().view(np.int16 if npdt == np.uint16 else np.uint8)).cuda()
    q_out = torch.empty(n, H, 576, dtype=torch.bfloat16, device="cuda")
    code = m.MLA_KV_BF16 if kv_dtype == "bf16" else m.MLA_KV_FP8_E4M3
    m.mla_rope_q_cache(q_nope, q_pe, q_out, kv_c, k_pe, torch.from_numpy(inp.positions).cuda(),
                       torch.from_numpy(inp.cos_sin).cuda(), torch.from_numpy(inp.slot_mapping).cuda(), pool,
                       code, 0.05, rope_style=style)
    torch.cuda.synchronize()
    return q_out.view(torch.int16).cpu().numpy().view(np.uint16), pool.cpu().numpy().view(npdt), pool0


@pytest.mark.parametrize("style", [m.MLA_ROPE_NEOX, m.MLA_ROPE_INTERLEAVED], ids=["neox", "interleaved"])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("fused_views", [False, True], ids=["separate", "views"])
def test_rope_q_cache_bit_exact(style, kv_dtype, fused_views):
    inp = mi.rope_inputs(num_tokens=77, num_heads=24, max_pos=8192, num_slots=256, seed=61)
    inp.positions[:3] = [-5, 8192, 100000]                 # outside the table: clamped
    inp.slot_mapping[3:6] = [-1, 256, 9999]                # padding / outside the pool: no write
    q, pool, pool0 = _run(inp, kv_dtype, style, fused_views)
    q_ref, pool_ref = rc.rope_q_cache(inp.q_nope_bits, inp.q_pe_bits, inp.kv_c_bits, inp.k_pe_bits, inp.positions,
                                      inp.cos_sin, style, inp.slot_mapping, pool0, kv_dtype, 0.05)
    assert np.array_equal(q, q_ref)
    assert np.array_equal(pool, pool_ref)


def test_rope_then_decode():
    """q and the pool come from mla_rope_q_cache; the decode over them matches the
    oracle decode over the oracle's q and pool (same bytes, checked first)."""
    B, T, H, L = 2, 2, 64, 300
    n_ctx = B * L
    inp = mi.rope_inputs(num_tokens=n_ctx, num_heads=H, max_pos=4096, num_slots=1024, seed=67)
    q, pool, pool0 = _run(inp, "fp8", m.MLA_ROPE_NEOX)
    q_ref, pool_ref = rc.rope_q_cache(inp.q_nope_bits, inp.q_pe_bits, inp.kv_c_bits, inp.k_pe_bits, inp.positions,
                                      inp.cos_sin, m.MLA_ROPE_NEOX, inp.slot_mapping, pool0, "fp8", 0.05)
    assert np.array_equal(q, q_ref) and np.array_equal(pool, pool_ref)
    # the last T tokens of each request are its query block; all L tokens are its KV
    qsel = np.concatenate([np.arange(b * L + L - T, b * L + L) for b in range(B)])
    w = mi.Workload(name="rope_decode", num_heads=H, q_bits=np.ascontiguousarray(q[qsel]), kv_bits=pool,
                    kv_dtype="fp8", kv_indptr=np.array([0, L, 2 * L], np.int32),
                    kv_indices=inp.slot_mapping.astype(np.int32), qo_indptr=np.array([0, T, 2 * T], np.int32),
                    causal=True, softmax_scale=mi.SOFTMAX_SCALE, kv_scale=0.05)
    O, Ls, runner = hz.run(w, algo=m.MLA_ALGO_TENSOR, num_workers=24)
    assert hz.device_error(runner) == (0, 0)
    Oref, Lref = mo.mla_decode_workload(w)
    hz.assert_close(O, Ls, Oref, Lref, "fp8")


def test_rope_rejects_bad_arguments():
    x = torch.zeros(4, 2, 512, dtype=torch.float32, device="cuda")
    with pytest.raises(m.MlaError):
        m.mla_rope_q_cache(x, x, x, x, x, None, None, None, None, m.MLA_KV_BF16)


@pytest.mark.parametrize("style", [m.MLA_ROPE_NEOX, m.MLA_ROPE_INTERLEAVED], ids=["neox", "interleaved"])
def test_rope_q_cache_full_size(style):
    """The benchmarked size: 512 tokens x 128 heads into a 131072-slot fp8 pool with a
    131072-position table; every q row and every pool row bit-exact."""
    import bench
    inp = mi.rope_inputs(bench.RC_TOKENS, bench.RC_HEADS, max_pos=bench.RC_MAXPOS, num_slots=bench.RC_SLOTS)
    q, pool, pool0 = _run(inp, "fp8", style)
    q_ref, pool_ref = rc.rope_q_cache(inp.q_nope_bits, inp.q_pe_bits, inp.kv_c_bits, inp.k_pe_bits, inp.positions,
                                      inp.cos_sin, style, inp.slot_mapping, pool0, "fp8", 0.05)
    assert np.array_equal(q, q_ref)
    assert np.array_equal(pool, pool_ref)
