"""GPU parity of the absorb BMMs (mla_absorb_bmm) against oracle/absorb_bmm.py.

Tolerance, from the arithmetic: the products of bf16 activations and bf16 / e4m3
weights are exact in float32, the tensor cores add them in float32 (error at most
about k * 2^-24 * sum|x w|, allowed twice over: k * 2^-23, and never below the
2^-14 the k <= 512 shapes were first checked with), and the scaled sum is rounded
once to bf16 (at most 2^-9 relative).  So every element must satisfy
|y - y*| <= 2^-8 |y*| + max(2^-14, k * 2^-23) * |s| * sum_k |x_k w_k|.

Covered: the absorb shape (k=128, n=512) and the un-absorb shape (k=512, n=128),
bf16 and fp8 weights, token counts from 1 to 300 (one to two token tiles, ragged
tails), every fp8 code and bf16 subnormal weights bit-exact through a
one-hot x, strided activations (q_nope as a view of a [n, H, 192] projection) and a
strided output (the first 512 columns of the 576-wide decode q, the RoPE columns
left untouched), zero tokens, repeatability, CUDA-graph replay, the full-size
workload (256 tokens x 128 heads), and the absorb -> decode -> un-absorb chain
against the oracle chain.
"""
import numpy as np
import pytest

import mla_inputs as mi
from oracle import absorb_bmm as ab
from oracle import cache_write as cw
from oracle import formats as fm
from oracle import mla_oracle as mo

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import token_mla_paged_gb300 as m  # noqa: E402
from tests import harness as hz  # noqa: E402


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _weight(inp):
    if inp.w_dtype == "bf16":
        return _bf16(inp.w_bits)
    return torch.from_numpy(np.ascontiguousarray(inp.w_bits)).cuda()


def _to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def sum_bound(k: int) -> float:
    """Relative bound of a float32 sum of k exact products, with a factor 2 of margin."""
    return max(2.0 ** -14, k * 2.0 ** -23)


def _check(y, inp, what=""):
    ref = ab.absorb_bmm(inp.x_bits, inp.w_bits, inp.w_dtype, inp.w_scale)
    mag = ab.head_bmm_f64(np.abs(fm.decode_bf16(inp.x_bits)), np.abs(ab.decode_weight(inp.w_bits, inp.w_dtype)),
                          abs(float(np.float32(inp.w_scale))))
    err = np.abs(y - ref)
    bound = 2.0 ** -8 * np.abs(ref) + sum_bound(inp.x_bits.shape[2]) * mag
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements out of bound, worst excess {np.max(err - bound):.3e}"


def _run(inp, x=None, out=None, status=None):
    if x is None:
        x = _bf16(inp.x_bits)
    n, H, _ = x.shape
    if out is None:
        out = torch.empty(n, H, inp.w_bits.shape[2], dtype=torch.bfloat16, device="cuda")
    m.mla_absorb_bmm(x, _weight(inp), out, inp.w_scale, status=status)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("w_dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("k,n", [(4096, 256), (8192, 128)], ids=["k4096", "k8192"])
def test_bmm_parity_long_k(w_dtype, k, n):
    """The longest sums the ABI accepts, where the float32 sum bound grows with k."""
    inp = mi.bmm_inputs(130, 3, k, n, w_dtype, seed=77 + k)
    y = _run(inp)
    _check(_to_f64(y), inp, f"{w_dtype} k={k} n={n}")


@pytest.mark.parametrize("w_dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("k,n", [(128, 512), (512, 128)], ids=["absorb", "unabsorb"])
@pytest.mark.parametrize("tokens,heads", [(1, 3), (7, 16), (37, 8), (64, 16), (256, 4), (300, 5)])
def test_bmm_parity(w_dtype, k, n, tokens, heads):
    inp = mi.bmm_inputs(tokens, heads, k, n, w_dtype, seed=1000 + tokens * 7 + heads + k)
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    y = _run(inp, status=status)
    _check(_to_f64(y), inp, f"{w_dtype} k={k} n={n} T={tokens} H={heads}")
    assert status.tolist() == [0, 0]


@pytest.mark.parametrize("w_dtype", ["bf16", "fp8"])
def test_strided_views(w_dtype):
    """q_nope is the first 128 columns of a [n, H, 192] projection; q_lat goes into
    the first 512 columns of the [n, H, 576] decode q, leaving columns 512-575."""
    tokens, heads = 45, 12
    inp = mi.bmm_inputs(tokens, heads, 128, 512, w_dtype, seed=77)
    proj_bits = np.concatenate([inp.x_bits, mi.to_bf16_bits(np.ones((tokens, heads, 64), np.float32))], axis=-1)
    proj = _bf16(proj_bits)
    q = torch.full((tokens, heads, 576), 3.0, dtype=torch.bfloat16, device="cuda")
    _run(inp, x=proj[..., :128], out=q[..., :512])
    _check(_to_f64(q[..., :512]), inp, "strided")
    assert bool((q[..., 512:] == 3.0).all())


def test_zero_tokens_is_a_no_op():
    inp = mi.bmm_inputs(1, 2, 128, 512, "fp8", seed=3)
    x = torch.empty(0, 2, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(0, 2, 512, dtype=torch.bfloat16, device="cuda")
    m.mla_absorb_bmm(x, _weight(inp), out, inp.w_scale)
    torch.cuda.synchronize()


def test_repeatable_and_graph_replay():
    inp = mi.bmm_inputs(96, 32, 512, 128, "fp8", seed=5)
    x = _bf16(inp.x_bits)
    w = _weight(inp)
    out = torch.empty(96, 32, 128, dtype=torch.bfloat16, device="cuda")
    m.mla_absorb_bmm(x, w, out, inp.w_scale)
    torch.cuda.synchronize()
    first = out.clone()
    m.mla_absorb_bmm(x, w, out, inp.w_scale)
    torch.cuda.synchronize()
    assert torch.equal(first, out)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    out.zero_()
    with torch.cuda.graph(g, stream=s):
        m.mla_absorb_bmm(x, w, out, inp.w_scale, stream=s)
    inp2 = mi.bmm_inputs(96, 32, 512, 128, "fp8", seed=6)
    x.copy_(_bf16(inp2.x_bits))
    g.replay()
    torch.cuda.synchronize()
    inp2.w_bits, inp2.w_scale = inp.w_bits, inp.w_scale
    _check(_to_f64(out), inp2, "graph replay")


@pytest.mark.parametrize("k,n", [(128, 512), (512, 128)], ids=["absorb", "unabsorb"])
def test_full_size_workload(k, n):
    """256 tokens (32 requests x 8-token blocks) x 128 heads, fp8 weights: the
    configuration the benchmark times, compared element by element."""
    inp = mi.bmm_inputs(256, 128, k, n, "fp8", seed=mi.SEED_BASE + 11)
    _check(_to_f64(_run(inp)), inp, f"full k={k}")


def test_absorb_decode_unabsorb_chain():
    """q_nope -> absorb -> (with q_pe) decode over a bf16 latent cache -> un-absorb,
    against the oracle chain with its own bf16 roundings of q_lat and O."""
    B, T, H, L = 2, 2, 16, 100
    n = B * T
    rng = np.random.default_rng(91)
    wk = mi.bmm_inputs(n, H, 128, 512, "fp8", seed=92)
    wv = mi.bmm_inputs(n, H, 512, 128, "fp8", seed=93)
    q_pe_bits = mi.to_bf16_bits(rng.standard_normal((n, H, 64), dtype=np.float32))
    kv_bits = mi.to_bf16_bits(rng.standard_normal((B * L, 576), dtype=np.float32))
    kv_indices = rng.permutation(B * L).astype(np.int32)

    # GPU chain
    q = torch.empty(n, H, 576, dtype=torch.bfloat16, device="cuda")
    m.mla_absorb_bmm(_bf16(wk.x_bits), _weight(wk), q[..., :512], wk.w_scale)
    q[..., 512:] = _bf16(q_pe_bits)
    torch.cuda.synchronize()
    q_bits = q.view(torch.int16).cpu().numpy().view(np.uint16)
    w = mi.Workload(name="chain", num_heads=H, q_bits=q_bits, kv_bits=kv_bits, kv_dtype="bf16",
                    kv_indptr=np.array([0, L, 2 * L], np.int32), kv_indices=kv_indices,
                    qo_indptr=np.array([0, T, 2 * T], np.int32), causal=True,
                    softmax_scale=mi.SOFTMAX_SCALE, kv_scale=1.0)
    O, _, runner = hz.run(w, algo=m.MLA_ALGO_TENSOR, num_workers=8)
    assert hz.device_error(runner) == (0, 0)
    o_lat = torch.from_numpy(np.ascontiguousarray(O, dtype=np.float32)).to(torch.bfloat16).cuda()
    out = torch.empty(n, H, 128, dtype=torch.bfloat16, device="cuda")
    m.mla_absorb_bmm(o_lat, _weight(wv), out, wv.w_scale)
    torch.cuda.synchronize()

    # oracle chain (its own roundings; nothing taken from the GPU)
    q_lat = ab.absorb_bmm(wk.x_bits, wk.w_bits, "fp8", wk.w_scale)
    q_ref_bits = np.concatenate([cw.f32_to_bf16_rne(q_lat.astype(np.float32)), q_pe_bits], axis=-1)
    w_ref = mi.Workload(name="chain", num_heads=H, q_bits=q_ref_bits, kv_bits=kv_bits, kv_dtype="bf16",
                        kv_indptr=w.kv_indptr, kv_indices=kv_indices, qo_indptr=w.qo_indptr, causal=True,
                        softmax_scale=mi.SOFTMAX_SCALE, kv_scale=1.0)
    O_ref, _ = mo.mla_decode_workload(w_ref)
    o_bits = cw.f32_to_bf16_rne(O_ref.astype(np.float32))
    ref = ab.absorb_bmm(o_bits, wv.w_bits, "fp8", wv.w_scale)
    got = _to_f64(out)
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.all(np.abs(got - ref) <= 2e-2 * (np.abs(ref) + rms))


def _one_hot_x(tokens, heads, k):
    x = np.zeros((tokens, heads, k), np.float32)
    x[np.arange(tokens), :, np.arange(tokens) % k] = 1.0
    return mi.to_bf16_bits(x)


def test_every_fp8_code_is_exact():
    """A one-hot x picks one weight row per token, so each output is the single
    product bf16(fp32(w) * fp32(s)): every finite e4m3fn code (subnormals, zeros of
    both signs, +-448) must come out bit-exact."""
    H, K, N = 2, 128, 512
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    w_bits = np.resize(codes, H * K * N).reshape(H, K, N)
    w_bits[1] = np.roll(w_bits[1], 37, axis=1)
    scale = 0.3711
    inp = mi.BmmInputs(x_bits=_one_hot_x(K, H, K), w_bits=w_bits, w_dtype="fp8", w_scale=scale)
    y = _run(inp).view(torch.int16).cpu().numpy().view(np.uint16)
    wv = fm.decode_e4m3fn(w_bits).astype(np.float32)                     # exact
    t = np.arange(K)
    want = cw.f32_to_bf16_rne((wv[:, t % K, :] * np.float32(scale)).astype(np.float32)).transpose(1, 0, 2)
    # a -0 product summed with the +0 products of the other rows is +0 (IEEE)
    same = (y == want) | (((y & 0x7FFF) == 0) & ((want & 0x7FFF) == 0))
    bad = np.argwhere(~same)
    assert bad.size == 0, [(int(w_bits[h, tt % K, j]), int(y[tt, h, j]), int(want[tt, h, j])) for tt, h, j in bad[:8]]


def test_bf16_weights_including_subnormals_are_exact():
    rng = np.random.default_rng(17)
    H, K, N = 3, 64, 256
    w = rng.standard_normal((H, K, N)).astype(np.float32) * rng.choice(
        np.array([1e-39, 1e-30, 1e-3, 1.0, 300.0], np.float32), size=(H, K, N))
    inp = mi.BmmInputs(x_bits=_one_hot_x(K, H, K), w_bits=mi.to_bf16_bits(w), w_dtype="bf16", w_scale=1.0)
    y = _run(inp).view(torch.int16).cpu().numpy().view(np.uint16)
    t = np.arange(K)
    want = inp.w_bits[:, t % K, :].transpose(1, 0, 2)
    same = (y == want) | (((y & 0x7FFF) == 0) & ((want & 0x7FFF) == 0))
    bad = np.argwhere(~same)
    assert bad.size == 0, [(int(y[tt, h, j]), int(want[tt, h, j])) for tt, h, j in bad[:8]]


def test_rejects_bad_arguments():
    x = torch.zeros(4, 2, 128, dtype=torch.float32, device="cuda")
    w = torch.zeros(2, 128, 512, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(4, 2, 512, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.MlaError):
        m.mla_absorb_bmm(x, w, out)
    with pytest.raises(m.MlaError):
        m.mla_absorb_bmm(x.to(torch.bfloat16), w[:, :96], out)
