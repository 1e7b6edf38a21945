"""Pins of the fused RoPE + q concat + cache-write oracle (oracle/rope_cache.py).

* the rotation against the same rotation done as complex multiplication in
  float64 (an independent formulation), within float32 rounding;
* angle zero (cos 1, sin 0) is exactly the identity, a quarter turn (cos 0, sin 1)
  maps each pair (a, b) to (-b, a) exactly, rotating back by -theta returns the
  input; pair norms are preserved;
* the interleaved style is exactly the neox style on de-interleaved columns;
* the fused outputs: q's latent columns are copied bit for bit, its RoPE
  columns are the bf16 of the rotation, the cache rows are the cache-write
  oracle's rows of (kv_c, rotated k_pe); positions outside the table clamp;
* a planted sign error in the rotation fails the complex-rotation pin.
"""
import numpy as np
import pytest

import mla_inputs as mi
from oracle import cache_write as cw
from oracle import rope_cache as rc


def _tables(max_pos, seed=0):
    inp = mi.rope_inputs(num_tokens=1, num_heads=1, max_pos=max_pos, seed=seed)
    return inp.cos_sin


def _complex_ref(x, cos, sin, style):
    x = x.astype(np.float64)
    a, b = (x[..., :32], x[..., 32:]) if style == rc.NEOX else (x[..., 0::2], x[..., 1::2])
    z = (a + 1j * b) * (cos.astype(np.float64) + 1j * sin.astype(np.float64))
    y = np.empty_like(x)
    if style == rc.NEOX:
        y[..., :32], y[..., 32:] = z.real, z.imag
    else:
        y[..., 0::2], y[..., 1::2] = z.real, z.imag
    return y


@pytest.mark.parametrize("style", [rc.NEOX, rc.INTERLEAVED])
def test_rotation_matches_complex_multiplication(style):
    rng = np.random.default_rng(1)
    cs = _tables(4096)
    p = rng.integers(0, 4096, size=500)
    x = (rng.standard_normal((500, 64)) * rng.choice([1e-3, 1, 30], size=(500, 1))).astype(np.float32)
    y = rc.rope_f32(x, cs[p, :32], cs[p, 32:], style)
    ref = _complex_ref(x, cs[p, :32], cs[p, 32:], style)
    scale = np.abs(x).max(axis=1, keepdims=True)
    assert np.all(np.abs(y - ref) <= 4 * np.finfo(np.float32).eps * scale)


def test_angle_zero_is_identity_and_norms_are_kept():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((50, 64)).astype(np.float32)
    one, zero = np.ones((50, 32), np.float32), np.zeros((50, 32), np.float32)
    for style in (rc.NEOX, rc.INTERLEAVED):
        assert np.array_equal(rc.rope_f32(x, one, zero, style), x)
    cs = _tables(1024)
    p = rng.integers(0, 1024, size=50)
    y = rc.rope_f32(x, cs[p, :32], cs[p, 32:], rc.NEOX).astype(np.float64)
    n_in = x[:, :32].astype(np.float64) ** 2 + x[:, 32:].astype(np.float64) ** 2
    n_out = y[:, :32] ** 2 + y[:, 32:] ** 2
    assert np.allclose(n_in, n_out, rtol=1e-5)


def test_interleaved_is_neox_on_deinterleaved_columns():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((40, 64)).astype(np.float32)
    cs = _tables(512)
    p = rng.integers(0, 512, size=40)
    c, s = cs[p, :32], cs[p, 32:]
    perm = np.concatenate([np.arange(0, 64, 2), np.arange(1, 64, 2)])
    y_int = rc.rope_f32(x, c, s, rc.INTERLEAVED)
    y_neox = rc.rope_f32(x[:, perm], c, s, rc.NEOX)
    assert np.array_equal(y_int[:, perm], y_neox)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_fused_outputs_follow_the_parts(kv_dtype):
    inp = mi.rope_inputs(num_tokens=9, num_heads=3, max_pos=300, seed=4)
    inp.positions[0] = 1000                    # outside the table: clamps to the last row
    pool0 = np.zeros((16, 576), np.uint16 if kv_dtype == "bf16" else np.uint8)
    q, pool = rc.rope_q_cache(inp.q_nope_bits, inp.q_pe_bits, inp.kv_c_bits, inp.k_pe_bits, inp.positions,
                              inp.cos_sin, rc.NEOX, inp.slot_mapping, pool0, kv_dtype, 0.05)
    assert np.array_equal(q[..., :512], inp.q_nope_bits)
    p = np.clip(inp.positions, 0, 299)
    qr = rc.rope_f32(cw.bf16_bits_to_f32(inp.q_pe_bits), inp.cos_sin[p, None, :32], inp.cos_sin[p, None, 32:], rc.NEOX)
    assert np.array_equal(q[..., 512:], cw.f32_to_bf16_rne(qr))
    kr = rc.rope_f32(cw.bf16_bits_to_f32(inp.k_pe_bits), inp.cos_sin[p, :32], inp.cos_sin[p, 32:], rc.NEOX)
    want = cw.cache_write(pool0, cw.bf16_bits_to_f32(inp.kv_c_bits), kr, inp.slot_mapping, kv_dtype, 0.05)
    assert np.array_equal(pool, want)


def test_planted_sign_error_fails(monkeypatch):
    orig = rc.rope_f32

    def wrong(x, cos, sin, style):
        return orig(x, cos, -np.asarray(sin), style)

    monkeypatch.setattr(rc, "rope_f32", wrong)
    with pytest.raises(AssertionError):
        test_rotation_matches_complex_multiplication(rc.NEOX)


@pytest.mark.parametrize("style", [rc.NEOX, rc.INTERLEAVED])
def test_quarter_turn_is_exact(style):
    """cos 0, sin 1: every pair (a, b) becomes (-b, a) exactly (products by 0 and 1
    and sums with zero are exact), which fixes the sign convention of the rotation."""
    rng = np.random.default_rng(8)
    x = rng.standard_normal((30, 64)).astype(np.float32)
    zero, one = np.zeros((30, 32), np.float32), np.ones((30, 32), np.float32)
    y = rc.rope_f32(x, zero, one, style)
    if style == rc.NEOX:
        a, b, ya, yb = x[:, :32], x[:, 32:], y[:, :32], y[:, 32:]
    else:
        a, b, ya, yb = x[:, 0::2], x[:, 1::2], y[:, 0::2], y[:, 1::2]
    assert np.array_equal(ya, -b) and np.array_equal(yb, a)


@pytest.mark.parametrize("style", [rc.NEOX, rc.INTERLEAVED])
def test_rotation_then_inverse_returns_the_input(style):
    rng = np.random.default_rng(9)
    x = rng.standard_normal((40, 64)).astype(np.float32)
    cs = _tables(2048)
    p = rng.integers(0, 2048, size=40)
    c, s = cs[p, :32], cs[p, 32:]
    back = rc.rope_f32(rc.rope_f32(x, c, s, style), c, -s, style)
    assert np.all(np.abs(back - x) <= 8 * np.finfo(np.float32).eps * np.abs(x).max(axis=1, keepdims=True))
