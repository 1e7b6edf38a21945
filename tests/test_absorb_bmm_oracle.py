"""Pins of the absorb BMM oracle (oracle/absorb_bmm.py).

* brute force on tiny inputs: Python loops with math.fsum over the products of
  values decoded by torch's own casts (not the oracle's decoders), square and
  non-square weights, bf16 and fp8 weights;
* closed form: a one-hot (selection) weight returns the selected input columns
  times the scale, exactly;
* the absorption identity the decode rests on: absorb -> latent attention ->
  un-absorb equals multi-head attention with explicitly up-projected keys and
  values, in float64;
* planted mistakes (one head's weight for every head, a transposed weight, a
  dropped scale) each fail one of these pins.
"""
import math

import numpy as np
import pytest
import torch

import mla_inputs as mi
from oracle import absorb_bmm as ab
from oracle import mla_oracle as mo


def _torch_decode(bits, w_dtype):
    t = torch.from_numpy(np.ascontiguousarray(bits))
    if w_dtype == "bf16":
        return t.view(torch.int16).view(torch.bfloat16).to(torch.float64).numpy()
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _brute(x_bits, w_bits, w_dtype, scale):
    x = _torch_decode(x_bits, "bf16")
    w = _torch_decode(w_bits, w_dtype)
    n, H, K = x.shape
    N = w.shape[2]
    y = np.zeros((n, H, N))
    mag = np.zeros((n, H, N))
    for t in range(n):
        for h in range(H):
            for j in range(N):
                prods = [x[t, h, k] * w[h, k, j] for k in range(K)]
                y[t, h, j] = float(np.float32(scale)) * math.fsum(prods)
                mag[t, h, j] = abs(float(np.float32(scale))) * math.fsum(abs(p) for p in prods)
    return y, mag


@pytest.mark.parametrize("w_dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("k,n", [(16, 16), (24, 40), (64, 8)])
def test_brute_force(w_dtype, k, n):
    inp = mi.bmm_inputs(3, 2, k, n, w_dtype, seed=k * 100 + n)
    y = ab.absorb_bmm(inp.x_bits, inp.w_bits, w_dtype, inp.w_scale)
    ref, mag = _brute(inp.x_bits, inp.w_bits, w_dtype, inp.w_scale)
    assert y.shape == ref.shape
    assert np.all(np.abs(y - ref) <= 1e-14 * mag + 1e-300)


@pytest.mark.parametrize("w_dtype", ["bf16", "fp8"])
def test_selection_weight_is_exact(w_dtype):
    rng = np.random.default_rng(5)
    H, K, N = 3, 32, 48
    inp = mi.bmm_inputs(4, H, K, N, "bf16", seed=6)
    pick = rng.integers(0, K, size=(H, N))
    one = 0x3F80 if w_dtype == "bf16" else 0x38           # the codes of 1.0
    w = np.zeros((H, K, N), np.uint16 if w_dtype == "bf16" else np.uint8)
    for h in range(H):
        w[h, pick[h], np.arange(N)] = one
    scale = 0.25 if w_dtype == "fp8" else 1.0
    y = ab.absorb_bmm(inp.x_bits, w, w_dtype, scale)
    x = _torch_decode(inp.x_bits, "bf16")
    for h in range(H):
        assert np.array_equal(y[:, h, :], scale * x[:, h, pick[h]])


def test_absorbed_attention_equals_up_projected_attention():
    """q_nope W_UK k_c^T = q_nope (k_c W_UK^T)^T and (P k_c) W_UV = P (k_c W_UV)."""
    rng = np.random.default_rng(7)
    T, H, L, dn, dl, dr, dv = 3, 4, 19, 128, 512, 64, 128
    q_nope = rng.standard_normal((T, H, dn))
    q_pe = rng.standard_normal((T, H, dr))
    c = rng.standard_normal((L, dl))
    k_pe = rng.standard_normal((L, dr))
    W_UK = rng.standard_normal((H, dn, dl)) / math.sqrt(dn)
    W_UV = rng.standard_normal((H, dl, dv)) / math.sqrt(dl)
    sigma = 1.0 / math.sqrt(192.0)

    # absorbed: the oracle's BMM, the decode oracle's attention over latent rows, the BMM again
    q_lat = ab.head_bmm_f64(q_nope, W_UK)
    qrows = np.concatenate([q_lat, q_pe], axis=-1).reshape(T * H, dl + dr)
    KV = np.concatenate([c, k_pe], axis=1)
    o_lat, lse = mo.attend_rows(qrows, KV, np.ones((T * H, L), bool), sigma)
    out = ab.head_bmm_f64(o_lat.reshape(T, H, dl), W_UV)

    # multi-head attention with per-head keys [k_nope | k_pe] and values up-projected
    want = np.empty((T, H, dv))
    for h in range(H):
        k_nope = c @ W_UK[h].T                     # [L, 128]
        v = c @ W_UV[h]                            # [L, 128]
        s = sigma * (q_nope[:, h] @ k_nope.T + q_pe[:, h] @ k_pe.T)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        want[:, h] = (p / p.sum(axis=1, keepdims=True)) @ v
    assert np.allclose(out, want, rtol=1e-10, atol=1e-12)


def test_planted_head_mixup_fails(monkeypatch):
    orig = ab.head_bmm_f64

    def wrong(x, w, scale=1.0):
        w = np.asarray(w)
        return orig(x, np.broadcast_to(w[:1], w.shape), scale)

    monkeypatch.setattr(ab, "head_bmm_f64", wrong)
    with pytest.raises(AssertionError):
        test_absorbed_attention_equals_up_projected_attention()


def test_planted_transpose_fails(monkeypatch):
    orig = ab.head_bmm_f64

    def wrong(x, w, scale=1.0):
        return orig(x, np.swapaxes(np.asarray(w), 1, 2), scale)

    monkeypatch.setattr(ab, "head_bmm_f64", wrong)
    with pytest.raises(AssertionError):
        test_brute_force("bf16", 16, 16)


def test_planted_dropped_scale_fails(monkeypatch):
    orig = ab.head_bmm_f64
    monkeypatch.setattr(ab, "head_bmm_f64", lambda x, w, scale=1.0: orig(x, w, 1.0))
    with pytest.raises(AssertionError):
        test_selection_weight_is_exact("fp8")
