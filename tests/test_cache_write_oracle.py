"""Pins of the KV-cache write oracle (oracle/cache_write.py) to things other than itself.

* the fp8 encoder against torch's own float8_e4m3fn cast (a library routine) on
  every midpoint between neighbouring codes, one float32 step either side of it,
  and random values, wherever torch does not produce NaN (|y| < 464);
* the encoder against the decoder: every finite code encodes back to itself;
* saturation, NaN and signed zero from the format's definition;
* bf16 rounding against torch's .to(bfloat16);
* the write itself: the rows of the written slots, untouched slots, padding and
  out-of-range slots, strided (non-contiguous) input rows through the harness.
Planted mistakes (truncation instead of rounding, no saturation) must fail a pin.
"""
import numpy as np
import pytest

from oracle import cache_write as cw
from oracle import formats as fm

torch = pytest.importorskip("torch")


def _torch_e4m3(y):
    return torch.from_numpy(np.asarray(y, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _finite_codes():
    return np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def test_every_finite_code_encodes_back_to_itself():
    codes = _finite_codes()
    assert np.array_equal(cw.encode_e4m3fn_satfinite(fm.decode_e4m3fn(codes)), codes)


def test_encoder_matches_torch_on_midpoints_and_neighbours():
    v = np.sort(np.unique(fm.decode_e4m3fn(_finite_codes())))
    mids = (v[:-1] + v[1:]) / 2                       # exact in float32 for this grid
    m32 = mids.astype(np.float32)
    assert np.array_equal(m32.astype(np.float64), mids)
    up = np.nextafter(m32, np.float32(np.inf))
    dn = np.nextafter(m32, np.float32(-np.inf))
    rng = np.random.default_rng(3)
    rnd = (rng.standard_normal(20000) * rng.choice([1e-3, 0.05, 1, 30, 200], 20000)).astype(np.float32)
    y = np.concatenate([m32, up, dn, rnd, -m32, -up, -dn])
    y = y[np.abs(y) < 464]
    assert np.array_equal(cw.encode_e4m3fn_satfinite(y), _torch_e4m3(y))


def test_ties_go_to_the_even_code():
    # 1.0625 lies halfway between 1.0 (code 0x38, mantissa 0) and 1.125 (0x39)
    assert cw.encode_e4m3fn_satfinite(np.array([1.0625]))[0] == 0x38
    # 1.1875 lies halfway between 1.125 (0x39) and 1.25 (0x3A, even mantissa)
    assert cw.encode_e4m3fn_satfinite(np.array([1.1875]))[0] == 0x3A
    # half the smallest subnormal (2^-10) rounds to zero; 1.5 steps rounds to 2
    assert list(cw.encode_e4m3fn_satfinite(np.array([2.0 ** -10, 3 * 2.0 ** -10]))) == [0, 2]


def test_saturation_nan_and_signed_zero():
    y = np.array([448.0, 449.0, 464.0, 1e6, np.inf, -500.0, -np.inf, np.nan, -0.0, 0.0])
    assert list(cw.encode_e4m3fn_satfinite(y)) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F, 0x80, 0x00]


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal(50000) * rng.choice([1e-30, 1e-3, 1, 1e4, 1e30], 50000)).astype(np.float32)
    # exact ties: low 16 bits 0x8000 with both parities of the kept part
    u = rng.integers(0, 2 ** 31, 1000, dtype=np.uint64).astype(np.uint32)
    ties = ((u & 0xFFFF0000) | 0x8000).view(np.float32)
    x = np.concatenate([x, ties[np.isfinite(ties)]])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(cw.f32_to_bf16_rne(x), ref)


def test_planted_mistakes_fail_the_pins():
    y = np.array([1.0625, 1.1875, 449.0], dtype=np.float64)
    truncate = lambda v: cw.encode_e4m3fn_satfinite(np.floor(v * 8) / 8)  # noqa: E731
    assert not np.array_equal(truncate(np.array([1.1875])), cw.encode_e4m3fn_satfinite(np.array([1.1875])))
    # without saturation a value above 464 would become NaN, as torch's cast does
    assert _torch_e4m3(np.array([500.0]))[0] == 0x7F
    assert cw.encode_e4m3fn_satfinite(np.array([500.0]))[0] == 0x7E
    assert list(cw.encode_e4m3fn_satfinite(y)) == [0x38, 0x3A, 0x7E]


def test_write_places_rows_and_skips_padding_and_bad_slots():
    rng = np.random.default_rng(5)
    n, slots = 6, 10
    kv_c = rng.standard_normal((n, 512)).astype(np.float32)
    k_pe = rng.standard_normal((n, 64)).astype(np.float32)
    slot_mapping = np.array([3, -1, 7, 10, 0, 99], dtype=np.int32)   # -1 padding, 10/99 outside
    for kv_dtype, dt in (("bf16", np.uint16), ("fp8", np.uint8)):
        pool = rng.integers(0, 120, size=(slots, 576)).astype(dt)
        out = cw.cache_write(pool, kv_c, k_pe, slot_mapping, kv_dtype, kv_scale=0.05)
        for t, s in enumerate(slot_mapping):
            if 0 <= s < slots:
                row = np.concatenate([kv_c[t], k_pe[t]])
                want = cw.f32_to_bf16_rne(row) if kv_dtype == "bf16" else \
                    cw.encode_e4m3fn_satfinite((row * (np.float32(1) / np.float32(0.05))).astype(np.float32))
                assert np.array_equal(out[s], want)
        untouched = [s for s in range(slots) if s not in (3, 7, 0)]
        assert np.array_equal(out[untouched], pool[untouched])


def test_fp8_write_decodes_to_the_value_within_half_a_step():
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((4, 576)) * 3).astype(np.float32)
    pool = np.zeros((4, 576), np.uint8)
    out = cw.cache_write(pool, x[:, :512], x[:, 512:], np.arange(4), "fp8", kv_scale=0.05)
    back = fm.decode_e4m3fn(out) * 0.05
    # relative step of e4m3 is 2^-3: half a step is 1/16 of the magnitude (normal range)
    big = np.abs(x) > 0.05 * 2.0 ** -6 * 8
    assert np.all(np.abs(back - x)[big] <= np.abs(x)[big] / 16 * (1 + 1e-6))
