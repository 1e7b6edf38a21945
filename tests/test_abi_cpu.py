"""CPU checks of the C ABI: the library loads, exports every declared symbol, and
its host planner reproduces the plan specification bit for bit."""
import os
import re

import numpy as np
import pytest

import token_mla_paged_gb300 as m
from oracle import plan_oracle as po

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "mla_gb300.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = m.library()
    decl = _declared()
    assert set(decl) == set(m.ABI_SYMBOLS)
    for name in decl:
        assert hasattr(lib, name), name


def test_abi_version_and_status_strings():
    hdr = open(os.path.join(ROOT, "include", "mla_gb300.h")).read()
    assert m.mla_abi_version() == int(re.search(r"#define MLA_ABI_VERSION (\d+)", hdr).group(1))
    for s in range(7):
        assert m.mla_status_string(s) and m.mla_status_string(s) != "unknown status"
    assert m.mla_status_string(99) == "unknown status"


def _host_vs_oracle(B, H, maxT, W, cap, mode, kvp, qop):
    params = m.plan_params(B, H, maxT, W, cap, mode)
    ours = m.mla_decode_plan(params, None if mode == po.STATIC else kvp, qop)
    ref = po.build_plan(B, H, maxT, W, cap, mode, kvp, qop)
    assert ours.shape == ref.shape
    assert np.array_equal(ours, ref)


def test_host_plan_matches_spec_worked_examples():
    import json
    cases = json.load(open(os.path.join(ROOT, "tests", "golden", "plan_worked_examples.json")))["cases"]
    for c in cases:
        kvp = None if c["kv_indptr"] is None else np.array(c["kv_indptr"], dtype=np.int32)
        _host_vs_oracle(c["batch"], c["num_heads"], c["max_q_len"], c["num_workers"], c["kv_len_cap"],
                        c["mode"], kvp, np.array(c["qo_indptr"], dtype=np.int32))


@pytest.mark.parametrize("seed", range(60))
def test_host_plan_matches_spec_random(seed):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(0, 70))
    H = int(rng.choice([1, 3, 16, 64, 96, 128]))
    maxT = int(rng.integers(0, 9))
    W = int(rng.integers(1, 400))
    mode = int(rng.integers(0, 3))
    T = rng.integers(0, maxT + 1, size=B)
    L = np.floor(np.exp(rng.uniform(0, np.log(300000), size=B))).astype(np.int64)
    L[rng.random(B) < 0.15] = 0
    kvp = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    qop = np.concatenate([[0], np.cumsum(T)]).astype(np.int32)
    cap = int(rng.integers(0, 200000))
    _host_vs_oracle(B, H, maxT, W, cap, mode, kvp, qop)


def test_host_plan_for_the_five_workloads():
    import mla_inputs as mi
    shapes = [(2, 16, 2, [37, 100], [2, 2]), (8, 64, 8, [8192] * 8, [8] * 8)]
    rng = np.random.default_rng(7)
    shapes.append((32, 128, 8, list(rng.integers(1024, 16385, 32)), [8] * 32))
    shapes.append((64, 128, 4, list(np.floor(np.exp(rng.uniform(np.log(256), np.log(131072), 64))).astype(int)),
                   list(rng.choice([1, 2, 4], 64))))
    shapes.append((128, 96, 8, [4096] * 128, [8] * 128))
    for B, H, maxT, L, T in shapes:
        for W in (1, 76, 152, 608):
            for mode in (po.STATIC, po.DYNAMIC, po.HOST):
                kvp = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
                qop = np.concatenate([[0], np.cumsum(T)]).astype(np.int32)
                _host_vs_oracle(B, H, maxT, W, 16384, mode, kvp, qop)
    assert mi.D_QK == 576


def test_plan_sizes_follow_the_bounds():
    p = m.plan_params(64, 128, 4, 76, 0, m.MLA_PLAN_DYNAMIC)
    plan_bytes, ws_bytes = m.mla_decode_plan_size(p)
    rows = po.ROWS                       # 256 query rows per item: 128 x 4 rows -> 2 groups
    g_max = -(-128 * 4 // rows)
    cap = 76 + 64 * g_max
    assert plan_bytes == 4 * (16 + 64 + 65 + 64 + 4 * cap)
    # partial O and LSE per item, two merge counters (one per row half) per group
    assert ws_bytes >= 4 * cap * rows * 512 + 4 * cap * rows + 4 * 2 * 64 * g_max + 256


def test_host_plan_rejects_bad_input():
    with pytest.raises(m.MlaError):
        m.mla_decode_plan(m.plan_params(2, 16, 2, 4, 0, m.MLA_PLAN_DYNAMIC),
                          np.array([0, 5, 3]), np.array([0, 1, 2]))
    with pytest.raises(m.MlaError):
        m.mla_decode_plan(m.plan_params(2, 16, 1, 4, 0, m.MLA_PLAN_DYNAMIC),
                          np.array([0, 5, 9]), np.array([0, 2, 3]))
    with pytest.raises(m.MlaError):
        m.mla_decode_plan(m.plan_params(2, 0, 1, 4, 0, m.MLA_PLAN_DYNAMIC),
                          np.array([0, 5, 9]), np.array([0, 1, 2]))
    with pytest.raises(m.MlaError):
        m.mla_decode_plan_size(m.plan_params(1, 16, 1, 0, 0, m.MLA_PLAN_DYNAMIC))
    with pytest.raises(m.MlaError):   # a HOST plan is built from the real lengths
        m.mla_decode_plan(m.plan_params(2, 16, 1, 4, 0, m.MLA_PLAN_HOST), None, np.array([0, 1, 2]))
    with pytest.raises(m.MlaError):   # no such mode
        m.mla_decode_plan(m.plan_params(2, 16, 1, 4, 0, 3), np.array([0, 5, 9]), np.array([0, 1, 2]))


def test_host_mode_plan_is_the_real_length_plan():
    """HOST and DYNAMIC plans are the same plan from the same lengths (only the
    header's mode word differs); a STATIC plan ignores the lengths."""
    rng = np.random.default_rng(5)
    L = rng.integers(1, 20000, size=24)
    kvp = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    qop = np.arange(0, 25 * 4, 4, dtype=np.int32)[:25]
    host = m.mla_decode_plan(m.plan_params(24, 128, 4, 76, 0, m.MLA_PLAN_HOST), kvp, qop)
    dyn = m.mla_decode_plan(m.plan_params(24, 128, 4, 76, 0, m.MLA_PLAN_DYNAMIC), kvp, qop)
    diff = np.nonzero(host != dyn)[0]
    assert list(diff) == [6] and host[6] == m.MLA_PLAN_HOST and dyn[6] == m.MLA_PLAN_DYNAMIC


def test_fwd_rejects_bad_arguments_before_touching_the_device():
    """Invalid host-visible arguments come back as a status; nothing is enqueued."""
    import ctypes
    lib = m.library()
    params = m.plan_params(1, 16, 1, 4, 0, m.MLA_PLAN_DYNAMIC)
    a = m.FwdArgs()
    a.params = ctypes.pointer(params)
    a.kv_dtype = 7
    assert lib.mla_decode_fwd(ctypes.byref(a), None) == 1
    a.kv_dtype = 0
    a.softmax_scale = float("nan")
    assert lib.mla_decode_fwd(ctypes.byref(a), None) == 1
    a.softmax_scale = 0.07
    a.pos_stride = 0
    assert lib.mla_decode_fwd(ctypes.byref(a), None) == 1
    a.pos_stride = 1
    a.window = -1
    assert lib.mla_decode_fwd(ctypes.byref(a), None) == 1      # negative window
    a.window = 0
    a.kv_pos = 18
    assert lib.mla_decode_fwd(ctypes.byref(a), None) == 1      # misaligned positions
    a.kv_pos = None
    a.num_slots = 10
    a.q = a.kv_pool = a.kv_indptr = a.kv_indices = a.qo_indptr = a.o = a.lse = 16
    a.plan_d = 256
    a.workspace_d = 256
    a.plan_bytes = 4
    a.ws_bytes = 1 << 30
    assert lib.mla_decode_fwd(ctypes.byref(a), None) == 3      # plan buffer too small
    a.plan_bytes = 1 << 20
    a.ws_bytes = 16
    assert lib.mla_decode_fwd(ctypes.byref(a), None) == 3      # workspace too small
    a.ws_bytes = 1 << 30
    a.workspace_d = None
    assert lib.mla_decode_fwd(ctypes.byref(a), None) != 0     # no workspace (e.g. during capture)
    a.workspace_d = 256
    a.q = 18
    assert lib.mla_decode_fwd(ctypes.byref(a), None) == 1      # misaligned q
    assert lib.mla_merge_states(None, 0, None, 0, 1, 512, None, 0, None, None) == 1


def test_cache_write_rejects_bad_arguments_before_touching_the_device():
    """mla_cache_write validates dtypes, sizes, strides and alignment on the host;
    an empty call returns before any CUDA work."""
    import ctypes
    lib = m.library()

    def args(**kw):
        a = m.CacheWriteArgs()
        a.kv_c, a.kv_c_dtype, a.kv_c_stride = 0x10000, m.MLA_ACT_BF16, 512
        a.k_pe, a.k_pe_dtype, a.k_pe_stride = 0x20000, m.MLA_ACT_BF16, 64
        a.slot_mapping, a.num_tokens = 0x30000, 0
        a.kv_pool, a.num_slots, a.kv_dtype, a.kv_scale = 0x40000, 16, m.MLA_KV_FP8_E4M3, 0.05
        for k, v in kw.items():
            setattr(a, k, v)
        return ctypes.byref(a)

    assert lib.mla_cache_write(args(), None) == 0                      # nothing to write
    assert lib.mla_cache_write(None, None) == 1
    assert lib.mla_cache_write(args(kv_c_dtype=2), None) == 1          # not an activation dtype
    assert lib.mla_cache_write(args(k_pe_dtype=-1), None) == 1
    assert lib.mla_cache_write(args(kv_dtype=2), None) == 1
    assert lib.mla_cache_write(args(kv_scale=0.0), None) == 1          # fp8 needs a scale
    assert lib.mla_cache_write(args(kv_scale=float("nan")), None) == 1
    assert lib.mla_cache_write(args(num_tokens=-1), None) == 1
    assert lib.mla_cache_write(args(num_slots=0), None) == 1
    assert lib.mla_cache_write(args(kv_c_stride=511), None) == 1
    assert lib.mla_cache_write(args(k_pe_stride=63), None) == 1
    # with tokens to write: null, misaligned or non-16-byte strides are refused
    assert lib.mla_cache_write(args(num_tokens=4, kv_c=None), None) == 1
    assert lib.mla_cache_write(args(num_tokens=4, k_pe=0x20008), None) == 1
    assert lib.mla_cache_write(args(num_tokens=4, kv_c_stride=516), None) == 1
    assert lib.mla_cache_write(args(num_tokens=4, k_pe_dtype=m.MLA_ACT_FP32, k_pe_stride=66), None) == 1


def test_rope_q_cache_rejects_bad_arguments_before_touching_the_device():
    import ctypes
    lib = m.library()

    def args(**kw):
        a = m.RopeArgs()
        a.q_nope, a.q_nope_stride_token, a.q_nope_stride_head = 0x10000, 1024, 512
        a.q_pe, a.q_pe_stride_token, a.q_pe_stride_head = 0x20000, 128, 64
        a.q_out, a.num_heads, a.rope_style = 0x30000, 2, m.MLA_ROPE_NEOX
        a.kv_c, a.kv_c_stride, a.k_pe, a.k_pe_stride = 0x40000, 512, 0x50000, 64
        a.positions, a.cos_sin, a.max_pos = 0x60000, 0x70000, 128
        a.slot_mapping, a.num_tokens = 0x80000, 0
        a.kv_pool, a.num_slots, a.kv_dtype, a.kv_scale = 0x90000, 16, m.MLA_KV_FP8_E4M3, 0.05
        for k, v in kw.items():
            setattr(a, k, v)
        return ctypes.byref(a)

    assert lib.mla_rope_q_cache(args(), None) == 0                      # nothing to do
    assert lib.mla_rope_q_cache(None, None) == 1
    assert lib.mla_rope_q_cache(args(rope_style=2), None) == 1
    assert lib.mla_rope_q_cache(args(num_heads=0), None) == 1
    assert lib.mla_rope_q_cache(args(max_pos=0), None) == 1
    assert lib.mla_rope_q_cache(args(kv_scale=-1.0), None) == 1
    assert lib.mla_rope_q_cache(args(kv_dtype=5), None) == 1
    assert lib.mla_rope_q_cache(args(num_tokens=3, q_out=None), None) == 1
    assert lib.mla_rope_q_cache(args(num_tokens=3, q_pe_stride_head=68), None) == 1   # not 16-byte rows
    assert lib.mla_rope_q_cache(args(num_tokens=3, kv_c=0x40008), None) == 1          # misaligned


def test_absorb_bmm_rejects_bad_arguments_before_touching_the_device():
    import ctypes
    lib = m.library()

    def args(**kw):
        a = m.BmmArgs()
        a.x, a.x_stride_token, a.x_stride_head = 0x10000, 4 * 128, 128
        a.w, a.w_dtype, a.w_scale = 0x20000, m.MLA_W_FP8_E4M3, 0.01
        a.out, a.out_stride_token, a.out_stride_head = 0x30000, 4 * 576, 576
        a.num_tokens, a.num_heads, a.k, a.n = 0, 4, 128, 512
        a.status_d = None
        for k, v in kw.items():
            setattr(a, k, v)
        return ctypes.byref(a)

    assert lib.mla_absorb_bmm(args(), None) == 0                         # nothing to do
    assert lib.mla_absorb_bmm(None, None) == 1
    assert lib.mla_absorb_bmm(args(k=96), None) == 1                     # k not a multiple of 64
    assert lib.mla_absorb_bmm(args(n=192), None) == 1                    # n not a multiple of 128
    assert lib.mla_absorb_bmm(args(num_heads=0), None) == 1
    assert lib.mla_absorb_bmm(args(num_heads=70000), None) == 1
    assert lib.mla_absorb_bmm(args(w_dtype=2), None) == 1
    assert lib.mla_absorb_bmm(args(w_scale=float("nan")), None) == 1
    assert lib.mla_absorb_bmm(args(x_stride_head=64), None) == 1         # rows overlap
    assert lib.mla_absorb_bmm(args(out_stride_head=500), None) == 1
    assert lib.mla_absorb_bmm(args(num_tokens=3, out_stride_token=4 * 576 + 4), None) == 1  # not 16-byte rows
    assert lib.mla_absorb_bmm(args(num_tokens=3, w=None), None) == 1
    assert lib.mla_absorb_bmm(args(num_tokens=3, x=0x10008), None) == 1  # misaligned
    assert lib.mla_absorb_bmm(args(num_tokens=3, status_d=0x40002), None) == 1
