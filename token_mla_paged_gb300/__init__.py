"""Python binding of the GB300 MLA paged-decode library (libmla_gb300.so).

Argument marshalling only: every step of the decode runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  The functions keep the
C ABI's names (include/mla_gb300.h); tensors are passed by data pointer and the
current torch stream is used unless one is given.

If the shared library is missing the import fails: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla_gb300.so")

MLA_OK = 0
MLA_KV_BF16, MLA_KV_FP8_E4M3 = 0, 1
MLA_OUT_BF16, MLA_OUT_FP32 = 0, 1
MLA_PLAN_STATIC, MLA_PLAN_DYNAMIC, MLA_PLAN_HOST = 0, 1, 2
MLA_ALGO_TENSOR, MLA_ALGO_CUDA_CORE = 0, 1
MLA_ACT_BF16, MLA_ACT_FP32 = 0, 1
MLA_ROPE_NEOX, MLA_ROPE_INTERLEAVED = 0, 1
MLA_W_BF16, MLA_W_FP8_E4M3 = 0, 1
D_QK, D_V = 576, 512

DEVICE_ERRORS = {0: "ok", 1: "kv index out of range", 2: "decreasing indptr",
                 3: "plan does not match the call", 4: "q length differs from the plan",
                 5: "bounded wait ran out", 6: "plan item capacity exceeded"}


class MlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {mla_status_string(status)} (status {status})")


class PlanParams(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("max_q_len", ctypes.c_int32), ("num_workers", ctypes.c_int32),
                ("kv_len_cap", ctypes.c_int64), ("mode", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class FwdArgs(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("kv_pool", ctypes.c_void_p), ("num_slots", ctypes.c_int64),
                ("kv_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
                ("kv_indptr", ctypes.c_void_p), ("kv_indices", ctypes.c_void_p),
                ("qo_indptr", ctypes.c_void_p), ("causal", ctypes.c_int32),
                ("pos_base", ctypes.c_int32), ("pos_stride", ctypes.c_int32),
                ("algo", ctypes.c_int32), ("pos_base_per_req", ctypes.c_void_p),
                ("g_kv_indptr", ctypes.c_void_p), ("softmax_scale", ctypes.c_float),
                ("kv_scale", ctypes.c_float), ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("params", ctypes.POINTER(PlanParams)), ("plan_d", ctypes.c_void_p),
                ("plan_bytes", ctypes.c_size_t), ("workspace_d", ctypes.c_void_p),
                ("ws_bytes", ctypes.c_size_t), ("kv_pos", ctypes.c_void_p), ("window", ctypes.c_int32),
                ("reserved2", ctypes.c_int32)]


class CacheWriteArgs(ctypes.Structure):
    _fields_ = [("kv_c", ctypes.c_void_p), ("kv_c_dtype", ctypes.c_int32), ("kv_c_stride", ctypes.c_int64),
                ("k_pe", ctypes.c_void_p), ("k_pe_dtype", ctypes.c_int32), ("k_pe_stride", ctypes.c_int64),
                ("slot_mapping", ctypes.c_void_p), ("num_tokens", ctypes.c_int64),
                ("kv_pool", ctypes.c_void_p), ("num_slots", ctypes.c_int64), ("kv_dtype", ctypes.c_int32),
                ("kv_scale", ctypes.c_float)]


class RopeArgs(ctypes.Structure):
    _fields_ = [("q_nope", ctypes.c_void_p), ("q_nope_stride_token", ctypes.c_int64),
                ("q_nope_stride_head", ctypes.c_int64), ("q_pe", ctypes.c_void_p),
                ("q_pe_stride_token", ctypes.c_int64), ("q_pe_stride_head", ctypes.c_int64),
                ("q_out", ctypes.c_void_p), ("num_heads", ctypes.c_int32), ("rope_style", ctypes.c_int32),
                ("kv_c", ctypes.c_void_p), ("kv_c_stride", ctypes.c_int64), ("k_pe", ctypes.c_void_p),
                ("k_pe_stride", ctypes.c_int64), ("positions", ctypes.c_void_p), ("cos_sin", ctypes.c_void_p),
                ("max_pos", ctypes.c_int64), ("slot_mapping", ctypes.c_void_p), ("num_tokens", ctypes.c_int64),
                ("kv_pool", ctypes.c_void_p), ("num_slots", ctypes.c_int64), ("kv_dtype", ctypes.c_int32),
                ("kv_scale", ctypes.c_float)]


class BmmArgs(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("x_stride_token", ctypes.c_int64), ("x_stride_head", ctypes.c_int64),
                ("w", ctypes.c_void_p), ("w_dtype", ctypes.c_int32), ("w_scale", ctypes.c_float),
                ("out", ctypes.c_void_p), ("out_stride_token", ctypes.c_int64),
                ("out_stride_head", ctypes.c_int64), ("num_tokens", ctypes.c_int32),
                ("num_heads", ctypes.c_int32), ("k", ctypes.c_int32), ("n", ctypes.c_int32),
                ("status_d", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; "
                          "g.build()'` first (there is no fallback path)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    pp = ctypes.POINTER(PlanParams)
    sig = {
        "mla_abi_version": (ctypes.c_int, []),
        "mla_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "mla_decode_plan_size": (ctypes.c_int, [pp, ctypes.POINTER(sz), ctypes.POINTER(sz)]),
        "mla_decode_plan": (ctypes.c_int, [pp, vp, vp, vp, sz]),
        "mla_decode_plan_device": (ctypes.c_int, [pp, vp, vp, vp, sz, vp, sz, vp]),
        "mla_decode_fwd": (ctypes.c_int, [ctypes.POINTER(FwdArgs), vp]),
        "mla_decode_fwd_noalloc": (ctypes.c_int, [ctypes.POINTER(FwdArgs), vp]),
        "mla_merge_states": (ctypes.c_int, [vp, i32, vp, i32, i64, i32, vp, i32, vp, vp]),
        "mla_cache_write": (ctypes.c_int, [ctypes.POINTER(CacheWriteArgs), vp]),
        "mla_rope_q_cache": (ctypes.c_int, [ctypes.POINTER(RopeArgs), vp]),
        "mla_absorb_bmm": (ctypes.c_int, [ctypes.POINTER(BmmArgs), vp]),
        "mla_get_device_error": (ctypes.c_int, [vp, vp, ctypes.POINTER(i32), ctypes.POINTER(i32)]),
        "mla_decode_workers": (ctypes.c_int, [i32, ctypes.POINTER(i32)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()

# Symbols the header declares; tests check the library exports each one.
ABI_SYMBOLS = ("mla_abi_version", "mla_status_string", "mla_decode_plan_size", "mla_decode_plan",
               "mla_decode_plan_device", "mla_decode_fwd", "mla_merge_states",
               "mla_get_device_error", "mla_decode_fwd_noalloc", "mla_cache_write", "mla_rope_q_cache",
               "mla_absorb_bmm", "mla_decode_workers")


def library():
    return _lib


def _check(status: int, where: str):
    if status != MLA_OK:
        raise MlaError(status, where)


def mla_abi_version() -> int:
    return int(_lib.mla_abi_version())


def mla_status_string(status: int) -> str:
    return _lib.mla_status_string(int(status)).decode()


def plan_params(batch: int, num_heads: int, max_q_len: int, num_workers: int,
                kv_len_cap: int = 0, mode: int = MLA_PLAN_DYNAMIC) -> PlanParams:
    return PlanParams(batch, num_heads, max_q_len, num_workers, kv_len_cap, mode, 0)


def mla_decode_workers(algo: int) -> int:
    """Work items the decode kernel of `algo` runs at once on the current device."""
    n = ctypes.c_int32(0)
    _check(_lib.mla_decode_workers(algo, ctypes.byref(n)), "mla_decode_workers")
    return int(n.value)


def mla_decode_plan_size(params: PlanParams) -> Tuple[int, int]:
    pb, wb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(_lib.mla_decode_plan_size(ctypes.byref(params), ctypes.byref(pb), ctypes.byref(wb)),
           "mla_decode_plan_size")
    return pb.value, wb.value


def mla_decode_plan(params: PlanParams, kv_indptr: Optional[np.ndarray],
                    qo_indptr: np.ndarray) -> np.ndarray:
    """Host plan as an int32 array (a pure function of its inputs)."""
    pb, _ = mla_decode_plan_size(params)
    out = np.zeros(pb // 4, dtype=np.int32)
    kv = None if kv_indptr is None else np.ascontiguousarray(kv_indptr, dtype=np.int32)
    qo = np.ascontiguousarray(qo_indptr, dtype=np.int32)
    _check(_lib.mla_decode_plan(ctypes.byref(params),
                                None if kv is None else kv.ctypes.data_as(ctypes.c_void_p),
                                qo.ctypes.data_as(ctypes.c_void_p),
                                out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(pb)),
           "mla_decode_plan")
    return out


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream))


def mla_decode_plan_device(params: PlanParams, kv_indptr, qo_indptr, plan_d, workspace_d,
                           stream=None) -> None:
    _check(_lib.mla_decode_plan_device(ctypes.byref(params), _ptr(kv_indptr), _ptr(qo_indptr),
                                       _ptr(plan_d), plan_d.numel() * plan_d.element_size(),
                                       _ptr(workspace_d),
                                       workspace_d.numel() * workspace_d.element_size(),
                                       _stream(stream)),
           "mla_decode_plan_device")


def mla_decode_fwd(*, q, kv_pool, kv_dtype: int, kv_indptr, kv_indices, qo_indptr, causal: bool,
                   softmax_scale: float, kv_scale: float, o, lse, params: PlanParams, plan_d,
                   workspace_d, pos_base: int = 0, pos_stride: int = 1, pos_base_per_req=None,
                   g_kv_indptr=None, algo: int = MLA_ALGO_TENSOR, kv_pos=None, window: int = 0,
                   stream=None) -> None:
    import torch
    out_dtype = MLA_OUT_FP32 if o.dtype == torch.float32 else MLA_OUT_BF16
    a = FwdArgs()
    a.q = _ptr(q)
    a.kv_pool = _ptr(kv_pool)
    a.num_slots = int(kv_pool.shape[0])
    a.kv_dtype = kv_dtype
    a.out_dtype = out_dtype
    a.kv_indptr = _ptr(kv_indptr)
    a.kv_indices = _ptr(kv_indices)
    a.qo_indptr = _ptr(qo_indptr)
    a.causal = 1 if causal else 0
    a.pos_base = pos_base
    a.pos_stride = pos_stride
    a.algo = algo
    a.pos_base_per_req = _ptr(pos_base_per_req)
    a.g_kv_indptr = _ptr(g_kv_indptr)
    a.softmax_scale = softmax_scale
    a.kv_scale = kv_scale
    a.o = _ptr(o)
    a.lse = _ptr(lse)
    a.params = ctypes.pointer(params)
    a.plan_d = _ptr(plan_d)
    a.plan_bytes = plan_d.numel() * plan_d.element_size()
    a.workspace_d = _ptr(workspace_d)
    a.ws_bytes = workspace_d.numel() * workspace_d.element_size()
    a.kv_pos = _ptr(kv_pos)
    a.window = int(window)
    _check(_lib.mla_decode_fwd(ctypes.byref(a), _stream(stream)), "mla_decode_fwd")


def mla_merge_states(o_parts, lse_parts, o, lse, stream=None) -> None:
    """o_parts [n, rows, dv] fp32|bf16, lse_parts fp32 [n, rows] -> o [rows, dv], lse [rows]."""
    import torch
    n, rows, dv = o_parts.shape
    _check(_lib.mla_merge_states(_ptr(o_parts), MLA_OUT_FP32 if o_parts.dtype == torch.float32
                                 else MLA_OUT_BF16, _ptr(lse_parts), n, rows, dv, _ptr(o),
                                 MLA_OUT_FP32 if o.dtype == torch.float32 else MLA_OUT_BF16,
                                 _ptr(lse), _stream(stream)),
           "mla_merge_states")


def _act_dtype(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return MLA_ACT_BF16
    if t.dtype == torch.float32:
        return MLA_ACT_FP32
    raise MlaError(1, f"mla_cache_write: unsupported activation dtype {t.dtype}")


def mla_cache_write(kv_c, k_pe, slot_mapping, kv_pool, kv_dtype: int, kv_scale: float = 1.0,
                    stream=None) -> None:
    """kv_c [n, 512] and k_pe [n, 64] (bf16 or fp32, unit stride along the row,
    k_pe may also be [n, 1, 64]); slot_mapping int32 [n]; kv_pool [slots, 576]."""
    if k_pe.dim() == 3:
        k_pe = k_pe.reshape(k_pe.shape[0], k_pe.shape[-1])
    if kv_c.stride(-1) != 1 or k_pe.stride(-1) != 1:
        raise MlaError(1, "mla_cache_write: rows must be contiguous along the columns")
    a = CacheWriteArgs()
    a.kv_c = _ptr(kv_c)
    a.kv_c_dtype = _act_dtype(kv_c)
    a.kv_c_stride = kv_c.stride(0)
    a.k_pe = _ptr(k_pe)
    a.k_pe_dtype = _act_dtype(k_pe)
    a.k_pe_stride = k_pe.stride(0)
    a.slot_mapping = _ptr(slot_mapping)
    a.num_tokens = int(slot_mapping.shape[0])
    a.kv_pool = _ptr(kv_pool)
    a.num_slots = int(kv_pool.shape[0])
    a.kv_dtype = kv_dtype
    a.kv_scale = kv_scale
    _check(_lib.mla_cache_write(ctypes.byref(a), _stream(stream)), "mla_cache_write")


def mla_rope_q_cache(q_nope, q_pe, q_out, kv_c, k_pe, positions, cos_sin, slot_mapping, kv_pool,
                     kv_dtype: int, kv_scale: float = 1.0, rope_style: int = MLA_ROPE_NEOX,
                     stream=None) -> None:
    """q_nope [n, H, 512], q_pe [n, H, 64], kv_c [n, 512], k_pe [n, 64] (bf16, unit
    stride along the row); q_out bf16 [n, H, 576] contiguous; positions and
    slot_mapping int32 [n]; cos_sin fp32 [max_pos, 64]; kv_pool [slots, 576]."""
    import torch
    for t in (q_nope, q_pe, kv_c, k_pe, q_out):
        if t.dtype != torch.bfloat16 or t.stride(-1) != 1:
            raise MlaError(1, "mla_rope_q_cache: activations must be bf16 with unit stride along the row")
    if not q_out.is_contiguous() or cos_sin.dtype != torch.float32 or not cos_sin.is_contiguous():
        raise MlaError(1, "mla_rope_q_cache: q_out must be contiguous and cos_sin contiguous fp32")
    a = RopeArgs()
    a.q_nope, a.q_nope_stride_token, a.q_nope_stride_head = _ptr(q_nope), q_nope.stride(0), q_nope.stride(1)
    a.q_pe, a.q_pe_stride_token, a.q_pe_stride_head = _ptr(q_pe), q_pe.stride(0), q_pe.stride(1)
    a.q_out, a.num_heads, a.rope_style = _ptr(q_out), int(q_nope.shape[1]), rope_style
    a.kv_c, a.kv_c_stride = _ptr(kv_c), kv_c.stride(0)
    a.k_pe, a.k_pe_stride = _ptr(k_pe), k_pe.stride(0)
    a.positions, a.cos_sin, a.max_pos = _ptr(positions), _ptr(cos_sin), int(cos_sin.shape[0])
    a.slot_mapping, a.num_tokens = _ptr(slot_mapping), int(slot_mapping.shape[0])
    a.kv_pool, a.num_slots, a.kv_dtype, a.kv_scale = _ptr(kv_pool), int(kv_pool.shape[0]), kv_dtype, kv_scale
    _check(_lib.mla_rope_q_cache(ctypes.byref(a), _stream(stream)), "mla_rope_q_cache")


def mla_get_device_error(workspace_d, stream=None) -> Tuple[int, int]:
    code, info = ctypes.c_int32(0), ctypes.c_int32(0)
    st = _lib.mla_get_device_error(_ptr(workspace_d), _stream(stream), ctypes.byref(code),
                                   ctypes.byref(info))
    if st not in (MLA_OK, 6):
        _check(st, "mla_get_device_error")
    return code.value, info.value


from .runner import DecodeRunner, default_workers_for  # noqa: E402  (plumbing: buffers + calls, no compute)
from .cp import gather_states, cp_merge  # noqa: E402  (plumbing: the CP exchange, then the merge kernel)


def mla_absorb_bmm(x, w, out, w_scale: float = 1.0, status=None, stream=None) -> None:
    """Per-head product out[t, h] = bf16(w_scale * x[t, h] @ w[h]).

    x bf16 [n, H, k] and out bf16 [n, H, n_out] (unit stride along the last dim,
    any token/head strides, e.g. a column slice of the 576-wide q); w [H, k, n_out]
    contiguous, bf16 or uint8 holding e4m3fn codes (float8_e4m3fn also accepted);
    status: optional int32 [2] device tensor for a wait timeout record."""
    import torch
    if x.dtype != torch.bfloat16 or out.dtype != torch.bfloat16 or x.stride(-1) != 1 or out.stride(-1) != 1:
        raise MlaError(1, "mla_absorb_bmm: x and out must be bf16 with unit stride along the last dim")
    if not w.is_contiguous():
        raise MlaError(1, "mla_absorb_bmm: w must be contiguous [H, k, n]")
    if w.dtype == torch.bfloat16:
        w_dtype = MLA_W_BF16
    elif w.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        w_dtype = MLA_W_FP8_E4M3
    else:
        raise MlaError(1, f"mla_absorb_bmm: unsupported weight dtype {w.dtype}")
    if w.dim() != 3 or x.dim() != 3 or out.dim() != 3 or w.shape[0] != x.shape[1] or w.shape[1] != x.shape[2] \
            or out.shape[:2] != x.shape[:2] or out.shape[2] != w.shape[2]:
        raise MlaError(1, "mla_absorb_bmm: shapes must be x [n, H, k], w [H, k, m], out [n, H, m]")
    a = BmmArgs()
    a.x, a.x_stride_token, a.x_stride_head = _ptr(x), x.stride(0), x.stride(1)
    a.w, a.w_dtype, a.w_scale = _ptr(w), w_dtype, w_scale
    a.out, a.out_stride_token, a.out_stride_head = _ptr(out), out.stride(0), out.stride(1)
    a.num_tokens, a.num_heads, a.k, a.n = int(x.shape[0]), int(x.shape[1]), int(x.shape[2]), int(w.shape[2])
    a.status_d = _ptr(status)
    _check(_lib.mla_absorb_bmm(ctypes.byref(a), _stream(stream)), "mla_absorb_bmm")
