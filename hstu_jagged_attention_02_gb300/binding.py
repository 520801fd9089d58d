"""Thin Python binding of libhstu_attn.so (include/hstu_attn.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  PyTorch supplies device memory and the stream.
If the library cannot be loaded the import of the calls fails loudly; there
is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

from . import build as _build

HSTU_OK, HSTU_ERR_INVALID_ARG, HSTU_ERR_UNSUPPORTED, HSTU_ERR_WORKSPACE = 0, 1, 2, 3
HSTU_ERR_CUDA, HSTU_ERR_TIMEOUT, HSTU_ERR_DEVICE_CHECK = 4, 5, 6
HSTU_BF16, HSTU_FP32 = 0, 1
HSTU_NORM_NONE, HSTU_NORM_LAYERNORM = 0, 1
HSTU_FLAG_FORCE_SIMT = 1 << 0
HSTU_FLAG_TEST_TIMEOUT = 1 << 1
HSTU_FLAG_U_FP32 = 1 << 2
HSTU_FLAG_PLAN_BWD = 1 << 3
HSTU_FLAG_REUSE_PLAN = 1 << 4

_vp = ctypes.c_void_p


class hstu_attn_desc(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32), ("dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("B", ctypes.c_int32),
                ("H", ctypes.c_int32), ("d_qk", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("total_tokens", ctypes.c_int64), ("max_seq_len", ctypes.c_int32),
                ("alpha", ctypes.c_float), ("num_pos_buckets", ctypes.c_int32),
                ("num_time_buckets", ctypes.c_int32), ("norm", ctypes.c_int32),
                ("ln_eps", ctypes.c_float), ("flags", ctypes.c_uint32),
                ("dropout_p", ctypes.c_float), ("reserved", ctypes.c_uint32)]

_DROP = [("dropout_seed", ctypes.c_uint64), ("dropout_offset", ctypes.c_uint64)]


class hstu_attn_fwd_args(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("seq_offsets", "num_targets", "num_contexts", "timestamps",
                                   "rab_pos", "rab_time", "q", "k", "v", "u", "o", "y",
                                   "ln_mean", "ln_rstd")] + _DROP


class hstu_attn_bwd_args(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("seq_offsets", "num_targets", "num_contexts", "timestamps",
                                   "rab_pos", "rab_time", "q", "k", "v", "u", "o", "dy",
                                   "dq", "dk", "dv", "du", "d_rab_pos", "d_rab_time")] + _DROP


class hstu_layer_fwd_args(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("seq_offsets", "num_targets", "num_contexts", "timestamps",
                                   "rab_pos", "rab_time", "x", "w1", "w2", "out", "z1", "u", "vqk", "o", "y")] + _DROP


class hstu_layer_bwd_args(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("seq_offsets", "num_targets", "num_contexts", "timestamps",
                                   "rab_pos", "rab_time", "x", "w1", "w2", "z1", "u", "vqk", "o", "y",
                                   "dout", "dx", "dw1", "dw2", "d_rab_pos", "d_rab_time")] + _DROP


class hstu_attn_delta_args(ctypes.Structure):
    _fields_ = [("cand_offsets", _vp), ("cache_offsets", _vp), ("cache_tokens", ctypes.c_int64)] + \
        [(n, _vp) for n in ("cand_timestamps", "cache_timestamps", "rab_pos", "rab_time", "q", "k", "v", "u",
                            "k_cache", "v_cache", "o", "y", "ln_mean", "ln_rstd")]


EXPORTED = ("hstu_attn_workspace_size", "hstu_attn_fwd", "hstu_attn_bwd", "hstu_attn_debug_plan",
            "hstu_get_device_error", "hstu_status_string", "hstu_last_launch_count",
            "hstu_time_next_attention_kernel", "hstu_last_error_detail", "hstu_attn_fwd_noalloc",
            "hstu_layer_workspace_size", "hstu_layer_fwd", "hstu_layer_bwd", "hstu_attn_fwd_delta")

_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libhstu_attn.so (building it with nvcc if needed)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build() if build_if_missing else _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libhstu_attn.so not found at {path}; run the package build first")
    L = ctypes.CDLL(path)
    P = ctypes.POINTER
    L.hstu_attn_workspace_size.argtypes = [P(hstu_attn_desc), P(ctypes.c_size_t), P(ctypes.c_size_t)]
    L.hstu_attn_fwd.argtypes = [P(hstu_attn_desc), P(hstu_attn_fwd_args), _vp, ctypes.c_size_t, _vp]
    L.hstu_attn_bwd.argtypes = [P(hstu_attn_desc), P(hstu_attn_bwd_args), _vp, ctypes.c_size_t, _vp]
    L.hstu_attn_debug_plan.argtypes = [P(hstu_attn_desc), _vp, _vp, _vp, ctypes.c_int32, _vp,
                                       ctypes.c_size_t, _vp, ctypes.c_int64, P(ctypes.c_int64), _vp]
    L.hstu_get_device_error.argtypes = [_vp, _vp, P(ctypes.c_int32)]
    L.hstu_status_string.argtypes = [ctypes.c_int]
    L.hstu_status_string.restype = ctypes.c_char_p
    L.hstu_last_launch_count.restype = ctypes.c_int32
    L.hstu_time_next_attention_kernel.argtypes = [_vp, _vp]
    L.hstu_time_next_attention_kernel.restype = ctypes.c_int
    L.hstu_last_error_detail.restype = ctypes.c_char_p
    L.hstu_attn_fwd_noalloc.argtypes = [P(hstu_attn_desc), P(hstu_attn_fwd_args), _vp, P(ctypes.c_int32)]
    L.hstu_attn_fwd_noalloc.restype = ctypes.c_int
    L.hstu_layer_workspace_size.argtypes = [P(hstu_attn_desc), P(ctypes.c_size_t), P(ctypes.c_size_t)]
    L.hstu_layer_fwd.argtypes = [P(hstu_attn_desc), P(hstu_layer_fwd_args), _vp, ctypes.c_size_t, _vp]
    L.hstu_layer_bwd.argtypes = [P(hstu_attn_desc), P(hstu_layer_bwd_args), _vp, ctypes.c_size_t, _vp]
    L.hstu_attn_fwd_delta.argtypes = [P(hstu_attn_desc), P(hstu_attn_delta_args), _vp, ctypes.c_size_t, _vp]
    for name in ("hstu_attn_workspace_size", "hstu_attn_fwd", "hstu_attn_bwd", "hstu_attn_debug_plan",
                 "hstu_get_device_error", "hstu_layer_workspace_size", "hstu_layer_fwd", "hstu_layer_bwd",
                 "hstu_attn_fwd_delta"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


class HSTUError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {hstu_status_string(status)} (status {status})"
        if status == HSTU_ERR_CUDA:
            msg += f": {hstu_last_error_detail()}"
        super().__init__(msg)


def hstu_last_error_detail() -> str:
    return load().hstu_last_error_detail().decode()


def hstu_status_string(status: int) -> str:
    return load().hstu_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != HSTU_OK:
        raise HSTUError(status, where)


def make_desc(*, dtype: str, out_dtype: Optional[str] = None, B: int, H: int, d_qk: int, d_v: int, total_tokens: int,
              max_seq_len: int, alpha: float, num_pos_buckets: int = 128,
              num_time_buckets: int = 64, norm: str = "layernorm", ln_eps: float = 1e-5,
              flags: int = 0, dropout_p: float = 0.0) -> hstu_attn_desc:
    d = hstu_attn_desc()
    d.struct_size = ctypes.sizeof(hstu_attn_desc)
    d.dtype = HSTU_BF16 if dtype == "bf16" else HSTU_FP32
    d.out_dtype = d.dtype if out_dtype is None else (HSTU_BF16 if out_dtype == "bf16" else HSTU_FP32)
    d.B, d.H, d.d_qk, d.d_v = B, H, d_qk, d_v
    d.total_tokens = total_tokens
    d.max_seq_len = max_seq_len
    d.alpha = alpha
    d.num_pos_buckets, d.num_time_buckets = num_pos_buckets, num_time_buckets
    d.norm = HSTU_NORM_LAYERNORM if norm == "layernorm" else HSTU_NORM_NONE
    d.ln_eps = ln_eps
    d.flags = flags
    d.dropout_p = dropout_p
    return d


# ----------------------------------------------------------- raw C calls

def hstu_attn_workspace_size(desc: hstu_attn_desc):
    f, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(load().hstu_attn_workspace_size(ctypes.byref(desc), ctypes.byref(f), ctypes.byref(b)),
           "hstu_attn_workspace_size")
    return int(f.value), int(b.value)


def hstu_attn_fwd(desc, args, workspace: int, workspace_bytes: int, stream: int):
    _check(load().hstu_attn_fwd(ctypes.byref(desc), ctypes.byref(args), workspace, workspace_bytes,
                                stream), "hstu_attn_fwd")


def hstu_attn_bwd(desc, args, workspace: int, workspace_bytes: int, stream: int):
    _check(load().hstu_attn_bwd(ctypes.byref(desc), ctypes.byref(args), workspace, workspace_bytes,
                                stream), "hstu_attn_bwd")


def hstu_attn_fwd_noalloc(desc, args, stream: int, want_device_error: bool = True) -> Optional[int]:
    """The forward with the library's built-in scratch buffer (no workspace).
    Returns the device error code when want_device_error (the call then
    synchronises the stream), else None."""
    code = ctypes.c_int32(-1)
    _check(load().hstu_attn_fwd_noalloc(ctypes.byref(desc), ctypes.byref(args), stream,
                                        ctypes.byref(code) if want_device_error else None),
           "hstu_attn_fwd_noalloc")
    return int(code.value) if want_device_error else None


def hstu_attn_fwd_delta(desc, args, workspace: int, workspace_bytes: int, stream: int):
    _check(load().hstu_attn_fwd_delta(ctypes.byref(desc), ctypes.byref(args), workspace, workspace_bytes,
                                      stream), "hstu_attn_fwd_delta")


def hstu_layer_workspace_size(desc: hstu_attn_desc):
    f, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(load().hstu_layer_workspace_size(ctypes.byref(desc), ctypes.byref(f), ctypes.byref(b)),
           "hstu_layer_workspace_size")
    return int(f.value), int(b.value)


def hstu_layer_fwd(desc, args, workspace: int, workspace_bytes: int, stream: int):
    _check(load().hstu_layer_fwd(ctypes.byref(desc), ctypes.byref(args), workspace, workspace_bytes,
                                 stream), "hstu_layer_fwd")


def hstu_layer_bwd(desc, args, workspace: int, workspace_bytes: int, stream: int):
    _check(load().hstu_layer_bwd(ctypes.byref(desc), ctypes.byref(args), workspace, workspace_bytes,
                                 stream), "hstu_layer_bwd")


def hstu_get_device_error(workspace: int, stream: int) -> int:
    code = ctypes.c_int32(0)
    _check(load().hstu_get_device_error(workspace, stream, ctypes.byref(code)), "hstu_get_device_error")
    return int(code.value)


def hstu_last_launch_count() -> int:
    return int(load().hstu_last_launch_count())


def hstu_time_next_attention_kernel(start_event: Optional[int], stop_event: Optional[int]):
    _check(load().hstu_time_next_attention_kernel(start_event, stop_event), "hstu_time_next_attention_kernel")


def hstu_attn_debug_plan(desc, seq_offsets: int, num_targets: Optional[int], num_contexts: Optional[int],
                         pass_: int, workspace: int, workspace_bytes: int, capacity: int, stream: int):
    """Returns an int32 numpy array [n, 6] of (b, q_block, k_block, class, q_rows, k_rows)."""
    import numpy as np
    host = np.zeros((max(capacity, 1), 6), np.int32)
    n = ctypes.c_int64(0)
    _check(load().hstu_attn_debug_plan(ctypes.byref(desc), seq_offsets, num_targets, num_contexts, pass_,
                                       workspace, workspace_bytes, host.ctypes.data, capacity,
                                       ctypes.byref(n), stream), "hstu_attn_debug_plan")
    if n.value > capacity:
        raise HSTUError(HSTU_ERR_WORKSPACE, f"hstu_attn_debug_plan: {n.value} tiles > capacity {capacity}")
    return host[: n.value]
