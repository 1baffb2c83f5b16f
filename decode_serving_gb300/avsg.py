"""Python binding of libavsg (include/avsg.h): argument marshalling only.

Every function keeps the C name and raises ``AvsgError`` on a non-zero return.
Pointers are plain integers (``tensor.data_ptr()``, ``array.ctypes.data``);
streams are ``torch.cuda.Stream.cuda_stream`` integers or 0.  All compute runs
in the CUDA kernels of the library; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libavsg.so")

AVSG_OK = 0
AVSG_ERR_INVALID_ARG = -1
AVSG_ERR_CAPACITY = -2
AVSG_ERR_CUDA = -3
AVSG_ERR_BAD_SELECTION = -4
AVSG_ERR_TIMEOUT = -5
AVSG_ERR_BAD_STEP = -6
AVSG_ERR_UNSUPPORTED = -7
AVSG_ERR_LATCHED = -8
AVSG_ERR_INTERNAL = -9
AVSG_FLAG_NO_REUSE = 1
AVSG_FLAG_REQUEST_GATHER = 2

ERROR_NAMES = {0: "OK", -1: "INVALID_ARG", -2: "CAPACITY", -3: "CUDA", -4: "BAD_SELECTION",
               -5: "TIMEOUT", -6: "BAD_STEP", -7: "UNSUPPORTED", -8: "LATCHED", -9: "INTERNAL"}


class avsg_config(ctypes.Structure):
    _fields_ = [
        ("num_requests", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("q_per_kv", ctypes.c_int32),
        ("entry_tokens", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("v_dim", ctypes.c_int32),
        ("kv_shared", ctypes.c_int32),
        ("reserved0", ctypes.c_int32),
        ("num_entries", ctypes.c_int64),
        ("buffer_slots", ctypes.c_int32),
        ("max_select", ctypes.c_int32),
        ("max_tokens_per_step", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("flags", ctypes.c_uint32),
        ("initial_entries", ctypes.c_int32),
    ]


class avsg_stats(ctypes.Structure):
    _fields_ = [
        ("steps", ctypes.c_uint64),
        ("selected", ctypes.c_uint64),
        ("unique_selected", ctypes.c_uint64),
        ("hits", ctypes.c_uint64),
        ("misses", ctypes.c_uint64),
        ("miss_bytes", ctypes.c_uint64),
        ("device_error", ctypes.c_int32),
        ("error_unit", ctypes.c_int32),
        ("error_position", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class avsg_info(ctypes.Structure):
    _fields_ = [
        ("device_bytes", ctypes.c_uint64),
        ("hash_capacity", ctypes.c_int32),
        ("miss_set_capacity", ctypes.c_int32),
        ("attn_splits", ctypes.c_int32),
        ("gather_ctas", ctypes.c_int32),
        ("num_sms", ctypes.c_int32),
        ("host_registered", ctypes.c_int32),
    ]


AVSG_NUM_KERNELS = 8


class avsg_kernel_times(ctypes.Structure):
    _fields_ = [("ms", ctypes.c_double * AVSG_NUM_KERNELS),
                ("launches", ctypes.c_uint64 * AVSG_NUM_KERNELS)]


KERNEL_NAMES = ("match", "victims", "gather", "attention", "attention_miss", "commit", "finish",
                "place")

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
SIGNATURES = {
    "avsg_create": [ctypes.POINTER(avsg_config), _P, _P, ctypes.POINTER(_P)],
    "avsg_destroy": [_P],
    "avsg_step": [_P, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P],
    "avsg_step_host": [_P, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P],
    "avsg_append": [_P, _P, _P, _P],
    "avsg_set_budget": [_P, _P, _P],
    "avsg_plan_budget": [ctypes.c_int64, _I32, _I32, _I32, _P, _P],
    "avsg_get_stats": [_P, ctypes.POINTER(avsg_stats)],
    "avsg_get_info": [_P, ctypes.POINTER(avsg_info)],
    "avsg_read_state": [_P, _I32, _P, _P, _P, _P],
    "avsg_reset": [_P, _P],
    "avsg_clear_error": [_P],
    "avsg_profile": [_P, _I32],
    "avsg_profile_read": [_P, ctypes.POINTER(avsg_kernel_times)],
    "avsg_host_alloc": [ctypes.c_size_t, ctypes.POINTER(_P)],
    "avsg_host_free": [_P],
    "avsg_strerror": [ctypes.c_int],
    "avsg_cuda_error": [_P],
    "avsg_attention_noalloc": [_I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _P,
                               _P, _P, ctypes.c_float, _P],
    "avsg_read_rows": [_P, ctypes.c_int64, ctypes.c_int64, _P, ctypes.c_int64, _I32, _P, _P],
}

_lib = None


class AvsgError(RuntimeError):
    def __init__(self, code: int, where: str, cuda: int = 0):
        msg = f"{where}: {ERROR_NAMES.get(code, code)}"
        if code == AVSG_ERR_CUDA and cuda:
            msg += f" (cudaError {cuda})"
        super().__init__(msg)
        self.code = code
        self.cuda = cuda


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libavsg.so (or the library AVSG_LIBRARY names, e.g. the
    bounds-checked build); raises if it has not been built (no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or os.environ.get("AVSG_LIBRARY") or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libavsg.so is not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    for name, args in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_char_p if name == "avsg_strerror" else ctypes.c_int
    _lib = lib
    return lib


def _check(rc: int, where: str, handle=None):
    if rc != AVSG_OK:
        cuda = load_library().avsg_cuda_error(handle) if (handle and rc == AVSG_ERR_CUDA) else 0
        raise AvsgError(rc, where, cuda)


def avsg_create(cfg: avsg_config, host_k: int, host_v: int | None) -> int:
    h = _P()
    _check(load_library().avsg_create(ctypes.byref(cfg), host_k, host_v or None, ctypes.byref(h)),
           "avsg_create")
    return h.value


def avsg_destroy(h: int) -> None:
    _check(load_library().avsg_destroy(h), "avsg_destroy")


def avsg_set_budget(h, slots_per_unit: np.ndarray, stream=0) -> None:
    a = np.ascontiguousarray(slots_per_unit, dtype=np.int32)
    _check(load_library().avsg_set_budget(h, a.ctypes.data, stream or None), "avsg_set_budget", h)


def avsg_plan_budget(total_slots: int, num_units: int, mandatory: int, max_slots: int,
                     weights=None) -> np.ndarray:
    out = np.zeros(num_units, np.int32)
    w = None if weights is None else np.ascontiguousarray(weights, dtype=np.float32)
    _check(load_library().avsg_plan_budget(int(total_slots), int(num_units), int(mandatory),
                                           int(max_slots), None if w is None else w.ctypes.data,
                                           out.ctypes.data), "avsg_plan_budget")
    return out


def avsg_append(h, d_k, d_v=0, stream=0) -> None:
    _check(load_library().avsg_append(h, d_k, d_v or None, stream or None), "avsg_append", h)


def avsg_step(h, t, n_tok, k, d_sel, d_q, d_out, d_slot_map=0, d_hit=0, stream=0) -> None:
    _check(load_library().avsg_step(h, t, n_tok, k, d_sel or None, d_q or None, d_out,
                                    d_slot_map or None, d_hit or None, stream or None),
           "avsg_step", h)


def avsg_step_host(h, t, n_tok, k, h_sel, h_q, h_out, h_slot_map=0, h_hit=0, stream=0) -> None:
    _check(load_library().avsg_step_host(h, t, n_tok, k, h_sel or None, h_q or None, h_out,
                                         h_slot_map or None, h_hit or None, stream or None),
           "avsg_step_host", h)


def avsg_get_stats(h) -> avsg_stats:
    st = avsg_stats()
    _check(load_library().avsg_get_stats(h, ctypes.byref(st)), "avsg_get_stats", h)
    return st


def avsg_get_info(h) -> avsg_info:
    info = avsg_info()
    _check(load_library().avsg_get_info(h, ctypes.byref(info)), "avsg_get_info", h)
    return info


def avsg_read_state(h, unit, tag=0, last_step=0, k_rows=0, v_rows=0) -> None:
    _check(load_library().avsg_read_state(h, unit, tag or None, last_step or None,
                                          k_rows or None, v_rows or None), "avsg_read_state", h)


def avsg_reset(h, stream=0) -> None:
    _check(load_library().avsg_reset(h, stream or None), "avsg_reset", h)


def avsg_clear_error(h) -> None:
    _check(load_library().avsg_clear_error(h), "avsg_clear_error", h)


def avsg_profile(h, enable: bool) -> None:
    _check(load_library().avsg_profile(h, 1 if enable else 0), "avsg_profile", h)


def avsg_profile_read(h) -> avsg_kernel_times:
    kt = avsg_kernel_times()
    _check(load_library().avsg_profile_read(h, ctypes.byref(kt)), "avsg_profile_read", h)
    return kt


def avsg_host_alloc(nbytes: int) -> int:
    p = _P()
    _check(load_library().avsg_host_alloc(nbytes, ctypes.byref(p)), "avsg_host_alloc")
    return p.value


def avsg_host_free(p: int) -> None:
    _check(load_library().avsg_host_free(p), "avsg_host_free")


def avsg_attention_noalloc(num_units, rows_per_unit, q_per_kv, head_dim, v_dim, entry_tokens,
                           kv_shared, n_tok, k, d_k_rows, d_v_rows, d_index, d_q, d_out,
                           softmax_scale=0.0, stream=0) -> None:
    """Attention over caller-held device rows; allocates nothing (see avsg.h)."""
    _check(load_library().avsg_attention_noalloc(
        num_units, rows_per_unit, q_per_kv, head_dim, v_dim, entry_tokens, 1 if kv_shared else 0,
        n_tok, k, d_k_rows, d_v_rows or None, d_index or None, d_q or None, d_out,
        float(softmax_scale), stream or None), "avsg_attention_noalloc")


def avsg_read_rows(src, num_rows, row_bytes, d_idx, n, d_sink, ctas=0, stream=0) -> None:
    """Reads n rows at the given indices and discards them (a measurement aid)."""
    _check(load_library().avsg_read_rows(src, int(num_rows), int(row_bytes), d_idx, int(n),
                                         int(ctas), d_sink, stream or None), "avsg_read_rows")


def avsg_strerror(code: int) -> str:
    return load_library().avsg_strerror(code).decode()


def avsg_cuda_error(h) -> int:
    return load_library().avsg_cuda_error(h)
