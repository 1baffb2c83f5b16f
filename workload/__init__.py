"""Seeded synthetic inputs for the sparse-KV reuse decode step.

This module is the one thing the CPU oracle and the CUDA path share: it draws
the top-k selections, the queries and the host K/V rows, and holds none of the
method's arithmetic.  The generator itself is plain C (``gen.c``), compiled on
first use with the host compiler; see ``gen.c`` for the random streams and the
selection recipe, and ``configs.py`` for the five workload shapes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .configs import WORKLOADS, Workload, get_workload  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "_gen.so")
_lock = threading.Lock()
_lib = None

PURPOSE_K, PURPOSE_V, PURPOSE_Q, PURPOSE_SEL = 1, 2, 3, 4
DEFAULT_SEED = 0x5EED


class _SelParams(ctypes.Structure):
    _fields_ = [
        ("units", ctypes.c_int32),
        ("num_entries", ctypes.c_int32),
        ("k", ctypes.c_int32),
        ("steps", ctypes.c_int32),
        ("tokens", ctypes.c_int32),
        ("p_keep", ctypes.c_double),
        ("p_keep_token", ctypes.c_double),
        ("zipf_frac", ctypes.c_double),
        ("zipf_s", ctypes.c_double),
        ("num_forced", ctypes.c_int32),
        ("forced", ctypes.POINTER(ctypes.c_int32)),
        ("seed", ctypes.c_uint64),
        ("unit_base", ctypes.c_int32),
    ]


def build_generator(force: bool = False) -> str:
    """Compile gen.c into _gen.so next to it (host compiler, portable flags)."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_generator())
        lib.gen_normal.restype = ctypes.c_int
        lib.gen_normal.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                   ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64,
                                   ctypes.c_int64, ctypes.c_int]
        lib.gen_selections.restype = ctypes.c_int
        lib.gen_selections.argtypes = [ctypes.c_void_p, ctypes.POINTER(_SelParams),
                                       ctypes.c_int]
        _lib = lib
    return _lib


def _threads() -> int:
    """Generator threads: WORKLOAD_THREADS if set, else every core (at most 64)."""
    env = os.environ.get("WORKLOAD_THREADS", "")
    if env.isdigit() and int(env) > 0:
        return int(env)
    return max(1, min(64, os.cpu_count() or 1))


def fill_normal(out: np.ndarray, per_stream: int, purpose: int, seed: int = DEFAULT_SEED,
                stream_base: int = 0) -> np.ndarray:
    """Fill a C-contiguous array with N(0,1) draws: uint16 arrays get bf16 bit
    patterns (round-to-nearest-even), float32 arrays get fp32 values.  The
    array is viewed as [n_streams][per_stream]; stream s is keyed by
    (seed, purpose, stream_base + s), so a slice of streams can be drawn alone."""
    if not out.flags["C_CONTIGUOUS"]:
        raise ValueError("output must be C-contiguous")
    if out.dtype == np.uint16:
        is_bf16 = 1
    elif out.dtype == np.float32:
        is_bf16 = 0
    else:
        raise TypeError("output must be uint16 (bf16 bits) or float32")
    if out.size % per_stream:
        raise ValueError("size is not a multiple of per_stream")
    rc = _load().gen_normal(out.ctypes.data, is_bf16, out.size // per_stream, per_stream,
                            seed, purpose, stream_base, _threads())
    if rc:
        raise RuntimeError(f"gen_normal failed ({rc})")
    return out


def selections(w: Workload, steps: int | None = None, seed: int = DEFAULT_SEED,
               unit_base: int = 0) -> np.ndarray:
    """Top-k selections, int32 [steps][units][tokens_per_step][k]; unit u is
    drawn as unit ``unit_base + u`` of a larger job."""
    steps = w.steps if steps is None else steps
    out = np.empty((steps, w.units, w.tokens_per_step, w.k), dtype=np.int32)
    forced = np.ascontiguousarray(w.forced_ids(), dtype=np.int32)
    p = _SelParams(w.units, w.num_entries, w.k, steps, w.tokens_per_step,
                   w.p_keep, w.p_keep_token, w.zipf_frac, w.zipf_s, len(forced),
                   forced.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), seed, int(unit_base))
    rc = _load().gen_selections(out.ctypes.data, ctypes.byref(p), _threads())
    if rc:
        raise RuntimeError(f"gen_selections failed ({rc})")
    return out


def queries(w: Workload, steps: int | None = None, seed: int = DEFAULT_SEED,
            step_base: int = 0, unit_base: int = 0, units_total: int | None = None) -> np.ndarray:
    """Queries, float32 [steps][units][tokens_per_step][q_per_kv][head_dim].
    The stream of (step t, unit u) is t * units_total + unit_base + u: the
    units are units [unit_base, unit_base + units) of a job of units_total."""
    steps = w.steps if steps is None else steps
    total = w.units if units_total is None else int(units_total)
    out = np.empty((steps, w.units, w.tokens_per_step, w.q_per_kv, w.head_dim),
                   dtype=np.float32)
    per = w.tokens_per_step * w.q_per_kv * w.head_dim
    if unit_base == 0 and total == w.units:
        return fill_normal(out, per, PURPOSE_Q, seed, stream_base=step_base * w.units)
    for t in range(steps):
        fill_normal(out[t], per, PURPOSE_Q, seed, stream_base=(step_base + t) * total + unit_base)
    return out


def host_kv_shape(w: Workload) -> tuple:
    """Host K (or V) array shape: [units][num_entries][entry_tokens * width]."""
    return (w.units, w.num_entries, w.entry_tokens * w.head_dim)


def fill_host_kv(w: Workload, k_out: np.ndarray, v_out: np.ndarray | None,
                 seed: int = DEFAULT_SEED, unit_base: int = 0) -> None:
    """Fill caller-owned host K (and V unless K and V are shared) bf16 arrays,
    uint16 storage, shape ``host_kv_shape(w)`` (V uses v_dim); unit u's rows
    are those of unit ``unit_base + u``."""
    per_unit = w.num_entries * w.entry_tokens * w.head_dim
    fill_normal(k_out.reshape(-1), per_unit, PURPOSE_K, seed, stream_base=unit_base)
    if not w.kv_shared:
        if v_out is None:
            raise ValueError("V output required when K and V are separate")
        fill_normal(v_out.reshape(-1), w.num_entries * w.entry_tokens * w.v_dim,
                    PURPOSE_V, seed, stream_base=unit_base)


def host_kv(w: Workload, seed: int = DEFAULT_SEED):
    """Allocate and fill host K/V with numpy (unpinned; for small workloads)."""
    k = np.empty(host_kv_shape(w), dtype=np.uint16)
    v = None
    if not w.kv_shared:
        v = np.empty((w.units, w.num_entries, w.entry_tokens * w.v_dim), dtype=np.uint16)
    fill_host_kv(w, k, v, seed)
    return k, v
