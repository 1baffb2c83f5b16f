"""Resource handling around the C interface: pinned host KV and one handle.

Marshalling only -- every step runs in the library's CUDA kernels.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import avsg as C


class PinnedArray:
    """Pinned, mapped host memory (avsg_host_alloc) viewed as a numpy array."""

    def __init__(self, shape, dtype):
        self.shape = tuple(int(x) for x in shape)
        self.dtype = np.dtype(dtype)
        self.nbytes = int(np.prod(self.shape)) * self.dtype.itemsize
        self.ptr = C.avsg_host_alloc(max(self.nbytes, 1))
        buf = (ctypes.c_char * max(self.nbytes, 1)).from_address(self.ptr)
        self.array = np.frombuffer(buf, dtype=self.dtype, count=int(np.prod(self.shape))).reshape(self.shape)

    def free(self):
        if self.ptr:
            self.array = None
            C.avsg_host_free(self.ptr)
            self.ptr = 0

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def make_config(requests, kv_heads, q_per_kv, num_entries, head_dim, v_dim, buffer_slots,
                max_select, entry_tokens=1, kv_shared=False, max_tokens_per_step=1,
                softmax_scale=0.0, no_reuse=False, request_gather=False,
                initial_entries=0) -> C.avsg_config:
    flags = (C.AVSG_FLAG_NO_REUSE if no_reuse else 0) | (C.AVSG_FLAG_REQUEST_GATHER if request_gather else 0)
    return C.avsg_config(int(requests), int(kv_heads), int(q_per_kv), int(entry_tokens),
                         int(head_dim), int(v_dim), 1 if kv_shared else 0, 0, int(num_entries),
                         int(buffer_slots), int(max_select), int(max_tokens_per_step),
                         float(softmax_scale), flags, int(initial_entries))


class Session:
    """One handle.  host_k / host_v: integer addresses of the host KV (kept
    alive by the caller for the life of the session)."""

    def __init__(self, cfg: C.avsg_config, host_k: int, host_v: int | None):
        self.cfg = cfg
        self.handle = C.avsg_create(cfg, host_k, host_v)
        self.units = cfg.num_requests * cfg.num_kv_heads
        self.slots = cfg.buffer_slots

    def step(self, t, sel, q, out, slot_map=None, hit=None, stream=0):
        """sel [U][n_tok][k] int32, q [U][n_tok][G][D] fp32, out [U][n_tok][G][Dv]
        fp32, slot_map int32 / hit uint8 like sel: CUDA tensors (data_ptr)."""
        n_tok, k = int(sel.shape[-2]), int(sel.shape[-1])
        C.avsg_step(self.handle, int(t), n_tok, k, sel.data_ptr(), q.data_ptr(), out.data_ptr(),
                    slot_map.data_ptr() if slot_map is not None else 0,
                    hit.data_ptr() if hit is not None else 0, stream)

    def step_host(self, t, sel: np.ndarray, q: np.ndarray, out: np.ndarray, slot_map=None,
                  hit=None, stream=0):
        n_tok, k = int(sel.shape[-2]), int(sel.shape[-1])
        C.avsg_step_host(self.handle, int(t), n_tok, k, sel.ctypes.data, q.ctypes.data,
                         out.ctypes.data, slot_map.ctypes.data if slot_map is not None else 0,
                         hit.ctypes.data if hit is not None else 0, stream)

    def append(self, k_rows, v_rows=None, stream=0):
        """One new entry per unit (Offload): k_rows [U][entry_tokens*D] bf16 bits,
        v_rows like it for V (None when K and V are shared): CUDA tensors."""
        C.avsg_append(self.handle, k_rows.data_ptr(),
                      v_rows.data_ptr() if v_rows is not None else 0, stream)

    def set_budget(self, slots_per_unit, stream=0):
        """Usable slots per unit from the next step on (buffer elasticity)."""
        C.avsg_set_budget(self.handle, slots_per_unit, stream)

    def stats(self) -> C.avsg_stats:
        return C.avsg_get_stats(self.handle)

    def info(self) -> C.avsg_info:
        return C.avsg_get_info(self.handle)

    def read_state(self, unit: int, rows: bool = True):
        """(tag [B], last [B], k_rows [B][ek/2] uint16, v_rows or None)."""
        B = self.slots
        row_k = self.cfg.entry_tokens * self.cfg.head_dim
        row_v = self.cfg.entry_tokens * self.cfg.v_dim
        tag = np.empty(B, np.int32)
        last = np.empty(B, np.int32)
        kr = np.empty((B, row_k), np.uint16) if rows else None
        vr = np.empty((B, row_v), np.uint16) if rows and not self.cfg.kv_shared else None
        C.avsg_read_state(self.handle, unit, tag.ctypes.data, last.ctypes.data,
                          kr.ctypes.data if kr is not None else 0,
                          vr.ctypes.data if vr is not None else 0)
        return tag, last, kr, vr

    def reset(self, stream=0):
        C.avsg_reset(self.handle, stream)

    def clear_error(self):
        C.avsg_clear_error(self.handle)

    def profile(self, enable: bool):
        C.avsg_profile(self.handle, enable)

    def profile_read(self) -> dict:
        kt = C.avsg_profile_read(self.handle)
        return {name: (kt.ms[i], kt.launches[i]) for i, name in enumerate(C.KERNEL_NAMES)}

    def close(self):
        if self.handle:
            C.avsg_destroy(self.handle)
            self.handle = 0

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
