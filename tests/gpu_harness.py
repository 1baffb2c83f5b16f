"""Runs the CUDA path (through the C interface) and the CPU oracle side by side
on the same seeded inputs and compares them step by step."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workload as W
from decode_serving_gb300.session import PinnedArray, Session, make_config

# Attention output: max abs error against the fp64 oracle (the bar the
# spec target sets for bf16 K/V with fp32 accumulation).
ATTN_TOL = 5e-3


def make_host_kv(w):
    hk = PinnedArray(W.host_kv_shape(w), np.uint16)
    hv = None
    if not w.kv_shared:
        hv = PinnedArray((w.units, w.num_entries, w.entry_tokens * w.v_dim), np.uint16)
    W.fill_host_kv(w, hk.array, hv.array if hv is not None else None)
    return hk, hv


def make_session(w, hk, hv, no_reuse=False, request_gather=False, initial_entries=0):
    cfg = make_config(w.requests, w.kv_heads, w.q_per_kv, w.num_entries, w.head_dim, w.v_dim,
                      w.slots, w.k, entry_tokens=w.entry_tokens, kv_shared=w.kv_shared,
                      max_tokens_per_step=w.tokens_per_step, no_reuse=no_reuse,
                      request_gather=request_gather, initial_entries=initial_entries)
    return Session(cfg, hk.ptr, hv.ptr if hv is not None else None)


def distinct_hits(sel_u, hit_u):
    """Distinct ids of one unit's step that the GPU flagged as hits."""
    return np.unique(sel_u[hit_u.astype(bool)]).size


class Parity:
    """GPU and oracle over the same inputs; ``units`` limits the oracle side,
    ``attn_units`` (default: all of ``units``) the units whose attention
    output the oracle computes and compares."""

    def __init__(self, w, steps=None, units=None, sel=None, q=None, no_reuse=False, seed=W.DEFAULT_SEED,
                 request_gather=False, initial_entries=0, attn_units=None):
        self.w = w
        self.steps = w.steps if steps is None else steps
        self.sel = W.selections(w, self.steps, seed=seed) if sel is None else sel
        self.q = W.queries(w, self.steps, seed=seed) if q is None else q
        self.units = list(range(w.units)) if units is None else list(units)
        self.attn_units = None if attn_units is None else set(attn_units)
        self.no_reuse = no_reuse
        self.hk, self.hv = make_host_kv(w)
        self.sess = make_session(w, self.hk, self.hv, no_reuse, request_gather, initial_entries)
        if initial_entries:
            # appends write the GPU side's host arrays: the oracle keeps its own copy
            self.ref = oracle.OracleRun(w.slots, self.hk.array.copy(),
                                        None if self.hv is None else self.hv.array.copy(),
                                        w.head_dim, w.v_dim, w.softmax_scale, units=self.units,
                                        live=initial_entries)
        else:
            self.ref = oracle.OracleRun(w.slots, self.hk.array,
                                        None if self.hv is None else self.hv.array,
                                        w.head_dim, w.v_dim, w.softmax_scale, units=self.units)
        dev = torch.device("cuda")
        shape = (w.units, w.tokens_per_step, w.k)
        self.out = torch.empty((w.units, w.tokens_per_step, w.q_per_kv, w.v_dim), dtype=torch.float32,
                               device=dev)
        self.sm = torch.empty(shape, dtype=torch.int32, device=dev)
        self.hit = torch.empty(shape, dtype=torch.uint8, device=dev)
        self.max_err = 0.0
        self.gpu_hits = 0
        self.ref_hits = 0

    def step(self, t, ti=None):
        """Run step index ti (into the input arrays) at step value t; compare."""
        ti = t if ti is None else ti
        w = self.w
        sel_t, q_t = self.sel[ti], self.q[ti]
        sel_d = torch.from_numpy(np.ascontiguousarray(sel_t)).cuda()
        q_d = torch.from_numpy(np.ascontiguousarray(q_t)).cuda()
        self.sess.step(t, sel_d, q_d, self.out, self.sm, self.hit)
        torch.cuda.synchronize()
        sm, hit, out = self.sm.cpu().numpy(), self.hit.cpu().numpy(), self.out.cpu().numpy()
        if self.no_reuse:
            for u in self.units:
                for j in range(w.tokens_per_step):
                    assert (sm[u, j] == j * w.k + np.arange(w.k)).all()
                    assert (hit[u, j] == 0).all()
                    o = oracle.attention_from_host(q_t[u][j], self.ref.host_k[u],
                                                   None if self.ref.host_v is None else self.ref.host_v[u],
                                                   sel_t[u][j], w.softmax_scale, w.head_dim, w.v_dim)
                    self.max_err = max(self.max_err, float(np.abs(out[u, j] - o).max()))
            assert self.max_err <= ATTN_TOL, self.max_err
            return None
        if self.attn_units is None:
            res = self.ref.step(t, sel_t, q_t)
        else:
            res = self.ref.step(t, sel_t, q_t, attention=False)
            for u in self.attn_units:
                st = self.ref.state[u]
                res[u] = (res[u][0], np.stack([
                    oracle.attention_from_host(q_t[u][j], st.host_k, st.host_v, sel_t[u][j],
                                               w.softmax_scale, w.head_dim, w.v_dim)
                    for j in range(w.tokens_per_step)]))
        for u in self.units:
            r, o = res[u]
            for j in range(w.tokens_per_step):
                assert (sm[u, j] == r.slot_maps[j]).all(), f"slot map t={t} unit={u} token={j}"
                assert (hit[u, j] == r.hit_flags[j]).all(), f"hit flags t={t} unit={u} token={j}"
            g = distinct_hits(sel_t[u], hit[u])
            assert g == r.hits, f"distinct hits t={t} unit={u}: {g} vs {r.hits}"
            self.gpu_hits += g
            self.ref_hits += r.hits
            if o is None:
                continue
            err = float(np.abs(out[u] - o).max())
            self.max_err = max(self.max_err, err)
            assert err <= ATTN_TOL, f"attention error {err} t={t} unit={u}"
        return res

    def append(self, k_rows, v_rows=None):
        """One new entry per unit on both sides: k_rows / v_rows uint16 [U][row]."""
        kd = torch.from_numpy(np.ascontiguousarray(k_rows).view(np.int16)).cuda()
        vd = None if v_rows is None else torch.from_numpy(np.ascontiguousarray(v_rows).view(np.int16)).cuda()
        self.sess.append(kd, vd)
        self.ref.append(k_rows, v_rows)

    def check_state(self, rows=True):
        for u in self.units:
            st = self.ref.state[u]
            tag, last, kr, vr = self.sess.read_state(u, rows=rows)
            assert (tag == st.tag).all(), f"tag unit={u}"
            assert (last == st.last).all(), f"last_step unit={u}"
            if rows:
                assert (kr == st.k_rows).all(), f"K rows unit={u}"
                if vr is not None:
                    assert (vr == st.v_rows).all(), f"V rows unit={u}"

    def run(self, state_every=8, rows_every=True):
        """All steps; tags and last_step compared every ``state_every`` steps
        and after the last, buffer rows with them (``rows_every``) or only
        after the last step."""
        for t in range(self.steps):
            self.step(t)
            last = t == self.steps - 1
            if not self.no_reuse and (t % state_every == state_every - 1 or last):
                self.check_state(rows=rows_every or last)
        return self

    def close(self):
        self.sess.close()
        self.hk.free()
        if self.hv is not None:
            self.hv.free()
