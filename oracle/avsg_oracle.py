"""Plain CPU oracle of the sparse-KV reuse decode step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code with the CUDA library.

What it computes, and where that comes from:

* The operator (AVSG page, arxivdaily 2609.37538, English abstract): for each
  (request, kv-head) *unit*, the step's dynamically selected token ids are
  matched against a device buffer of reusable slots; slots are reserved for the
  ids that are not resident; only those missing rows are copied from the host
  KV cache; entries stay resident across steps; in a multi-token-prediction
  iteration one shared reservation covers the tokens of the iteration; the
  token selection itself is kept exactly.
* The retention policy (Spin page, "Unifying Sparse Attention with Hierarchical
  Memory for Scalable Long-Context LLM Serving", section 2B, bucketed LRU with
  about 64 recency buckets).  The pages give no formula; the reading used here:
  empty slots are reserved first, by ascending slot index; then slots not
  selected in this step, by bucket min(63, t - last_step) from oldest to
  newest, ties by ascending slot index; the i-th missing id in ascending id
  order takes the i-th reserved slot; every selected id ends the step with
  last_step = t.
* The attention (Spin page, section 2A, the Attention operation): for every
  query head g of the unit, softmax(scale * q_g . K_j) over the selected rows j,
  then the probability-weighted sum of the V rows; computed in fp64, straight
  from the host KV rows of the selected ids, so it does not depend on the
  buffer at all.
* Offload (Spin page, section 2A, the Offload operation): a decode step's new
  KV entry is written to the host store; it is selectable from the next step
  on and, like any id, enters the buffer only as a miss.  Here the host store
  holds ``capacity`` entries per unit, of which the first ``live`` are
  selectable; ``append`` writes entry ``live`` and raises the count.
* Buffer elasticity (Spin page, section 2B): each unit's buffer is sized per
  step, mandatory slots (the current step's selection) plus buffer slots kept
  for locality, under a system-wide budget.  Here a unit has a budget of
  usable slots, slots [0, budget): lowering it drops the entries held at or
  above it, and the reservation takes only slots below it.

Everything is written as the plain definition: a dense id -> slot table, a
library sort for the victim order, a matmul and ``exp`` for attention.
Every function is pinned by ``tests/test_oracle_*.py`` (hand-worked examples,
brute force, invariants, closed forms); no function is parity unpinned.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

EMPTY = -1              # tag of a slot that holds no entry
EMPTY_BUCKET = 64       # empty slots rank before every occupied bucket
MAX_AGE_BUCKET = 63     # ages >= 63 share the oldest bucket (64 buckets, Spin 2B)

# Error kinds, named as in the C interface.
ERR_BAD_SELECTION = "BAD_SELECTION"
ERR_CAPACITY = "CAPACITY"
ERR_BAD_STEP = "BAD_STEP"


class OracleError(ValueError):
    def __init__(self, kind: str, msg: str):
        super().__init__(f"{kind}: {msg}")
        self.kind = kind


@dataclass
class StepResult:
    slot_maps: list      # per query token: int64 [k] slot of each selected id, input order
    hit_flags: list      # per query token: bool [k], id was resident before the step
    hits: int            # distinct selected ids that were resident
    misses: int          # distinct selected ids that had to be copied from host


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly: a bf16 value is the upper
    half of an IEEE-754 binary32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


class UnitBuffer:
    """The device buffer of one unit, as a plain state machine.

    host_k / host_v: this unit's host rows, uint16 [num_entries][row_elems]
    (bf16 bits; one row per entry, a 16-token page is one row of 16*D values).
    host_v is None when V aliases K (latent cache).
    """

    def __init__(self, num_slots: int, host_k: np.ndarray, host_v: np.ndarray | None = None,
                 live: int | None = None):
        self.B = int(num_slots)
        self.host_k = host_k
        self.host_v = host_v
        self.L = host_k.shape[0]            # capacity of the host store
        self.live = self.L if live is None else int(live)
        self.budget = self.B                # usable slots [0, budget)
        self.tag = np.full(self.B, EMPTY, dtype=np.int64)
        self.last = np.full(self.B, -1, dtype=np.int64)
        self.slot_of = np.full(self.L, EMPTY, dtype=np.int64)
        self.k_rows = np.zeros((self.B, host_k.shape[1]), dtype=np.uint16)
        self.v_rows = None if host_v is None else np.zeros((self.B, host_v.shape[1]), np.uint16)
        self.prev_t = None

    # -- validation ---------------------------------------------------------
    def _validate(self, t: int, sels: list) -> np.ndarray:
        if t < 0 or (self.prev_t is not None and t <= self.prev_t):
            raise OracleError(ERR_BAD_STEP, f"t={t} after t={self.prev_t}")
        for s in sels:
            if s.size and (s.min() < 0 or s.max() >= self.live):
                raise OracleError(ERR_BAD_SELECTION, "id out of range")
            if np.unique(s).size != s.size:
                raise OracleError(ERR_BAD_SELECTION, "duplicate id in one selection")
        union = np.unique(np.concatenate(sels)) if sels else np.zeros(0, np.int64)
        if union.size > self.budget:
            raise OracleError(ERR_CAPACITY, f"{union.size} distinct ids > {self.budget} usable slots")
        return union

    # -- offload ------------------------------------------------------------
    def append(self, k_row: np.ndarray, v_row: np.ndarray | None = None) -> int:
        """Writes a new entry to the host store; returns its id."""
        if self.live >= self.L:
            raise OracleError(ERR_CAPACITY, "host store full")
        self.host_k[self.live] = k_row
        if self.host_v is not None:
            self.host_v[self.live] = v_row
        self.live += 1
        return self.live - 1

    # -- elasticity -----------------------------------------------------------
    def set_budget(self, budget: int) -> None:
        """Usable slots [0, budget) from the next step on; entries held at or
        above a lowered budget are dropped."""
        budget = int(budget)
        if not 1 <= budget <= self.B:
            raise OracleError(ERR_CAPACITY, f"budget {budget} outside 1..{self.B}")
        for slot in range(budget, self.B):
            if self.tag[slot] != EMPTY:
                self.slot_of[self.tag[slot]] = EMPTY
                self.tag[slot] = EMPTY
                self.last[slot] = -1
        self.budget = budget

    # -- the step -----------------------------------------------------------
    def victim_order(self, t: int) -> np.ndarray:
        """Slots that may take a missing id at step t, in reservation order."""
        usable = np.arange(self.B) < self.budget
        cand = np.nonzero(((self.tag == EMPTY) | (self.last < t)) & usable)[0]
        bucket = np.where(self.tag[cand] == EMPTY, EMPTY_BUCKET,
                          np.minimum(MAX_AGE_BUCKET, t - self.last[cand]))
        # primary key: bucket, highest first; secondary: slot index, lowest first
        return cand[np.lexsort((cand, -bucket))]

    def step(self, t: int, selections) -> StepResult:
        """One decode step, or one multi-token-prediction iteration when
        ``selections`` holds one id list per query token (shared reservation
        over their union).  On error nothing changes."""
        sels = [np.asarray(s, dtype=np.int64).reshape(-1) for s in selections]
        union = self._validate(t, sels)              # ascending, distinct

        # match: which selected ids are resident
        resident = self.slot_of[union] != EMPTY
        hit_ids = union[resident]
        miss_ids = union[~resident]                  # ascending id order

        # hits count as accessed now; they are therefore never victims below
        self.last[self.slot_of[hit_ids]] = t

        # reserve victims and load the missing rows
        order = self.victim_order(t)
        for i, s in enumerate(miss_ids):
            v = order[i]
            if self.tag[v] != EMPTY:
                self.slot_of[self.tag[v]] = EMPTY    # evict
            self.tag[v] = s
            self.last[v] = t
            self.slot_of[s] = v
            self.k_rows[v] = self.host_k[s]
            if self.v_rows is not None:
                self.v_rows[v] = self.host_v[s]

        slot_maps = [self.slot_of[s].copy() for s in sels]
        hit_flags = [np.isin(s, hit_ids) for s in sels]
        self.prev_t = t
        return StepResult(slot_maps, hit_flags, int(hit_ids.size), int(miss_ids.size))


def sparse_attention(q: np.ndarray, k_rows: np.ndarray, v_rows: np.ndarray,
                     scale: float) -> np.ndarray:
    """softmax(scale * q K^T) V in fp64.

    q: [G][D] (any float); k_rows: [n][D] and v_rows: [n][Dv] bf16 bits.
    Returns [G][Dv] float64; an empty row set gives zeros."""
    qd = np.asarray(q, dtype=np.float64)
    if k_rows.shape[0] == 0:
        return np.zeros((qd.shape[0], v_rows.shape[1]), dtype=np.float64)
    K = widen_bf16(k_rows)
    V = widen_bf16(v_rows)
    s = scale * (qd @ K.T)                           # [G][n]
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    return (p @ V) / p.sum(axis=1, keepdims=True)


def attention_from_host(q: np.ndarray, host_k: np.ndarray, host_v: np.ndarray | None,
                        sel: np.ndarray, scale: float, head_dim: int, v_dim: int) -> np.ndarray:
    """Attention of one query token over the rows of the selected entries, read
    straight from this unit's host KV.  An entry of T tokens contributes its T
    rows; with host_v None, V is the K row (latent cache)."""
    sel = np.asarray(sel, dtype=np.int64).reshape(-1)
    k_rows = host_k[sel].reshape(-1, head_dim)
    v_src = host_k if host_v is None else host_v
    v_rows = v_src[sel].reshape(-1, v_dim)
    return sparse_attention(q, k_rows, v_rows, scale)


def attention_through_buffer(q: np.ndarray, unit: UnitBuffer, slot_map: np.ndarray,
                             scale: float, head_dim: int, v_dim: int) -> np.ndarray:
    """The same attention, read through the buffer slots the step assigned."""
    slot_map = np.asarray(slot_map, dtype=np.int64).reshape(-1)
    k_rows = unit.k_rows[slot_map].reshape(-1, head_dim)
    v_src = unit.k_rows if unit.v_rows is None else unit.v_rows
    v_rows = v_src[slot_map].reshape(-1, v_dim)
    return sparse_attention(q, k_rows, v_rows, scale)


class OracleRun:
    """Runs a set of units through successive steps (units are independent).

    host_k / host_v: uint16 [units][num_entries][row_elems] (host_v may be None).
    ``units`` restricts the run to a subset of unit indices.
    """

    def __init__(self, num_slots: int, host_k: np.ndarray, host_v: np.ndarray | None,
                 head_dim: int, v_dim: int, scale: float, units=None, live: int | None = None):
        self.units = list(range(host_k.shape[0])) if units is None else list(units)
        self.state = {u: UnitBuffer(num_slots, host_k[u], None if host_v is None else host_v[u],
                                    live)
                      for u in self.units}
        self.host_k, self.host_v = host_k, host_v
        self.head_dim, self.v_dim, self.scale = head_dim, v_dim, scale
        self.hits = 0
        self.misses = 0

    def set_budget(self, budgets) -> None:
        """budgets: usable slots per unit (indexed like the host store)."""
        for u in self.units:
            self.state[u].set_budget(budgets[u])

    def append(self, k_rows: np.ndarray, v_rows: np.ndarray | None = None):
        """One new entry per unit: k_rows / v_rows [units of the host store][row]."""
        for u in self.units:
            self.state[u].append(k_rows[u], None if v_rows is None else v_rows[u])

    def step(self, t: int, sel_t: np.ndarray, q_t: np.ndarray | None = None,
             attention: bool = True):
        """sel_t: [units][tokens][k]; q_t: [units][tokens][G][D].
        Returns {unit: (StepResult, out [tokens][G][Dv] or None)}."""
        res = {}
        for u in self.units:
            st = self.state[u]
            r = st.step(t, list(sel_t[u]))
            self.hits += r.hits
            self.misses += r.misses
            out = None
            if attention and q_t is not None:
                out = np.stack([attention_from_host(q_t[u][j], st.host_k, st.host_v, sel_t[u][j],
                                                    self.scale, self.head_dim, self.v_dim)
                                for j in range(sel_t.shape[1])])
            res[u] = (r, out)
        return res
