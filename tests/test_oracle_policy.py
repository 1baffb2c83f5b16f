"""Pins of the oracle's reuse state machine (match, reservation, residency).

Each pin comes from outside the oracle: hand-derived fixtures under
tests/golden/, brute force on tiny inputs written in a different form (scans
and repeated selection instead of tables and sorts), invariants, and special
cases whose result is known without running the policy.
"""
import json
import os

import numpy as np
import pytest

from oracle import EMPTY, OracleError, UnitBuffer

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FIXTURES = ["worked_example_8slot.json", "age_cap_example_4slot.json",
            "mtp_example_6slot.json"]


def _host_rows(entries, width=4, seed=0):
    rng = np.random.default_rng(seed)
    return rng.integers(0, 1 << 16, size=(entries, width), dtype=np.uint16)


def check_fixture(name, unit_cls=UnitBuffer):
    with open(os.path.join(GOLDEN, name)) as f:
        fx = json.load(f)
    hk = _host_rows(fx["entries"])
    hv = _host_rows(fx["entries"], seed=1)
    u = unit_cls(fx["slots"], hk, hv)
    total_hits = 0
    for st in fx["steps"]:
        r = u.step(st["t"], [np.array(s) for s in st["sel"]])
        assert [m.tolist() for m in r.slot_maps] == st["slot_map"], (name, st["t"])
        assert [h.astype(int).tolist() for h in r.hit_flags] == st["hit"], (name, st["t"])
        assert r.hits == st["hits"] and r.misses == st["misses"], (name, st["t"])
        assert u.tag.tolist() == st["tag"], (name, st["t"])
        assert u.last.tolist() == st["last"], (name, st["t"])
        total_hits += r.hits
    return total_hits


@pytest.mark.parametrize("name", FIXTURES)
def test_hand_worked_fixtures(name):
    check_fixture(name)


def test_worked_example_hit_rate():
    # 5 hits over 16 selected ids in the 8-slot example
    assert check_fixture("worked_example_8slot.json") == 5


# --------------------------------------------------------------------------
# Brute force on tiny inputs.

def brute_match(tag, sel):
    """Naive scan of the tag table: (hit, slot) per selected id."""
    out = []
    for s in sel:
        slot = -1
        for j, tg in enumerate(tag):
            if tg == s:
                slot = j
        out.append((slot >= 0, slot))
    return out


def merge_match(tag, sel):
    """Sorted two-pointer merge of (selected ids) against (resident ids)."""
    res = sorted((tg, j) for j, tg in enumerate(tag) if tg != EMPTY)
    order = sorted(range(len(sel)), key=lambda i: sel[i])
    out = [None] * len(sel)
    a = 0
    for i in order:
        while a < len(res) and res[a][0] < sel[i]:
            a += 1
        if a < len(res) and res[a][0] == sel[i]:
            out[i] = (True, res[a][1])
        else:
            out[i] = (False, -1)
    return out


def brute_step(tag, last, t, sels):
    """The reservation by repeated selection: each missing id, smallest first,
    takes the best remaining slot (empty beats occupied; older bucket beats
    newer; lower index breaks ties)."""
    tag, last = list(tag), list(last)
    union = sorted(set(x for s in sels for x in s))
    where = {tg: j for j, tg in enumerate(tag) if tg != EMPTY}
    for s in union:
        if s in where:
            last[where[s]] = t
    taken = set()
    for s in union:
        if s in where:
            continue
        best, best_key = None, None
        for j in range(len(tag)):
            if j in taken or (tag[j] != EMPTY and last[j] == t):
                continue
            key = (1, 0) if tag[j] == EMPTY else (0, min(63, t - last[j]))
            if best is None or key > best_key:
                best, best_key = j, key
        taken.add(best)
        if tag[best] != EMPTY:
            del where[tag[best]]
        tag[best], last[best] = s, t
        where[s] = best
    return tag, last, [[where[x] for x in s] for s in sels]


@pytest.mark.parametrize("seed", range(60))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(1000 + seed)
    L = int(rng.integers(4, 65))
    B = int(rng.integers(1, 17))
    ntok = int(rng.integers(1, 4))
    u = UnitBuffer(B, _host_rows(L), _host_rows(L, seed=2))
    t = -1
    for _ in range(40):
        t += int(rng.integers(1, 90))
        sels = []
        for _ in range(ntok):
            k = int(rng.integers(0, min(8, B // ntok, L) + 1))
            sels.append(rng.choice(L, size=k, replace=False))
        tag0, last0 = u.tag.tolist(), u.last.tolist()
        r = u.step(t, sels)
        for s, sm, hf in zip(sels, r.slot_maps, r.hit_flags):
            bm = brute_match(tag0, s.tolist())
            mm = merge_match(tag0, s.tolist())
            assert bm == mm
            for (h, slot), got_h, got_slot in zip(bm, hf, sm):
                assert bool(got_h) == h
                if h:
                    assert got_slot == slot
        btag, blast, bmaps = brute_step(tag0, last0, t, [s.tolist() for s in sels])
        assert u.tag.tolist() == btag
        assert u.last.tolist() == blast
        assert [m.tolist() for m in r.slot_maps] == bmaps


# --------------------------------------------------------------------------
# Invariants on random, moderate sizes.

@pytest.mark.parametrize("seed", range(6))
def test_invariants(seed):
    rng = np.random.default_rng(seed)
    L, B, k, ntok = 600, 96, 30, int(rng.integers(1, 4))
    hk, hv = _host_rows(L, 8, seed), _host_rows(L, 8, seed + 50)
    u = UnitBuffer(B, hk, hv)
    prev = None
    for t in range(50):
        sels = []
        for _ in range(ntok):
            if prev is not None and rng.random() < 0.7:
                keep = prev[rng.random(prev.size) < 0.8][:k]
                rest = np.setdiff1d(rng.choice(L, size=3 * k, replace=False), keep)[: k - keep.size]
                s = rng.permutation(np.concatenate([keep, rest]))
            else:
                s = rng.choice(L, size=k, replace=False)
            sels.append(s)
            prev = s
        tag0, last0 = u.tag.copy(), u.last.copy()
        r = u.step(t, sels)
        union = np.unique(np.concatenate(sels))
        assert r.hits + r.misses == union.size
        live = u.tag[u.tag != EMPTY]
        assert np.unique(live).size == live.size                 # no duplicate tags
        assert np.isin(union, u.tag).all()                       # every selected id resident
        for s in union:
            assert u.last[u.slot_of[s]] == t
        for v in np.nonzero(u.tag != EMPTY)[0]:                  # rows equal host rows
            assert (u.k_rows[v] == hk[u.tag[v]]).all()
            assert (u.v_rows[v] == hv[u.tag[v]]).all()
        changed = u.tag != tag0
        assert changed.sum() == r.misses                         # one slot per miss
        untouched = ~changed & ~np.isin(u.tag, union)
        assert (u.last[untouched] == last0[untouched]).all()
        for j, s in enumerate(sels):                             # slot map points at the id
            assert (u.tag[r.slot_maps[j]] == s).all()


# --------------------------------------------------------------------------
# Special cases with a known answer.

def test_k_equal_b_fills_every_slot():
    L, B = 100, 16
    u = UnitBuffer(B, _host_rows(L), _host_rows(L))
    rng = np.random.default_rng(3)
    for t in range(20):
        s = rng.choice(L, size=B, replace=False)
        r = u.step(t, [s])
        assert sorted(u.tag.tolist()) == sorted(s.tolist())
        assert (u.last == t).all()
        assert r.hits + r.misses == B


def test_old_ages_reduce_to_slot_order():
    L, B = 64, 10
    u = UnitBuffer(B, _host_rows(L), _host_rows(L))
    u.step(0, [np.arange(10)])
    u.step(5, [np.array([2, 7])])
    # at t=1000 all ages are >= 63: reservation is ascending slot order over
    # every slot (hits of this step excluded)
    r = u.step(1000, [np.array([40, 41, 42, 3])])
    assert r.slot_maps[0].tolist() == [0, 1, 2, 3]
    assert u.tag.tolist()[:4] == [40, 41, 42, 3]


def test_buffer_larger_than_context_never_evicts():
    L, B = 50, 64
    u = UnitBuffer(B, _host_rows(L), _host_rows(L))
    rng = np.random.default_rng(9)
    seen = set()
    for t in range(30):
        s = rng.choice(L, size=12, replace=False)
        before = len(seen & set(s.tolist()))
        tag0 = u.tag.copy()
        r = u.step(t, [s])
        assert r.hits == before                 # a hit is exactly "seen before"
        seen |= set(s.tolist())
        was = tag0 != EMPTY
        assert (u.tag[was] == tag0[was]).all()  # nothing resident is ever evicted


def test_constant_selection_is_all_hits_after_first_step():
    L, B = 300, 40
    u = UnitBuffer(B, _host_rows(L), _host_rows(L))
    s = np.random.default_rng(4).choice(L, size=25, replace=False)
    r0 = u.step(0, [s])
    assert (r0.hits, r0.misses) == (0, 25)
    for t in range(1, 10):
        r = u.step(t, [np.random.default_rng(t).permutation(s)])
        assert (r.hits, r.misses) == (25, 0)


def test_empty_selection_is_a_no_op():
    u = UnitBuffer(4, _host_rows(8), _host_rows(8))
    u.step(0, [np.array([1, 2])])
    tag0, last0 = u.tag.copy(), u.last.copy()
    r = u.step(1, [np.array([], dtype=np.int64)])
    assert (r.hits, r.misses) == (0, 0)
    assert (u.tag == tag0).all() and (u.last == last0).all()


# --------------------------------------------------------------------------
# Errors leave the state unchanged.

@pytest.mark.parametrize("t,sels,kind", [
    (5, [[1, 2, 2]], "BAD_SELECTION"),
    (5, [[1, 16]], "BAD_SELECTION"),
    (5, [[-1, 3]], "BAD_SELECTION"),
    (5, [[0, 1, 2, 3, 4], [5]], "CAPACITY"),
    (2, [[1]], "BAD_STEP"),
    (3, [[1]], "BAD_STEP"),
])
def test_errors_leave_state_unchanged(t, sels, kind):
    u = UnitBuffer(5, _host_rows(16), _host_rows(16))
    u.step(3, [np.array([7, 8])])
    snap = (u.tag.copy(), u.last.copy(), u.slot_of.copy(), u.k_rows.copy())
    with pytest.raises(OracleError) as e:
        u.step(t, [np.array(s) for s in sels])
    assert e.value.kind == kind
    assert (u.tag == snap[0]).all() and (u.last == snap[1]).all()
    assert (u.slot_of == snap[2]).all() and (u.k_rows == snap[3]).all()
    # a duplicate id across different tokens of one iteration is not an error
    u.step(10, [np.array([1, 2]), np.array([2, 3])])
