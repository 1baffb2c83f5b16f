"""Pins of the oracle's buffer elasticity (Spin page, section 2B: the buffer of
each request is sized per step, mandatory slots plus buffer slots, under a
system-wide budget), and of the host planner in the C interface.

The hand-worked example: B = 8 slots, step 0 selects ids 10..17, which fill
slots 0..7 in ascending id order.  Lowering the budget to 5 drops ids 15, 16
and 17 (slots 5..7).  At step 1 the selection {10, 20} hits 10.  Id 20 must
take a slot below the budget.  Those are slots 1..4, all age 1 (bucket 1), so
the lowest index wins: slot 1, evicting id 11.  Without the budget the empty
slots 5..7 would come first."""
import ctypes

import numpy as np
import pytest

import oracle.avsg_oracle as O
from test_oracle_mutants import mutant_module


def _unit(mod=O, B=8, L=64):
    hk = (np.arange(L * 2, dtype=np.uint16).reshape(L, 2) + 0x3F80)
    return mod.UnitBuffer(B, hk, None)


def _filled(mod=O):
    u = _unit(mod)
    u.step(0, [np.arange(10, 18)])
    return u


def check_shrink_drops_exactly(mod=O):
    u = _filled(mod)
    u.set_budget(5)
    assert list(u.tag) == [10, 11, 12, 13, 14, -1, -1, -1]
    assert list(u.last[5:]) == [-1, -1, -1]
    assert all(u.slot_of[i] == O.EMPTY for i in (15, 16, 17))
    assert [u.slot_of[i] for i in range(10, 15)] == [0, 1, 2, 3, 4]


def check_victim_below_budget(mod=O):
    u = _filled(mod)
    u.set_budget(5)
    r = u.step(1, [np.array([10, 20])])
    assert r.hits == 1 and r.misses == 1
    assert u.tag[1] == 20 and u.slot_of[11] == O.EMPTY
    assert list(u.tag[5:]) == [-1, -1, -1]


def check_dropped_id_is_a_miss(mod=O):
    u = _filled(mod)
    u.set_budget(5)
    r = u.step(1, [np.array([15])])
    assert r.misses == 1 and r.hits == 0


def check_capacity(mod=O):
    u = _filled(mod)
    u.set_budget(2)
    with pytest.raises(mod.OracleError):
        u.step(1, [np.array([1, 2, 3])])


def check_grow_reopens_empty_slots(mod=O):
    u = _filled(mod)
    u.set_budget(5)
    u.set_budget(8)
    u.step(1, [np.array([20])])
    assert u.tag[5] == 20        # empty slots first, lowest index


PINS = [check_shrink_drops_exactly, check_victim_below_budget, check_dropped_id_is_a_miss,
        check_capacity, check_grow_reopens_empty_slots]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_budget_pins(pin):
    pin()


BUDGET_MUTANTS = {
    "victims ignore the budget": ("((self.tag == EMPTY) | (self.last < t)) & usable",
                                  "((self.tag == EMPTY) | (self.last < t))"),
    "dropped ids stay indexed": ("                self.slot_of[self.tag[slot]] = EMPTY\n", ""),
    "drop one slot too few": ("for slot in range(budget, self.B):", "for slot in range(budget + 1, self.B):"),
    "capacity by B": ("if union.size > self.budget:", "if union.size > self.B:"),
}


@pytest.mark.parametrize("name", sorted(BUDGET_MUTANTS))
def test_budget_mutant_is_caught(name):
    mod = mutant_module(*BUDGET_MUTANTS[name])
    caught = 0
    for pin in PINS:
        try:
            pin(mod)
        except (Exception, pytest.fail.Exception):
            caught += 1
    assert caught > 0, f"mutant '{name}' passed every budget pin"


# -- the planner (host code of the C interface; no GPU) ----------------------

def _plan(lib, total, units, mandatory, max_slots, weights=None):
    out = np.zeros(units, np.int32)
    w = None if weights is None else np.ascontiguousarray(weights, np.float32)
    rc = lib.avsg_plan_budget(total, units, mandatory, max_slots,
                              None if w is None else w.ctypes.data, out.ctypes.data)
    return rc, out


def test_plan_equal_split_gives_the_remainder_to_the_lowest_units(lib):
    rc, out = _plan(lib, 3 * 100 + 7, 3, 100, 1000)
    assert rc == 0 and list(out) == [103, 102, 102]      # 7 extra: 3, 2, 2


def test_plan_weighted_split(lib):
    rc, out = _plan(lib, 4 * 10 + 100, 4, 10, 1000, [1.0, 0.0, 3.0, 0.0])
    assert rc == 0 and list(out) == [35, 10, 85, 10]     # 100 extra: 25 and 75


def test_plan_caps_at_the_buffer(lib):
    rc, out = _plan(lib, 2 * 10 + 1000, 2, 10, 300)
    assert rc == 0 and list(out) == [300, 300]


def test_plan_rejects_too_small_a_total(lib):
    rc, _ = _plan(lib, 2 * 10 - 1, 2, 10, 300)
    assert rc == -2


@pytest.mark.parametrize("args", [(100, 0, 10, 300), (100, 2, 0, 300), (100, 2, 10, 5), (-1, 2, 10, 300)])
def test_plan_rejects_bad_arguments(lib, args):
    rc, _ = _plan(lib, *args)
    assert rc == -1
