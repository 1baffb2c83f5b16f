"""Pins of the oracle's offload (Spin page, section 2A, the Offload operation):
a decode step's new KV entry is written to the host store and becomes
selectable from the next step on, entering the buffer only as a miss.

Each pin fixes a fact that follows from that reading and plain arithmetic:
ids at or above the live count are rejected, an appended entry is a miss whose
row arrives in the reserved slot, a single selected row's attention is its V
row exactly, appending never touches the buffer, and the store refuses an
entry past its capacity.  The mutants at the end plant the slips one would make
writing ``append`` (not raising the count, writing the wrong row) and check
that a pin catches each."""
import numpy as np
import pytest

import oracle.avsg_oracle as O
from test_oracle_mutants import mutant_module


def _unit(mod=O, B=4, cap=8, live=4, width=2):
    hk = np.zeros((cap, width), np.uint16)
    hv = np.zeros((cap, width), np.uint16)
    for i in range(cap):             # distinct, recognisable bf16 rows (1.0 + i/128)
        hk[i] = 0x3F80 + i
        hv[i] = 0x4000 + i
    return mod.UnitBuffer(B, hk, hv, live=live)


def _new_rows(width=2):
    return np.full(width, 0x4120, np.uint16), np.full(width, 0x4140, np.uint16)  # 10.0, 12.0


def check_range(mod=O):
    u = _unit(mod)
    with pytest.raises(mod.OracleError):
        u.step(0, [np.array([4])])           # id 4 is not live yet
    u2 = _unit(mod)
    assert u2.append(*_new_rows()) == 4
    r = u2.step(0, [np.array([4])])          # now it is
    assert r.misses == 1 and r.hits == 0


def check_row_arrives(mod=O):
    u = _unit(mod)
    k_new, v_new = _new_rows()
    u.append(k_new, v_new)
    u.step(0, [np.array([1, 4])])
    slot = int(np.nonzero(u.tag == 4)[0][0])
    assert np.array_equal(u.k_rows[slot], k_new) and np.array_equal(u.v_rows[slot], v_new)


def check_attention_of_new_row(mod=O):
    u = _unit(mod)
    k_new, v_new = _new_rows()
    u.append(k_new, v_new)
    q = np.array([[0.5, -0.25]])
    out = mod.attention_from_host(q, u.host_k, u.host_v, np.array([4]), 1.0, 2, 2)
    assert np.array_equal(out, np.array([[12.0, 12.0]]))   # one row: softmax weight 1


def check_buffer_untouched(mod=O):
    u = _unit(mod)
    u.step(0, [np.array([0, 2])])
    tag, last, k_rows = u.tag.copy(), u.last.copy(), u.k_rows.copy()
    u.append(*_new_rows())
    assert np.array_equal(u.tag, tag) and np.array_equal(u.last, last)
    assert np.array_equal(u.k_rows, k_rows)


def check_capacity(mod=O):
    u = _unit(mod, cap=6, live=4)
    u.append(*_new_rows())
    u.append(*_new_rows())
    with pytest.raises(mod.OracleError):
        u.append(*_new_rows())


PINS = [check_range, check_row_arrives, check_attention_of_new_row, check_buffer_untouched,
        check_capacity]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_append_pins(pin):
    pin()


def test_run_level_append_matches_unit_level():
    cap, U = 8, 2
    hk = np.arange(U * cap * 2, dtype=np.uint16).reshape(U, cap, 2) + 0x3F80
    hv = hk + 0x100
    run = O.OracleRun(4, hk.copy(), hv.copy(), 2, 2, 1.0, live=5)
    new_k = np.full((U, 2), 0x4120, np.uint16)
    new_v = np.full((U, 2), 0x4140, np.uint16)
    run.append(new_k, new_v)
    sel = np.array([[[5]], [[5]]])
    res = run.step(0, sel, np.zeros((U, 1, 1, 2)))
    for u in range(U):
        r, out = res[u]
        assert r.misses == 1 and np.array_equal(out[0][0], [12.0, 12.0])


APPEND_MUTANTS = {
    "count not raised": ("        self.live += 1\n        return self.live - 1",
                         "        return self.live"),
    "row written one late": ("        self.host_k[self.live] = k_row", "        self.host_k[self.live - 1] = k_row"),
    "capacity not checked": ("        if self.live >= self.L:\n            raise OracleError(ERR_CAPACITY, \"host store full\")",
                             "        if False:\n            pass"),
    "range by capacity": ("s.max() >= self.live", "s.max() >= self.L"),
}


@pytest.mark.parametrize("name", sorted(APPEND_MUTANTS))
def test_append_mutant_is_caught(name):
    mod = mutant_module(*APPEND_MUTANTS[name])
    caught = 0
    for pin in PINS:
        try:
            pin(mod)
        except (Exception, pytest.fail.Exception):
            caught += 1
    assert caught > 0, f"mutant '{name}' passed every append pin"
