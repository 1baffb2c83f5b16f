"""Mistakes planted in a copy of the oracle, on the CPU: every plausible slip
(a flipped sort key, a dropped term, a wrong index) must make at least one
pin fail.  The copy is made from the oracle's source text, so the real module
is never touched."""
import inspect
import sys
import types

import numpy as np
import pytest

import oracle.avsg_oracle as avsg_oracle
from test_oracle_attention import bf16_bits
from test_oracle_policy import FIXTURES, check_fixture

SRC = inspect.getsource(avsg_oracle)

POLICY_MUTANTS = {
    "bucket ascending": ("np.lexsort((cand, -bucket))", "np.lexsort((cand, bucket))"),
    "slot descending": ("np.lexsort((cand, -bucket))", "np.lexsort((-cand, -bucket))"),
    "no age cap": ("np.minimum(MAX_AGE_BUCKET, t - self.last[cand])", "(t - self.last[cand])"),
    "cap off by one": ("MAX_AGE_BUCKET = 63", "MAX_AGE_BUCKET = 62"),
    "hits not refreshed": ("self.last[self.slot_of[hit_ids]] = t", "pass"),
    "loads not stamped": ("            self.last[v] = t\n", "            self.last[v] = t - 1\n"),
    "misses descending": ("miss_ids = union[~resident]", "miss_ids = union[~resident][::-1]"),
    "empties last": ("EMPTY_BUCKET = 64", "EMPTY_BUCKET = 0"),
    "eviction keeps old id": ("self.slot_of[self.tag[v]] = EMPTY    # evict", "pass"),
    "hit flag after step": ("hit_flags = [np.isin(s, hit_ids) for s in sels]",
                            "hit_flags = [np.isin(s, union) for s in sels]"),
}

ATTENTION_MUTANTS = {
    "no max shift": ("p = np.exp(s - m)", "p = np.exp(s)"),
    "no normalisation": ("return (p @ V) / p.sum(axis=1, keepdims=True)", "return p @ V"),
    "scale dropped": ("s = scale * (qd @ K.T)", "s = (qd @ K.T)"),
    "V swapped for K": ("V = widen_bf16(v_rows)", "V = widen_bf16(k_rows)"),
}


def mutant_module(old, new):
    assert SRC.count(old) >= 1, old
    name = "avsg_oracle_mutant"
    mod = types.ModuleType(name)
    sys.modules[name] = mod          # dataclasses look the module up by name
    try:
        exec(compile(SRC.replace(old, new), name, "exec"), mod.__dict__)
    finally:
        del sys.modules[name]
    return mod


def test_mutation_targets_exist():
    for old, _ in list(POLICY_MUTANTS.values()) + list(ATTENTION_MUTANTS.values()):
        assert old in SRC, old


@pytest.mark.parametrize("name", sorted(POLICY_MUTANTS))
def test_policy_mutant_is_caught(name):
    mod = mutant_module(*POLICY_MUTANTS[name])
    caught = 0
    for fx in FIXTURES:
        try:
            check_fixture(fx, mod.UnitBuffer)
        except (AssertionError, IndexError, KeyError):
            caught += 1
    assert caught > 0, f"mutant '{name}' passed every hand-worked fixture"


def _two_row(mod):
    import math
    q = np.array([[1.0, 0.0]])
    o = mod.sparse_attention(q, bf16_bits([[1.0, 0.0], [0.0, 1.0]]),
                             bf16_bits([[1.0, 2.0], [3.0, 4.0]]), 1.0)
    w = math.e / (math.e + 1.0)
    assert abs(o[0, 0] - (3.0 - 2.0 * w)) < 1e-15 and abs(o[0, 1] - (4.0 - 2.0 * w)) < 1e-15


def _large(mod):
    import math
    o = mod.sparse_attention(np.array([[1000.0]]), bf16_bits([[1.0], [0.99609375]]),
                             bf16_bits([[2.0], [0.0]]), 1.0)
    assert abs(o[0, 0] - 2.0 / (1.0 + math.exp(-1000.0 * (1.0 - 0.99609375)))) < 1e-12


def _scaled(mod):
    # scale 0.5 on the two-row case: scores (0.5, 0)
    import math
    o = mod.sparse_attention(np.array([[1.0, 0.0]]), bf16_bits([[1.0, 0.0], [0.0, 1.0]]),
                             bf16_bits([[1.0, 2.0], [3.0, 4.0]]), 0.5)
    w = 1.0 / (1.0 + math.exp(-0.5))
    assert abs(o[0, 0] - (3.0 - 2.0 * w)) < 1e-15


@pytest.mark.parametrize("name", sorted(ATTENTION_MUTANTS))
def test_attention_mutant_is_caught(name):
    mod = mutant_module(*ATTENTION_MUTANTS[name])
    caught = 0
    for check in (_two_row, _large, _scaled):
        try:
            with np.errstate(all="ignore"):
                check(mod)
        except AssertionError:
            caught += 1
    assert caught > 0, f"mutant '{name}' passed every closed-form pin"


def test_unmutated_copy_passes():
    mod = mutant_module("EMPTY = -1", "EMPTY = -1")
    for fx in FIXTURES:
        check_fixture(fx, mod.UnitBuffer)
    for check in (_two_row, _large, _scaled):
        check(mod)
