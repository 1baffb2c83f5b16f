"""Buffer elasticity (Spin page, section 2B) on the GPU: per-unit slot budgets
from the host planner are lowered (dropping entries) and raised again between
steps, through the C interface; slot maps, hit flags, tags, last_step, buffer
rows and outputs follow the oracle given the same budgets."""
import numpy as np
import pytest

import workload as W
from decode_serving_gb300 import avsg
from gpu_harness import ATTN_TOL, Parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,kw", [
    ("batch_small", dict(requests=2, kv_heads=2, context=4096, k=300, slots=1024)),
    ("mtp_small", dict(requests=2, kv_heads=2, context=8192, k=200, slots=1024)),
])
def test_budgets_lowered_then_raised(name, kw):
    base = W.get_workload("mtp" if name.startswith("mtp") else "batch", steps=18, **kw)
    p = Parity(base, steps=18)
    mandatory = base.tokens_per_step * base.k
    try:
        plans = {
            6: avsg.avsg_plan_budget(base.units * mandatory + 600, base.units, mandatory, base.slots,
                                     [1.0, 0.0, 3.0, 0.0]),
            12: np.full(base.units, base.slots, np.int32),
        }
        for t in range(18):
            if t in plans:
                p.sess.set_budget(plans[t])
                p.ref.set_budget(plans[t])
                p.check_state()            # the drops themselves
            p.step(t)
            if t % 3 == 2:
                p.check_state()
        assert p.sess.stats().device_error == 0
        assert p.max_err <= ATTN_TOL
    finally:
        p.close()


def test_budget_arguments_are_checked():
    w = W.get_workload("tiny", steps=2)
    p = Parity(w, steps=2)
    try:
        with pytest.raises(avsg.AvsgError):
            p.sess.set_budget(np.zeros(w.units, np.int32))
        with pytest.raises(avsg.AvsgError):
            p.sess.set_budget(np.full(w.units, w.slots + 1, np.int32))
        p.sess.set_budget(np.full(w.units, w.k - 1, np.int32))   # below this step's k
        with pytest.raises(avsg.AvsgError):
            p.step(0)
    finally:
        p.close()
