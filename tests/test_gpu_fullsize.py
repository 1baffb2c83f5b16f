"""The five workloads at full size, in the launch configuration the bench uses.

Units are independent, so the oracle follows a sample of units over every
step (bit-exact state, hit counts, attention <= 5e-3); every unit is checked
at the end against properties that hold at any size: no repeated tag, every
id of the last step resident at the slot the slot map names, buffer rows equal
to the host rows of their tags (sampled slots)."""
import numpy as np
import pytest
import torch

import workload as W
from gpu_harness import ATTN_TOL, Parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def check_every_unit(p):
    sel_last = p.sel[p.steps - 1]
    sm = p.sm.cpu().numpy()
    rng = np.random.default_rng(7)
    for u in range(p.w.units):
        tag, last, kr, vr = p.sess.read_state(u, rows=True)
        live = tag[tag >= 0]
        assert np.unique(live).size == live.size, f"repeated tag unit={u}"
        for j in range(p.w.tokens_per_step):
            assert (tag[sm[u, j]] == sel_last[u, j]).all(), f"slot map unit={u}"
            assert (last[sm[u, j]] == p.steps - 1).all()
        slots = rng.choice(np.nonzero(tag >= 0)[0], size=min(64, live.size), replace=False)
        for v in slots:
            assert (kr[v] == p.hk.array[u, tag[v]]).all(), f"K row unit={u} slot={v}"
            if vr is not None:
                assert (vr[v] == p.hv.array[u, tag[v]]).all(), f"V row unit={u} slot={v}"


def run_full(w, units):
    p = Parity(w, units=units)
    try:
        p.run(state_every=32)
        check_every_unit(p)
        st = p.sess.stats()
        assert st.device_error == 0
        assert p.max_err <= ATTN_TOL
        return st
    finally:
        p.close()


def test_batch_full():
    w = W.get_workload("batch")
    run_full(w, units=[0, 29, 63])


def test_mtp_full():
    w = W.get_workload("mtp")
    run_full(w, units=[0, 127])


def test_pages_full():
    w = W.get_workload("pages")
    run_full(w, units=[0, 255])


@pytest.mark.parametrize("slots", W.configs.LATENT_SLOT_SWEEP)
def test_latent_full(slots):
    w = W.get_workload("latent", slots=slots)
    st = run_full(w, units=None)
    assert st.hits + st.misses == st.unique_selected
