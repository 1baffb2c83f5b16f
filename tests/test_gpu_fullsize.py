"""The five workloads at full size, in the launch configuration the bench uses.

The oracle follows every unit through every step: slot maps and hit flags
of every unit and step, tags and last_step of every unit every 32 steps, all
buffer rows of every unit after the last step, and the device's hit and miss
totals are compared bit for bit.  The attention output is compared (<= 5e-3
against fp64) on a sample of units at every step: the fp64 attention is the
oracle's costly part, and the buffer state it would read is already checked
whole."""
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


def run_full(w, attn_units):
    p = Parity(w, attn_units=attn_units)
    try:
        p.run(state_every=32, rows_every=False)
        st = p.sess.stats()
        assert st.device_error == 0
        assert p.max_err <= ATTN_TOL
        # every unit's distinct hits and misses, summed over all steps
        assert st.hits == p.ref.hits, (st.hits, p.ref.hits)
        assert st.misses == p.ref.misses, (st.misses, p.ref.misses)
        assert st.hits + st.misses == st.unique_selected
        return st
    finally:
        p.close()


def test_batch_full():
    run_full(W.get_workload("batch"), attn_units=[0, 29, 63])


def test_mtp_full():
    run_full(W.get_workload("mtp"), attn_units=[0, 77, 127])


def test_pages_full():
    run_full(W.get_workload("pages"), attn_units=[0, 101, 255])


def test_tiny_full():
    run_full(W.get_workload("tiny"), attn_units=None)


@pytest.mark.parametrize("slots", W.configs.LATENT_SLOT_SWEEP)
def test_latent_full(slots):
    run_full(W.get_workload("latent", slots=slots), attn_units=None)
