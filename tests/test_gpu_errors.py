"""Error behaviour of the CUDA path: host-side rejections, device-detected bad
selections latched before any state change, recovery, and edge inputs."""
import numpy as np
import pytest
import torch

import workload as W
from decode_serving_gb300 import avsg
from decode_serving_gb300.avsg import AvsgError
from gpu_harness import ATTN_TOL, Parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


W_ERR = W.get_workload("tiny", requests=2, kv_heads=2, q_per_kv=4, k=64, slots=256, steps=6)
# the 16-head pipeline (staged gather, clustered attention; k = 300 takes several clusters
# per pair, so the last-arriver merge and its counters are in play)
W_ERR_LATENT = W.get_workload("latent", requests=2, context=8192, k=300, slots=512, steps=6)


def _snapshot(p):
    return [p.sess.read_state(u) for u in range(p.w.units)]


def _same(a, b):
    for (t1, l1, k1, v1), (t2, l2, k2, v2) in zip(a, b):
        assert (t1 == t2).all() and (l1 == l2).all() and (k1 == k2).all()
        assert (v1 is None and v2 is None) or (v1 == v2).all()  # None: V is the K row


@pytest.mark.parametrize("shape", ["gqa4", "latent"])
@pytest.mark.parametrize("bad", ["duplicate", "out_of_range", "negative", "duplicate_hit"])
def test_bad_selection_is_latched_before_any_change(bad, shape):
    w = W_ERR if shape == "gqa4" else W_ERR_LATENT
    p = Parity(w)
    try:
        p.step(0)
        before = _snapshot(p)
        sel = p.sel[1].copy()
        if bad == "duplicate":
            sel[1, 0, 5] = sel[1, 0, 9]
        elif bad == "out_of_range":
            sel[1, 0, 3] = w.num_entries
        elif bad == "negative":
            sel[1, 0, 3] = -7
        else:  # repeat an id that is resident (a hit) within one token
            sel[1, 0, 5] = p.sel[0][1, 0, 0]
            sel[1, 0, 6] = p.sel[0][1, 0, 0]
        sel_d = torch.from_numpy(sel).cuda()
        q_d = torch.from_numpy(p.q[1]).cuda()
        p.sess.step(1, sel_d, q_d, p.out, p.sm, p.hit)
        st = p.sess.stats()
        assert st.device_error == avsg.AVSG_ERR_BAD_SELECTION
        assert st.error_unit == 1
        _same(before, _snapshot(p))
        with pytest.raises(AvsgError) as e:
            p.sess.step(2, sel_d, q_d, p.out, p.sm, p.hit)
        assert e.value.code == avsg.AVSG_ERR_LATCHED
        p.sess.clear_error()
        # the oracle never saw step 1; both continue from the same state
        for t in range(2, 5):
            p.step(t)
        p.check_state()
    finally:
        p.close()


def test_host_side_rejections():
    p = Parity(W_ERR)
    try:
        p.step(3, ti=0)
        sel_d = torch.from_numpy(p.sel[1]).cuda()
        q_d = torch.from_numpy(p.q[1]).cuda()
        for t in (3, 2, -1):
            with pytest.raises(AvsgError) as e:
                p.sess.step(t, sel_d, q_d, p.out, p.sm, p.hit)
            assert e.value.code == avsg.AVSG_ERR_BAD_STEP
        big = torch.zeros((W_ERR.units, 1, W_ERR.k + 1), dtype=torch.int32, device="cuda")
        with pytest.raises(AvsgError) as e:
            p.sess.step(4, big, q_d, p.out)
        assert e.value.code == avsg.AVSG_ERR_CAPACITY
        two = torch.zeros((W_ERR.units, 2, 4), dtype=torch.int32, device="cuda")
        with pytest.raises(AvsgError) as e:
            p.sess.step(4, two, q_d, p.out)
        assert e.value.code == avsg.AVSG_ERR_INVALID_ARG
        p.step(4, ti=1)  # nothing changed: the pair continues in lockstep
        p.check_state()
    finally:
        p.close()


@pytest.mark.parametrize("shape", ["gqa4", "latent"])
def test_empty_selection_gives_zeros_and_keeps_state(shape):
    w = W_ERR if shape == "gqa4" else W_ERR_LATENT
    p = Parity(w)
    try:
        p.step(0)
        before = _snapshot(p)
        empty = torch.zeros((w.units, 1, 0), dtype=torch.int32, device="cuda")
        q_d = torch.from_numpy(p.q[1]).cuda()
        p.out.fill_(float("nan"))
        p.sess.step(1, empty, q_d, p.out)
        torch.cuda.synchronize()
        assert (p.out == 0).all()
        _same(before, _snapshot(p))
        p.ref.step(1, np.zeros((w.units, 1, 0), np.int32))
        p.step(2)
        p.check_state()
    finally:
        p.close()


def test_step_host_matches_device_step():
    w = W.get_workload("tiny", requests=2, kv_heads=2, q_per_kv=4, k=128, slots=512, steps=5)
    p = Parity(w)
    try:
        for t in range(w.steps):
            sel, q = p.sel[t], p.q[t]
            out = np.empty((w.units, 1, w.q_per_kv, w.v_dim), np.float32)
            sm = np.empty(sel.shape, np.int32)
            hit = np.empty(sel.shape, np.uint8)
            p.sess.step_host(t, sel, q, out, sm, hit)
            torch.cuda.synchronize()
            res = p.ref.step(t, sel, q)
            for u, (r, o) in res.items():
                assert (sm[u, 0] == r.slot_maps[0]).all()
                assert (hit[u, 0] == r.hit_flags[0]).all()
                assert np.abs(out[u] - o).max() <= ATTN_TOL
        p.check_state()
    finally:
        p.close()


def test_reset_empties_the_buffer():
    p = Parity(W_ERR)
    try:
        p.step(0)
        p.sess.reset()
        torch.cuda.synchronize()
        tag, last, _, _ = p.sess.read_state(0)
        assert (tag == -1).all() and (last == -1).all()
        assert p.sess.stats().hits == 0
    finally:
        p.close()
