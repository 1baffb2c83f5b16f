"""The allocation-free attention entry point (avsg_attention_noalloc).

It serves callers that cannot call cudaMalloc -- code inside another
framework's memory pool or a serving process that must not allocate once it
runs.  Its split-K scratch is a fixed array inside the library.  These tests
check, through the C interface, that on two calls in a row (the second call
reuses the scratch the first one left behind) it returns the fp64 oracle's
attention over the selected host rows and what the existing entry point
(avsg_step) returns for the same selection and queries, that a call with
more (unit, token) pairs than the fixed scratch has partials for still runs
on a full grid, and that it rejects sizes beyond its limit and flags bad row
indices.

This file is collected last on purpose: a run that stops at the first failure
has already run every other test when it gets here.
"""
import numpy as np
import pytest
import torch

import oracle
import workload as W
from decode_serving_gb300 import avsg
from decode_serving_gb300.avsg import AvsgError
from gpu_harness import ATTN_TOL, make_host_kv, make_session

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _rows_on_device(pinned):
    return torch.from_numpy(pinned.array.view(np.int16)).cuda()


CASES = {
    "gqa4": W.get_workload("tiny", requests=2, kv_heads=2, q_per_kv=4, k=300, slots=1024, steps=2),
    "latent_shared": W.get_workload("latent", requests=2, context=16384, k=256, slots=512, steps=2),
    "pages": W.get_workload("pages", requests=1, kv_heads=2, context=16 * 256, k=40, slots=128,
                            steps=2),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_matches_the_step_entry_point_on_two_calls(name):
    w = CASES[name]
    sel = W.selections(w)
    q = W.queries(w)
    hk, hv = make_host_kv(w)
    sess = make_session(w, hk, hv)
    try:
        k_rows = _rows_on_device(hk)
        v_rows = None if hv is None else _rows_on_device(hv)
        shape = (w.units, w.tokens_per_step, w.q_per_kv, w.v_dim)
        for t in range(2):
            sel_d = torch.from_numpy(sel[t]).cuda()
            q_d = torch.from_numpy(q[t]).cuda()
            ref = torch.empty(shape, dtype=torch.float32, device="cuda")
            sess.step(t, sel_d, q_d, ref)
            got = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
            avsg.avsg_attention_noalloc(
                w.units, w.num_entries, w.q_per_kv, w.head_dim, w.v_dim, w.entry_tokens,
                w.kv_shared, w.tokens_per_step, w.k, k_rows.data_ptr(),
                0 if v_rows is None else v_rows.data_ptr(), sel_d.data_ptr(), q_d.data_ptr(),
                got.data_ptr(), 0.0, torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            assert torch.isfinite(got).all()
            err = (got - ref).abs().max().item()
            assert err <= ATTN_TOL, (name, t, err)
            got_h = got.cpu().numpy()
            for u in range(w.units):
                for j in range(w.tokens_per_step):
                    o = oracle.attention_from_host(q[t][u][j], hk.array[u],
                                                   None if hv is None else hv.array[u], sel[t][u][j],
                                                   w.softmax_scale, w.head_dim, w.v_dim)
                    e2 = float(np.abs(got_h[u, j] - o).max())
                    assert e2 <= ATTN_TOL, (name, t, u, j, e2)
    finally:
        sess.close()
        hk.free()
        if hv is not None:
            hv.free()


def test_many_pairs_run_on_a_full_grid():
    """2048 (unit, token) pairs: more than the fixed scratch would hold as one
    block of partials per pair.  The result matches the oracle on sampled
    units, and the call takes about as long per pair as one with 256 units
    (a grid that had collapsed to a few CTAs would take orders of magnitude
    longer)."""
    units, rows, k, G, D = 2048, 256, 64, 4, 128
    rng = np.random.default_rng(11)
    k_h = W.fill_normal(np.empty((units, rows, D), np.uint16).reshape(-1), rows * D, W.PURPOSE_K)
    v_h = W.fill_normal(np.empty((units, rows, D), np.uint16).reshape(-1), rows * D, W.PURPOSE_V)
    k_h, v_h = k_h.reshape(units, rows, D), v_h.reshape(units, rows, D)
    idx = np.stack([rng.permutation(rows)[:k] for _ in range(units)]).astype(np.int32)
    idx = idx.reshape(units, 1, k)
    q = W.fill_normal(np.empty((units, 1, G, D), np.float32).reshape(-1), G * D, W.PURPOSE_Q)
    q = q.reshape(units, 1, G, D)
    kd = torch.from_numpy(k_h.view(np.int16)).cuda()
    vd = torch.from_numpy(v_h.view(np.int16)).cuda()
    idx_d, q_d = torch.from_numpy(idx).cuda(), torch.from_numpy(q).cuda()
    out = torch.full((units, 1, G, D), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream()

    def call(n):
        avsg.avsg_attention_noalloc(n, rows, G, D, D, 1, False, 1, k, kd.data_ptr(), vd.data_ptr(),
                                    idx_d.data_ptr(), q_d.data_ptr(), out.data_ptr(), 0.0,
                                    st.cuda_stream)

    def timed(n):
        call(n)
        best = float("inf")
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            call(n)
            b.record(st)
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b))
        return best

    small, full = timed(256), timed(units)
    assert full <= 16 * small + 0.5, (full, small)
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    for u in [0, 1, 1023, 2046, 2047]:
        o = oracle.attention_from_host(q[u][0], k_h[u], v_h[u], idx[u][0], D ** -0.5, D, D)
        assert float(np.abs(got[u, 0] - o).max()) <= ATTN_TOL, u


def test_rejects_too_many_units():
    with pytest.raises(AvsgError) as e:
        avsg.avsg_attention_noalloc(5000, 16, 4, 128, 128, 1, False, 1, 4, 1 << 20, 1 << 20,
                                    1 << 20, 1 << 20, 1 << 20)
    assert e.value.code == avsg.AVSG_ERR_CAPACITY


def test_rejects_more_selected_than_rows():
    with pytest.raises(AvsgError) as e:
        avsg.avsg_attention_noalloc(4, 16, 4, 128, 128, 1, False, 1, 17, 1 << 20, 1 << 20,
                                    1 << 20, 1 << 20, 1 << 20)
    assert e.value.code == avsg.AVSG_ERR_CAPACITY


def test_bad_row_index_fills_nan():
    w = CASES["gqa4"]
    hk, hv = make_host_kv(w)
    try:
        k_rows, v_rows = _rows_on_device(hk), _rows_on_device(hv)
        idx = torch.from_numpy(W.selections(w)[0]).cuda()
        idx[1, 0, 7] = w.num_entries          # one index past the end
        q = torch.from_numpy(W.queries(w)[0]).cuda()
        out = torch.zeros((w.units, 1, w.q_per_kv, w.v_dim), dtype=torch.float32, device="cuda")
        avsg.avsg_attention_noalloc(w.units, w.num_entries, w.q_per_kv, w.head_dim, w.v_dim, 1,
                                    False, 1, w.k, k_rows.data_ptr(), v_rows.data_ptr(),
                                    idx.data_ptr(), q.data_ptr(), out.data_ptr())
        torch.cuda.synchronize()
        assert torch.isnan(out).all()
        # the next call starts clean
        idx[1, 0, 7] = 0 if 0 not in idx[1, 0].tolist() else int(
            np.setdiff1d(np.arange(w.num_entries), idx[1, 0].cpu().numpy())[0])
        avsg.avsg_attention_noalloc(w.units, w.num_entries, w.q_per_kv, w.head_dim, w.v_dim, 1,
                                    False, 1, w.k, k_rows.data_ptr(), v_rows.data_ptr(),
                                    idx.data_ptr(), q.data_ptr(), out.data_ptr())
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
    finally:
        hk.free()
        hv.free()
