"""Offload (Spin page, section 2A, the Offload operation) on the GPU: each step
first appends one new entry per unit to the host store through the C
interface, then selects it (and the few entries appended before it) beside the
generator's ids.  Slot maps, hit flags, buffer state and outputs follow the
oracle, which receives the same new rows in its own copy of the store."""
import numpy as np
import pytest

import workload as W
from gpu_harness import ATTN_TOL, Parity

pytestmark = pytest.mark.gpu


def _bf16_bits(x):
    """fp32 -> bf16 bits, round to nearest even (test data only)."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


@pytest.mark.parametrize("name,kw", [
    ("batch_small", dict(requests=2, kv_heads=2, context=4096, k=300, slots=1024)),
    ("shared_kv", dict(requests=1, kv_heads=3, context=4096, k=200, slots=512, kv_shared=True)),
])
def test_append_then_select(name, kw):
    steps, live0, recent = 12, 4000, 4
    base = W.get_workload("batch", steps=steps, **kw)
    # the generator draws ids below live0; appended ids are live0, live0 + 1, ...
    sel = W.selections(base.replace(context=live0), steps)
    p = Parity(base, steps=steps, sel=sel, initial_entries=live0)
    rng = np.random.default_rng(2609)
    row_k = base.entry_tokens * base.head_dim
    row_v = base.entry_tokens * base.v_dim
    try:
        for t in range(steps):
            k_new = _bf16_bits(rng.standard_normal((base.units, row_k)))
            v_new = None if base.kv_shared else _bf16_bits(rng.standard_normal((base.units, row_v)))
            p.append(k_new, v_new)
            live = live0 + t + 1
            newest = np.arange(live - 1, max(live0, live - recent) - 1, -1)
            p.sel[t][:, 0, :newest.size] = newest       # replaces generator ids (all < live0)
            p.step(t)
            if t % 4 == 3:
                p.check_state()
        st = p.sess.stats()
        assert st.device_error == 0
        assert p.max_err <= ATTN_TOL
    finally:
        p.close()


def test_select_beyond_live_is_rejected():
    w = W.get_workload("tiny", steps=2)
    sel = W.selections(w.replace(context=1000), 2)
    p = Parity(w, steps=2, sel=sel, initial_entries=1000)
    try:
        bad = sel[0].copy()
        bad[0, 0, 0] = 1000                               # not appended yet
        import torch
        out = torch.empty_like(p.out)
        p.sess.step(0, torch.from_numpy(bad).cuda(), torch.from_numpy(p.q[0]).cuda(), out)
        torch.cuda.synchronize()
        assert p.sess.stats().device_error != 0
    finally:
        p.close()
