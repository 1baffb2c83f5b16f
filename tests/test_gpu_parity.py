"""CUDA path vs CPU oracle, through the C interface, on the GPU.

Bit-exact: slot maps, hit flags, tags, last_step, buffer rows, hit counts.
Attention: max abs error <= 5e-3 against the fp64 oracle.
"""
import json
import os

import numpy as np
import pytest
import torch

import workload as W
from decode_serving_gb300.avsg import AvsgError
from gpu_harness import ATTN_TOL, Parity, make_host_kv, make_session

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def run_parity(w, **kw):
    p = Parity(w, **kw)
    try:
        p.run()
        st = p.sess.stats()
        assert st.device_error == 0
        if len(p.units) == w.units and not p.no_reuse:
            assert st.hits == p.ref.hits and st.misses == p.ref.misses
        return p.max_err, p.gpu_hits
    finally:
        p.close()


SMALL = {
    "tiny": W.get_workload("tiny"),
    "tiny_g4_ragged": W.get_workload("tiny", q_per_kv=4, k=300, steps=16),
    "batch_small": W.get_workload("batch", requests=2, kv_heads=2, context=4096, k=300, slots=1024,
                                  steps=24),
    "mtp_small": W.get_workload("mtp", requests=2, kv_heads=2, context=8192, k=300, slots=1024,
                                steps=12),
    "pages_small": W.get_workload("pages", requests=2, kv_heads=2, context=16 * 512, k=40, slots=128,
                                  steps=16),
    "latent_small": W.get_workload("latent", requests=2, context=65536, k=256, slots=512, steps=16),
    "latent_k_eq_b": W.get_workload("latent", requests=2, context=65536, k=256, slots=256, steps=12),
    # one CTA per (unit, token) over a ragged 20-row tile: output written without a merge
    "latent_one_tile": W.get_workload("latent", requests=2, context=4096, k=20, slots=64, steps=6,
                                      forced="none"),
    # three query tokens per step (one reservation over their union, token bits in the
    # staged gather, one cluster per (unit, token))
    "latent_mtp": W.get_workload("latent", requests=2, context=8192, k=200, slots=1024, steps=6,
                                 tokens_per_step=3),
    # two query tokens per step (the union miss pass with two sets of accumulators)
    "mtp2_small": W.get_workload("mtp", requests=2, kv_heads=2, context=8192, k=300, slots=1024,
                                 steps=10, tokens_per_step=2),
    # the union miss pass at D = 64, one query head per kv-head
    "mtp_d64_g1": W.get_workload("mtp", requests=2, kv_heads=3, context=8192, k=200, slots=1024,
                                 steps=8, head_dim=64, v_dim=64, q_per_kv=1),
    # 19 splits of 106 rows each: four tiles per CTA, the last one ragged
    "latent_multi_tile": W.get_workload("latent", requests=8, context=16384, k=2000, slots=2048,
                                        steps=4),
    "k1": W.get_workload("tiny", k=1, slots=32, steps=8, forced="none"),
    "g2": W.get_workload("tiny", q_per_kv=2, steps=8),
    "g8": W.get_workload("tiny", q_per_kv=8, steps=8),
    "d64": W.get_workload("tiny", head_dim=64, v_dim=64, q_per_kv=4, steps=8),
    "shared_d128": W.get_workload("batch", requests=1, kv_heads=3, context=4096, k=200, slots=512,
                                  steps=10, kv_shared=True),
    "odd_slots": W.get_workload("tiny", requests=3, kv_heads=1, slots=333, k=100, steps=20),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_parity(name):
    err, _ = run_parity(SMALL[name])
    assert err <= ATTN_TOL


@pytest.mark.parametrize("name", sorted(SMALL))
def test_no_reuse_path(name):
    w = SMALL[name].replace(steps=4)
    err, _ = run_parity(w, no_reuse=True)
    assert err <= ATTN_TOL


@pytest.mark.parametrize("name", ["batch_small", "mtp_small", "pages_small", "latent_small"])
def test_request_level_gather_gives_the_same_results(name):
    """Transfer assignment by request (one gather CTA per request) changes only
    which CTA copies which miss: every slot map, buffer row and output still
    follows the oracle."""
    err, _ = run_parity(SMALL[name].replace(steps=8), request_gather=True)
    assert err <= ATTN_TOL


def test_single_entry_returns_its_v_row():
    w = W.get_workload("tiny", k=1, slots=8, steps=3, forced="none")
    p = Parity(w)
    try:
        for t in range(3):
            p.step(t)
            sel = p.sel[t][0, 0, 0]
            v = p.hv.array[0, sel].astype(np.uint32) << 16
            out = p.out.cpu().numpy()[0, 0, 0]
            assert np.abs(out - v.view(np.float32)).max() <= 1e-6
    finally:
        p.close()


@pytest.mark.parametrize("name", ["worked_example_8slot.json", "age_cap_example_4slot.json",
                                  "mtp_example_6slot.json"])
def test_hand_worked_fixtures_on_gpu(name):
    with open(os.path.join(GOLDEN, name)) as f:
        fx = json.load(f)
    kmax = max(len(s) for st in fx["steps"] for s in st["sel"])
    ntok = max(len(st["sel"]) for st in fx["steps"])
    w = W.get_workload("tiny", context=fx["entries"], slots=fx["slots"], k=kmax,
                       tokens_per_step=ntok)
    hk, hv = make_host_kv(w)
    s = make_session(w, hk, hv)
    try:
        for st in fx["steps"]:
            nt, k = len(st["sel"]), len(st["sel"][0])
            sel = torch.tensor([st["sel"]], dtype=torch.int32, device="cuda")
            q = torch.zeros((1, nt, 1, w.head_dim), dtype=torch.float32, device="cuda")
            out = torch.empty((1, nt, 1, w.v_dim), dtype=torch.float32, device="cuda")
            sm = torch.empty((1, nt, k), dtype=torch.int32, device="cuda")
            hit = torch.empty((1, nt, k), dtype=torch.uint8, device="cuda")
            s.step(st["t"], sel, q, out, sm, hit)
            torch.cuda.synchronize()
            assert sm.cpu().numpy()[0].tolist() == st["slot_map"], st["t"]
            assert hit.cpu().numpy()[0].tolist() == st["hit"], st["t"]
            tag, last, kr, vr = s.read_state(0)
            assert tag.tolist() == st["tag"] and last.tolist() == st["last"], st["t"]
            for v, tg in enumerate(st["tag"]):
                if tg >= 0:
                    assert (kr[v] == hk.array[0, tg]).all() and (vr[v] == hv.array[0, tg]).all()
        stats = s.stats()
        assert stats.hits == sum(st["hits"] for st in fx["steps"])
        assert stats.misses == sum(st["misses"] for st in fx["steps"])
    finally:
        s.close()
        hk.free()
        hv.free()


SERIAL_SCRIPT = """
import sys
sys.path.insert(0, {tests!r})
import workload as W
from gpu_harness import ATTN_TOL, Parity
for w in ({cases}):
    p = Parity(w)
    try:
        p.run()
        st = p.sess.stats()
        assert st.device_error == 0
        assert st.hits == p.ref.hits and st.misses == p.ref.misses
        assert p.max_err <= ATTN_TOL, p.max_err
    finally:
        p.close()
print("serial ok")
"""


def test_serial_pipeline_gives_the_same_results():
    """With the overlapped pipeline switched off (AVSG_OVERLAP=0, read once per
    process, so in a child process) every kernel runs on one stream: match,
    reservation, gather into the slots, hash update, attention over the slot
    map.  Same oracle, same results."""
    import subprocess
    import sys
    cases = ", ".join([
        'W.get_workload("latent", requests=2, context=65536, k=256, slots=512, steps=8)',
        'W.get_workload("batch", requests=2, kv_heads=2, context=4096, k=300, slots=1024, steps=8)',
    ])
    here = os.path.dirname(os.path.abspath(__file__))
    code = SERIAL_SCRIPT.format(tests=here, cases=cases + ",")
    env = dict(os.environ, AVSG_OVERLAP="0")
    r = subprocess.run([sys.executable, "-c", code], cwd=os.path.dirname(here), env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "serial ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
