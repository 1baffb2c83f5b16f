"""The shared seeded input generator: shapes, determinism and the recipe's
structure (forced ids, distinctness, keep rate, Zipf skew)."""
import numpy as np
import pytest

import workload as W


def test_selection_shapes_and_validity():
    for name in ["tiny", "mtp", "pages", "latent"]:
        w = W.get_workload(name, requests=1, kv_heads=min(2, W.get_workload(name).kv_heads), steps=4)
        s = W.selections(w)
        assert s.shape == (4, w.units, w.tokens_per_step, w.k)
        assert s.min() >= 0 and s.max() < w.num_entries
        forced = set(w.forced_ids())
        for t in range(4):
            for u in range(w.units):
                for j in range(w.tokens_per_step):
                    row = s[t, u, j].tolist()
                    assert len(set(row)) == w.k
                    assert forced <= set(row)


def test_selection_is_deterministic_and_seeded():
    w = W.get_workload("tiny")
    a, b = W.selections(w), W.selections(w)
    c = W.selections(w, seed=123)
    assert (a == b).all() and not (a == c).all()


def test_keep_rate_tracks_p_keep():
    w = W.get_workload("tiny", steps=64)
    s = W.selections(w)
    forced = len(w.forced_ids())
    exp = forced / w.k + w.p_keep * (w.k - forced) / w.k
    ov = np.mean([len(set(s[t, 0, 0]) & set(s[t - 1, 0, 0])) / w.k for t in range(1, 64)])
    assert abs(ov - exp) < 0.02


def test_zipf_share_skews_to_recent_positions():
    w = W.get_workload("batch", requests=1, kv_heads=1, steps=2)
    s = W.selections(w)[0, 0, 0]
    forced = set(w.forced_ids())
    fresh = np.array([x for x in s if x not in forced])
    # 20% of fresh ids are Zipf(1.1) by rank from the end: far more than the
    # uniform share land in the last 1% of the context
    tail = (fresh >= w.num_entries * 0.99).mean()
    assert tail > 0.05


def test_mtp_chain_tokens_overlap():
    w = W.get_workload("mtp", requests=1, kv_heads=1, steps=3)
    s = W.selections(w)
    ov = len(set(s[1, 0, 1]) & set(s[1, 0, 0])) / w.k
    assert 0.8 < ov < 0.92


def test_normals():
    x = np.empty(1 << 16, np.float32)
    W.fill_normal(x, 1 << 12, purpose=9)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1.0) < 0.02
    b = np.empty(1 << 16, np.uint16)
    W.fill_normal(b, 1 << 12, purpose=9)
    # bf16 is fp32 rounded to nearest even on the upper 16 bits
    xf = x.view(np.uint32)
    rne = ((xf + 0x7FFF + ((xf >> 16) & 1)) >> 16).astype(np.uint16)
    assert (b == rne).all()
    # a slice of streams drawn alone equals the same slice of the full fill
    part = np.empty(1 << 12, np.float32)
    W.fill_normal(part, 1 << 12, purpose=9, stream_base=3)
    assert (part == x[3 << 12: 4 << 12]).all()


def test_host_kv_shapes():
    w = W.get_workload("pages", requests=1, kv_heads=2, context=16 * 64)
    k, v = W.host_kv(w)
    assert k.shape == (2, 64, 16 * 128) and v.shape == k.shape
    wl = W.get_workload("latent", requests=2, context=4096)
    k, v = W.host_kv(wl)
    assert k.shape == (2, 4096, 576) and v is None


@pytest.mark.parametrize("bad", [dict(k=5000), dict(k=-1)])
def test_generator_rejects_bad_parameters(bad):
    w = W.get_workload("tiny", **bad)
    with pytest.raises((RuntimeError, ValueError)):
        W.selections(w)


def test_unit_offset_draws_the_units_of_a_larger_job():
    """A rank holding units [2, 4) of a 4-unit job draws exactly those units'
    selections, queries and K/V rows."""
    whole = W.get_workload("tiny", requests=4, steps=5)
    part = W.get_workload("tiny", requests=2, steps=5)
    s_all, s_part = W.selections(whole), W.selections(part, unit_base=2)
    assert (s_all[:, 2:4] == s_part).all()
    q_all = W.queries(whole)
    q_part = W.queries(part, unit_base=2, units_total=4)
    assert (q_all[:, 2:4] == q_part).all()
    k_all, v_all = W.host_kv(whole)
    k_p = np.empty(W.host_kv_shape(part), np.uint16)
    v_p = np.empty_like(k_p)
    W.fill_host_kv(part, k_p, v_p, unit_base=2)
    assert (k_all[2:4] == k_p).all() and (v_all[2:4] == v_p).all()
