"""Pins of the oracle's sparse decode attention (fp64).

Closed forms, special cases that reduce to a known value, and the invariant
that attention read through the buffer equals attention read from host KV.
"""
import math

import numpy as np
import pytest

from oracle import (UnitBuffer, attention_from_host, attention_through_buffer,
                    sparse_attention, widen_bf16)


def rand_bf16(rng, shape):
    """Finite bf16 bit patterns of N(0,1) draws (truncated fp32)."""
    f = rng.standard_normal(shape).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def bf16_bits(x):
    """Exact bf16 bit patterns of values that are representable in bf16."""
    f = np.asarray(x, dtype=np.float32)
    b = f.view(np.uint32)
    assert ((b & 0xFFFF) == 0).all(), "value not exactly representable in bf16"
    return (b >> 16).astype(np.uint16)


def test_widen_bf16_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000, 0x8000, 0x7F7F, 0x0001], np.uint16)
    want = [1.0, -2.0, 1.0078125, 0.0, -0.0, 3.3895313892515355e38, 9.183549615799121e-41]
    got = widen_bf16(bits)
    assert got.dtype == np.float64
    for g, w in zip(got, want):
        assert g == w
    assert math.copysign(1.0, got[4]) == -1.0


def test_two_row_closed_form():
    # scores (1, 0): weights e/(e+1), 1/(e+1)
    q = np.array([[1.0, 0.0]])
    k = bf16_bits([[1.0, 0.0], [0.0, 1.0]])
    v = bf16_bits([[1.0, 2.0], [3.0, 4.0]])
    o = sparse_attention(q, k, v, 1.0)
    w = math.e / (math.e + 1.0)
    assert o.shape == (1, 2)
    assert abs(o[0, 0] - (3.0 - 2.0 * w)) < 1e-15
    assert abs(o[0, 1] - (4.0 - 2.0 * w)) < 1e-15


def test_single_row_returns_v_exactly():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((4, 16))
    k = rand_bf16(rng, (1, 16))
    v = rand_bf16(rng, (1, 16))
    o = sparse_attention(q, k, v, 0.25)
    assert (o == widen_bf16(v)[0][None, :]).all()


def test_equal_keys_give_the_mean_of_v():
    rng = np.random.default_rng(1)
    k = np.repeat(bf16_bits(np.array([[0.5, -1.0, 2.0, 0.25]], np.float32)), 7, axis=0)
    v = bf16_bits(rng.integers(-8, 8, size=(7, 3)).astype(np.float32))
    o = sparse_attention(rng.standard_normal((2, 4)), k, v, 1.0)
    mean = widen_bf16(v).sum(axis=0) / 7.0
    assert np.abs(o - mean[None, :]).max() < 1e-14


def test_zero_scale_gives_the_mean_of_v():
    rng = np.random.default_rng(2)
    k = rand_bf16(rng, (5, 8))
    v = bf16_bits(np.arange(15, dtype=np.float32).reshape(5, 3))
    o = sparse_attention(rng.standard_normal((3, 8)), k, v, 0.0)
    assert np.abs(o - np.array([6.0, 7.0, 8.0])[None, :]).max() < 1e-14


def test_large_scores_do_not_overflow():
    # scores 1000 and 999: the larger row dominates with weight e/(e+1)
    q = np.array([[1000.0]])
    k = bf16_bits([[1.0], [0.99609375]])          # 1 - 2^-8
    v = bf16_bits([[2.0], [0.0]])
    o = sparse_attention(q, k, v, 1.0)
    d = 1000.0 * (1.0 - 0.99609375)
    assert abs(o[0, 0] - 2.0 / (1.0 + math.exp(-d))) < 1e-12


def test_empty_selection_gives_zeros():
    o = sparse_attention(np.ones((2, 4)), np.zeros((0, 4), np.uint16), np.zeros((0, 3), np.uint16), 1.0)
    assert o.shape == (2, 3) and (o == 0).all()


def test_selection_order_does_not_matter():
    rng = np.random.default_rng(3)
    hk = rand_bf16(rng, (40, 32))
    hv = rand_bf16(rng, (40, 32))
    q = rng.standard_normal((4, 32))
    sel = rng.choice(40, 12, replace=False)
    a = attention_from_host(q, hk, hv, sel, 0.2, 32, 32)
    b = attention_from_host(q, hk, hv, rng.permutation(sel), 0.2, 32, 32)
    assert np.abs(a - b).max() < 1e-12


def test_pages_contribute_all_their_rows():
    # an entry of T tokens is T rows: attention over 2 pages of 3 rows equals
    # attention over the 6 rows listed one by one
    rng = np.random.default_rng(4)
    D, T = 8, 3
    hk = rand_bf16(rng, (5, T * D))
    hv = rand_bf16(rng, (5, T * D))
    q = rng.standard_normal((2, D))
    a = attention_from_host(q, hk, hv, np.array([4, 1]), 0.3, D, D)
    rows_k = np.concatenate([hk[4].reshape(T, D), hk[1].reshape(T, D)])
    rows_v = np.concatenate([hv[4].reshape(T, D), hv[1].reshape(T, D)])
    b = sparse_attention(q, rows_k, rows_v, 0.3)
    assert np.abs(a - b).max() < 1e-12


def test_shared_kv_uses_k_rows_as_values():
    rng = np.random.default_rng(5)
    hk = rand_bf16(rng, (9, 6))
    q = rng.standard_normal((3, 6))
    a = attention_from_host(q, hk, None, np.array([2, 5, 7]), 0.5, 6, 6)
    b = sparse_attention(q, hk[[2, 5, 7]], hk[[2, 5, 7]], 0.5)
    assert np.abs(a - b).max() == 0.0


@pytest.mark.parametrize("shared", [False, True])
def test_attention_through_buffer_equals_host(shared):
    # The buffer only changes where rows are read from, never the result.
    rng = np.random.default_rng(6)
    L, B, D, G, k = 200, 48, 16, 4, 20
    hk = rand_bf16(rng, (L, D))
    hv = None if shared else rand_bf16(rng, (L, D))
    u = UnitBuffer(B, hk, hv)
    for t in range(25):
        sel = rng.choice(L, size=k, replace=False)
        r = u.step(t, [sel])
        q = rng.standard_normal((G, D))
        a = attention_from_host(q, hk, hv, sel, 0.25, D, D)
        b = attention_through_buffer(q, u, r.slot_maps[0], 0.25, D, D)
        assert np.abs(a - b).max() == 0.0
