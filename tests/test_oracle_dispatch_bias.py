"""Pins for the oracle's dispatch (counting sort by expert) and bias update."""
import numpy as np
import pytest

from fine_grained_fp8_bias_b300 import workloads as wl


def random_topk(T, K, E, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,K,E", [(1, 1, 1), (7, 3, 5), (300, 8, 32), (64, 2, 256)])
def test_dispatch_is_a_stable_sort_by_expert(orc, T, K, E):
    idx = random_topk(T, K, E, T)
    r = orc.dispatch(idx, E)
    flat = idx.ravel()
    order = np.argsort(flat, kind="stable")          # library stable sort
    assert np.array_equal(r["perm_token"], (order // K).astype(np.int32))
    assert np.array_equal(r["counts"], np.bincount(flat, minlength=E))
    assert np.array_equal(r["offsets"], np.concatenate([[0], np.cumsum(r["counts"])]))
    inv = np.empty(T * K, np.int64)
    inv[order] = np.arange(T * K)
    assert np.array_equal(r["inv_row"].ravel(), inv)
    # every token appears K times, in distinct experts, rows ascending by token
    assert np.array_equal(np.bincount(r["perm_token"], minlength=T), np.full(T, K))
    for e in range(E):
        rows = r["perm_token"][r["offsets"][e]:r["offsets"][e + 1]]
        assert np.all(np.diff(rows) > 0)


def test_dispatch_rejects_bad_index(orc):
    with pytest.raises(ValueError):
        orc.dispatch(np.array([[0, 5]], np.int32), 5)


def test_empty_experts(orc):
    idx = np.array([[3, 1], [1, 3], [3, 0]], np.int32)
    r = orc.dispatch(idx, 6)
    assert r["counts"].tolist() == [1, 2, 0, 3, 0, 0]
    assert r["offsets"].tolist() == [0, 1, 3, 3, 6, 6, 6]
    assert r["perm_token"].tolist() == [2, 0, 1, 0, 1, 2]
    assert r["inv_row"].tolist() == [[3, 1], [2, 4], [5, 0]]


def test_bias_update_sign_rule(orc):
    g = np.float32(0.001)
    b = np.array([0.5, -0.25, 0.0, 0.125], np.float32)
    # T=3, K=2 -> n = 6 over E = 4 (mean 1.5, not an integer)
    out = orc.update_bias(np.array([3, 1, 2, 0], np.int32), b, 3, 2, 0.001)
    assert out.tolist() == [b[0] - g, b[1] + g, b[2] - g, b[3] + g]
    # T=2, K=2 -> n = 4, mean 1: equal load leaves the bias alone
    out = orc.update_bias(np.array([1, 1, 2, 0], np.int32), b, 2, 2, 0.001)
    assert out.tolist() == [b[0], b[1], b[2] - g, b[3] + g]


def test_bias_update_moves_by_exactly_gamma(orc):
    E = 64
    b = wl.uniform(wl.stream_key(5, 5), (E,), -0.05, 0.05).numpy()
    counts = np.random.default_rng(1).integers(0, 40, E).astype(np.int32)
    T, K = 100, 6
    out = orc.update_bias(counts, b, T, K, 0.001)
    over, under = counts * E > T * K, counts * E < T * K
    assert np.array_equal(out[over], (b[over] - np.float32(0.001)).astype(np.float32))
    assert np.array_equal(out[under], (b[under] + np.float32(0.001)).astype(np.float32))
    assert np.array_equal(out[~over & ~under], b[~over & ~under])
