"""Pins of the oracle's group-limited routing (reading R14: groups of E/n_groups
contiguous experts, group score = sum of the group's group_topk best biased
scores, keep the topk_groups best groups, top-K inside them)."""
import numpy as np
import pytest
import torch

from fine_grained_fp8_bias_b300 import workloads as wl
from tests.helpers import bits


def _inputs(T, d, E, seed):
    u = wl.normal(wl.stream_key(seed, 1), (T, d), 1.0).to(torch.bfloat16)
    c = wl.normal(wl.stream_key(seed, 2), (E, d), 1.0 / np.sqrt(d)).numpy()
    b = wl.uniform(wl.stream_key(seed, 3), (E,), -0.05, 0.05).numpy()
    return bits(u), c, b


def test_one_group_or_all_groups_is_plain_routing(orc):
    u, c, b = _inputs(40, 256, 32, 1)
    plain = orc.route(u, c, b, 4)
    for n_groups, keep in ((1, 1), (4, 4), (8, 8)):
        r = orc.route_grouped(u, c, b, 4, n_groups, keep, 2)
        assert np.array_equal(r["idx"], plain["idx"])
        assert np.array_equal(r["gate"], plain["gate"])
        assert np.array_equal(r["tie"], plain["tie"])


def _brute(s, b, K, n_groups, keep, gtk):
    """The definition with library sorts instead of selection passes."""
    T, E = s.shape
    gs = E // n_groups
    z = (s + b.astype(np.float32)).astype(np.float32)
    out = np.empty((T, K), np.int64)
    for t in range(T):
        score = np.empty(n_groups, np.float32)
        for g in range(n_groups):
            top = np.sort(z[t, g * gs:(g + 1) * gs])[::-1][:gtk]
            acc = np.float32(0)
            for v in top:
                acc = np.float32(acc + v)
            score[g] = acc
        groups = np.lexsort((np.arange(n_groups), -score))[:keep]
        allowed = np.concatenate([np.arange(g * gs, (g + 1) * gs) for g in sorted(groups)])
        order = np.lexsort((allowed, -z[t, allowed]))[:K]
        out[t] = allowed[order]
    return out


@pytest.mark.parametrize("E,n_groups,keep,gtk,K", [(16, 4, 2, 2, 3), (32, 8, 4, 2, 8), (24, 3, 1, 3, 5)])
def test_against_brute_force(orc, E, n_groups, keep, gtk, K):
    u, c, b = _inputs(60, 128, E, E + n_groups)
    r = orc.route_grouped(u, c, b, K, n_groups, keep, gtk)
    want = _brute(r["scores"], b, K, n_groups, keep, gtk)
    assert np.array_equal(r["idx"], want)
    # every token's experts lie in at most `keep` groups
    assert np.all([len(set((row // (E // n_groups)).tolist())) <= keep for row in r["idx"]])
    assert np.allclose(r["gate"].sum(1), 1.0, atol=1e-6)
    assert np.array_equal(r["counts"], np.bincount(r["idx"].ravel(), minlength=E))


def test_group_restriction_changes_the_choice(orc):
    # one group holds the 4 best experts of every token (a large bias), yet only
    # keep = 2 groups of 4 are allowed, so the top-4 may not be the plain top-4
    u, c, b = _inputs(30, 128, 16, 5)
    b = np.zeros(16, np.float32)
    b[[0, 4, 8, 12]] = 10.0         # the best expert of every group (s lies in (0, 1))
    b[[1, 5]] = 9.0                 # groups 0 and 1 also hold the second best
    r = orc.route_grouped(u, c, b, 4, 4, 2, 2)
    assert np.all(np.sort(r["idx"], 1) == np.array([0, 1, 4, 5]))
    plain = orc.route(u, c, b, 4)
    assert not np.array_equal(np.sort(plain["idx"], 1), np.sort(r["idx"], 1))


def test_gates_ignore_the_bias_for_a_fixed_choice(orc):
    u, c, b = _inputs(25, 128, 32, 7)
    r1 = orc.route_grouped(u, c, b, 6, 8, 4, 2)
    r2 = orc.route_grouped(u, c, b + np.float32(0.25), 6, 8, 4, 2)   # same shift everywhere
    same = np.all(r1["idx"] == r2["idx"], axis=1)
    assert same.mean() > 0.9
    assert np.allclose(r1["gate"][same], r2["gate"][same], rtol=0, atol=0)
