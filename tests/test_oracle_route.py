"""Pins for the oracle's router: sigmoid affinity, bias-steered top-K, normalised gates."""
import itertools
import json
import os

import numpy as np
import torch

from fine_grained_fp8_bias_b300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def inputs(T, d, E, seed, bias_scale=0.05):
    u = wl.normal(wl.stream_key(seed, 1), (T, d), 1.0).to(torch.bfloat16)
    c = wl.normal(wl.stream_key(seed, 2), (E, d), 1.0 / np.sqrt(d))
    b = wl.uniform(wl.stream_key(seed, 3), (E,), -bias_scale, bias_scale)
    return u, c.numpy(), b.numpy()


def bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def test_scores_match_library_sigmoid_of_fp64_logits(orc):
    u, c, b = inputs(64, 256, 16, 1)
    r = orc.route(bits(u), c, b, 2)
    logit = (u.float().double().numpy() @ c.astype(np.float64).T).astype(np.float32)
    s_ref = torch.sigmoid(torch.from_numpy(logit).double()).float().numpy()
    ulps = np.abs(r["scores"].view(np.int32).astype(np.int64) - s_ref.view(np.int32).astype(np.int64))
    assert ulps.max() <= 1 and (ulps == 0).mean() > 0.99


def test_brute_force_topk_over_all_subsets(orc):
    for (E, K, seed) in [(16, 2, 2), (8, 3, 3), (6, 6, 4), (5, 1, 5)]:
        u, c, b = inputs(24, 128, E, seed, bias_scale=0.2)
        r = orc.route(bits(u), c, b, K)
        z = (r["scores"] + b[None, :]).astype(np.float32)
        for t in range(24):
            best = max(itertools.combinations(range(E), K),
                       key=lambda S: (sum(float(z[t, i]) for i in S), [-i for i in S]))
            assert sorted(r["idx"][t].tolist()) == sorted(best)
            # ordered by descending biased score
            zs = z[t, r["idx"][t]]
            assert np.all(zs[:-1] >= zs[1:])


def test_gates_sum_to_one_and_keep_score_ratios(orc):
    u, c, b = inputs(200, 256, 16, 6)
    r = orc.route(bits(u), c, b, 4)
    g = r["gate"].astype(np.float64)
    assert np.all(np.abs(g.sum(1) - 1.0) < 1e-6)
    s_sel = np.take_along_axis(r["scores"], r["idx"], 1).astype(np.float64)
    assert np.allclose(g[:, 1:] / g[:, :1], s_sel[:, 1:] / s_sel[:, :1], rtol=1e-6)


def test_bias_changes_selection_not_gate_values(orc):
    u, c, _ = inputs(50, 128, 16, 7)
    b0 = np.zeros(16, np.float32)
    r0 = orc.route(bits(u), c, b0, 3)
    # a tiny bias that keeps every selection leaves the gates bit-identical
    b1 = np.full(16, 0.25, np.float32)
    r1 = orc.route(bits(u), c, b1, 3)
    assert np.array_equal(r0["idx"], r1["idx"]) and np.array_equal(r0["gate"], r1["gate"])
    # a large bias forces expert 11 in, and its gate comes from s, not s + b
    b2 = b0.copy()
    b2[11] = 10.0
    r2 = orc.route(bits(u), c, b2, 3)
    assert np.all(r2["idx"][:, 0] == 11)
    s11 = r2["scores"][:, 11].astype(np.float64)
    ssum = np.take_along_axis(r2["scores"], r2["idx"], 1).astype(np.float64).sum(1)
    assert np.allclose(r2["gate"][:, 0], s11 / ssum, rtol=1e-7)
    assert np.array_equal(r2["scores"], r0["scores"])


def test_zero_bias_is_plain_topk_of_scores(orc):
    u, c, _ = inputs(300, 256, 32, 8)
    r = orc.route(bits(u), c, np.zeros(32, np.float32), 6)
    ref = torch.topk(torch.from_numpy(r["scores"]), 6, dim=1)
    assert np.array_equal(r["idx"], ref.indices.numpy().astype(np.int32))


def test_exact_ties_break_by_lower_index_and_flag(orc):
    u, c, _ = inputs(10, 128, 8, 9)
    c[5] = c[2]                             # experts 2 and 5 always score the same
    b = np.zeros(8, np.float32)
    b[2] = b[5] = 5.0                       # and both are selected first
    r = orc.route(bits(u), c, b, 1)
    assert np.all(r["idx"][:, 0] == 2)
    assert np.all(r["tie"] == 1)            # z_(1) == z_(2)
    r = orc.route(bits(u), c, b, 2)
    assert np.all(r["idx"] == np.array([2, 5]))
    assert np.all(r["gate"] == np.float32(0.5))


def test_k_equals_e_selects_everything_without_flag(orc):
    u, c, b = inputs(5, 128, 4, 10)
    r = orc.route(bits(u), c, b, 4)
    assert np.all(np.sort(r["idx"], 1) == np.arange(4))
    assert np.all(r["tie"] == 0)
    assert np.all(r["counts"] == 5)


def test_counts_are_the_histogram(orc):
    u, c, b = inputs(333, 128, 16, 11)
    r = orc.route(bits(u), c, b, 3)
    assert np.array_equal(r["counts"], np.bincount(r["idx"].ravel(), minlength=16))


def test_worked_examples(orc):
    with open(os.path.join(GOLDEN, "route_worked_examples.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        d = case["d"]
        u = np.zeros((1, d), np.float32)
        u[0, 0] = 1.0
        c = np.zeros((len(case["logit"]), d), np.float32)
        c[:, 0] = np.array(case["logit"], np.float32)
        r = orc.route(bits(torch.from_numpy(u).to(torch.bfloat16)), c,
                      np.array(case["bias"], np.float32), case["K"])
        assert r["idx"][0].tolist() == case["idx"], case["name"]
        assert np.allclose(r["gate"][0], case["gate"], atol=1e-6), case["name"]
        assert int(r["tie"][0]) == case["tie"], case["name"]
        assert r["counts"].tolist() == case["counts"], case["name"]
        b = orc.update_bias(r["counts"], np.array(case["bias"], np.float32), 1, case["K"],
                            case["gamma"])
        assert np.allclose(b, case["bias_after"], atol=1e-7), case["name"]
