"""The V3-shape workloads and the method constants agree with the values the pages print."""
import json
import os

import numpy as np

from fine_grained_fp8_bias_b300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def consts():
    with open(os.path.join(GOLDEN, "pages_constants.json")) as f:
        return {c["name"]: c["value"] for c in json.load(f)["constants"]}


def test_v3_shapes_follow_the_pages():
    c = consts()
    for cfg in (wl.V3_PREFILL, wl.V3_DECODE, wl.V3_LONG):
        assert (cfg.S, cfg.E, cfg.K, cfg.d) == (c["shared_experts"], c["routed_experts"],
                                                c["active_routed"], c["hidden_size"])
        assert cfg.gamma == c["gamma"]


def test_tile_and_block_sizes(orc):
    c = consts()
    assert c["activation_tile"] == [1, 128] and c["weight_block"] == [128, 128]
    assert c["promotion_interval_Nc"] == 128 and c["fp8_format"] == "E4M3"
    # the oracle's scale arrays have exactly one scale per tile / block of those sizes
    q, s = orc.quant_1x128(np.ones((3, 512), np.float32))
    assert s.shape == (3, 512 // c["activation_tile"][1])
    q, s = orc.quant_128x128(np.ones((256, 384), np.float32))
    assert s.shape == (256 // c["weight_block"][0], 384 // c["weight_block"][1])


def test_generator_is_deterministic_and_has_the_requested_moments():
    a = wl.normal(wl.stream_key(3, 1, 2), (512, 512), 0.125)
    b = wl.normal(wl.stream_key(3, 1, 2), (512, 512), 0.125)
    c = wl.normal(wl.stream_key(3, 1, 3), (512, 512), 0.125)
    assert np.array_equal(a.numpy(), b.numpy()) and not np.array_equal(a.numpy(), c.numpy())
    assert abs(a.mean().item()) < 2e-3 and abs(a.std().item() / 0.125 - 1) < 5e-3
    # a slice of a longer draw equals the draw that starts at its offset
    full = wl.normal(wl.stream_key(3, 9), (1000,), 1.0)
    part = wl.normal(wl.stream_key(3, 9), (300,), 1.0, start=500)
    assert np.array_equal(full[500:800].numpy(), part.numpy())
    u = wl.uniform(wl.stream_key(3, 4), (100000,), -0.05, 0.05)
    assert u.min() >= -0.05 and u.max() < 0.05


def test_decode_skew_is_the_calibrated_one():
    # the workload's hot-expert shift is the one the calibration script found
    import json
    import os
    from fine_grained_fp8_bias_b300 import workloads as wl
    rec = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "decode_skew.json")))
    assert wl.V3_DECODE.hot_alpha == rec["hot_alpha"]
    assert abs(rec["hot_fraction_T256"] - rec["target"]) <= rec["tolerance"]
