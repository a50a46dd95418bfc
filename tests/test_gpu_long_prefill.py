"""Long-prefill workload: the bias trajectory over consecutive steps, each with a
fresh token batch, is bit-identical to the oracle's.  Routing must agree on
every token the oracle does not flag as a near tie; on a flagged token where
the two selections differ, the oracle adopts the GPU's selection (both choices
are correct there), so the counts and every bias update can be compared bit
for bit.  The batch is cut to 512 tokens so that the oracle routes a step in
about a second; the GPU runs the same workload at T = 32768 in the bench."""
import numpy as np
import pytest
import torch

from fine_grained_fp8_bias_b300 import workloads as wl
from tests.helpers import bits, routing_agreement

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from fine_grained_fp8_bias_b300 import lib
    return lib


def test_bias_trajectory_matches_oracle(L, orc):
    cfg = wl.V3_LONG.with_(T=512)
    steps = 8
    cent = wl.centroids(cfg)
    cent_d = cent.cuda()
    bias_g = wl.bias(cfg).cuda()
    bias_o = wl.bias(cfg).numpy().copy()
    adopted = 0
    for step in range(steps):
        u = wl.tokens(cfg, "cpu", step)
        g = L.moe_route(u.cuda(), cent_d, bias_g, cfg.K)
        torch.cuda.synchronize()
        r = orc.route(bits(u), cent.numpy(), bias_o, cfg.K)
        gidx = g["idx"].cpu().numpy()
        bad = routing_agreement(gidx, g["gate"].cpu().numpy(), r)
        idx_o = r["idx"].copy()
        idx_o[bad] = gidx[bad]
        adopted += len(bad)
        counts_o = np.bincount(idx_o.ravel(), minlength=cfg.E).astype(np.int32)
        assert np.array_equal(counts_o, g["counts"].cpu().numpy()), step
        L.moe_update_bias(g["counts"], bias_g, cfg.T, cfg.K, cfg.gamma)
        bias_o = orc.update_bias(counts_o, bias_o, cfg.T, cfg.K, cfg.gamma)
        torch.cuda.synchronize()
        assert np.array_equal(bias_g.cpu().numpy(), bias_o), step
    # the bias moved away from its start and stayed on the grid of gamma steps
    moved = np.abs(bias_o - wl.bias(cfg).numpy())
    assert moved.max() > 0
    print(f"long prefill T=512: {steps} steps, adopted {adopted} flagged tokens, "
          f"max |b - b0| = {moved.max():.4f}")
