"""Long-prefill workload (T = 32768 tokens from a 4-component mixture, V3 shapes).

- At the full batch size: routing of every token through moe_route and through
  the layer, the layer output on tokens whose rows cover every shared-expert M
  tile and the edge tiles of routed experts, and the bias trajectory of the
  first three steps (fresh batch each step, bias updated after each).
- At T = 4096: the bias trajectory over all 100 steps of the workload.

Routing must agree on every token the oracle does not flag as a near tie; on a
flagged token where the two selections differ, the oracle adopts the GPU's
selection (both choices are correct there), so counts and every bias update
can be compared bit for bit.  The oracle's routing runs on token chunks in a
thread pool (it is token-independent)."""
import numpy as np
import pytest
import torch

from fine_grained_fp8_bias_b300 import workloads as wl
from tests.helpers import bits, route_threaded, routing_agreement

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from fine_grained_fp8_bias_b300 import lib
    return lib


def trajectory(L, orc, cfg, steps, use_layer=None):
    """Routes `steps` fresh batches, updating the bias after each, on the GPU
    and in the oracle; asserts counts and bias agree bit for bit every step."""
    cent = wl.centroids(cfg)
    cent_d = cent.cuda()
    bias_g = wl.bias(cfg).cuda()
    bias_o = wl.bias(cfg).numpy().copy()
    ws = torch.empty(L.route_workspace_bytes(cfg.T, cfg.E, cfg.d), dtype=torch.uint8, device="cuda")
    adopted, ratios = 0, []
    for step in range(steps):
        u = wl.tokens(cfg, "cpu", step)
        g = L.moe_route(u.cuda(), cent_d, bias_g, cfg.K, ws=ws)
        torch.cuda.synchronize()
        r = route_threaded(orc, bits(u), cent.numpy(), bias_o, cfg.K)
        gidx = g["idx"].cpu().numpy()
        bad = routing_agreement(gidx, g["gate"].cpu().numpy(), r, bias=bias_o)
        idx_o = r["idx"].copy()
        idx_o[bad] = gidx[bad]
        adopted += len(bad)
        counts_o = np.bincount(idx_o.ravel(), minlength=cfg.E).astype(np.int32)
        assert np.array_equal(counts_o, g["counts"].cpu().numpy()), step
        ratios.append(counts_o.max() / (cfg.T * cfg.K / cfg.E))
        L.moe_update_bias(g["counts"], bias_g, cfg.T, cfg.K, cfg.gamma)
        bias_o = orc.update_bias(counts_o, bias_o, cfg.T, cfg.K, cfg.gamma)
        torch.cuda.synchronize()
        assert np.array_equal(bias_g.cpu().numpy(), bias_o), step
    moved = np.abs(bias_o - wl.bias(cfg).numpy())
    assert moved.max() > 0
    print(f"{cfg.name} T={cfg.T}: {steps} steps, adopted {adopted} flagged tokens, "
          f"max load / mean first {ratios[0]:.2f} last {ratios[-1]:.2f}, "
          f"max |b - b0| = {moved.max():.4f}")
    return ratios


def test_bias_trajectory_full_batch_three_steps(L, orc):
    trajectory(L, orc, wl.V3_LONG, 3)


def test_bias_trajectory_all_100_steps_at_4096(L, orc):
    ratios = trajectory(L, orc, wl.V3_LONG.with_(T=4096), 100)
    # the bias pulls the most loaded expert towards the mean
    assert np.mean(ratios[-10:]) < ratios[0]


def test_layer_full_batch(orc):
    # the whole layer at T = 32768: every token's routing, and the output on the
    # tokens of every shared M tile (256) plus edge rows of 32 routed experts
    from tests.test_gpu_layer import check_layer
    check_layer(orc, wl.V3_LONG, tokens="cover", cover=(32, 64))
    torch.cuda.empty_cache()
