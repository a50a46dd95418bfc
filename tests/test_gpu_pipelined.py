"""Two micro-batches in flight (moe_forward_pipelined): batch k's routing,
dispatch and quantisation, and batch k-1's combine, run on a side stream
while the other batch's expert GEMMs run; the bias steps after every batch.
The results must be bit-identical to moe_forward + moe_update_bias batch
after batch, for any number of SMs left to the side stream, and the layer
output agrees with the oracle."""
import numpy as np
import pytest
import torch

from fine_grained_fp8_bias_b300 import workloads as wl
from tests.helpers import (MAX_ABS, REL_FRO, bits, layer_forward_threaded, oracle_weights_threaded,
                           rel_fro, route_threaded, routing_agreement)

pytestmark = pytest.mark.gpu


def sequential(cfg, batches, gamma):
    from fine_grained_fp8_bias_b300.layer import MoELayer
    L = MoELayer.from_config(cfg, "cuda")
    res = []
    for u in batches:
        out = L.forward(u)
        L.update_bias(out["counts"], cfg.T, gamma)
        res.append({k: v.clone() for k, v in out.items()})
    torch.cuda.synchronize()
    assert L.status() == 0
    return res, L.bias.clone()


@pytest.mark.parametrize("name,reserve", [("tiny", 0), ("tiny", 16), ("ragged", 8), ("mid", 24)])
def test_pipelined_matches_sequential(name, reserve):
    from fine_grained_fp8_bias_b300.layer import MoELayer
    cfg = {"tiny": wl.TINY, "mid": wl.MID.with_(T=1024),
           "ragged": wl.LayerConfig("ragged", T=301, d=640, E=24, K=3, S=2, I=384, seed=23)}[name]
    gamma = 0.01
    batches = [wl.tokens(cfg, "cuda", step=k) for k in range(5)]
    ref, bias_ref = sequential(cfg, batches, gamma)
    L = MoELayer.from_config(cfg, "cuda")
    outs = L.forward_pipelined(batches, gamma, reserve_sms=reserve)
    torch.cuda.synchronize()
    assert L.pipelined_status() == 0
    for k in range(len(batches)):
        for key in ("h", "idx", "gate", "tie", "counts"):
            assert torch.equal(outs[k][key], ref[k][key]), (k, key)
    assert torch.equal(L.bias, bias_ref)
    assert not torch.equal(L.bias, wl.bias(cfg).cuda())


def test_pipelined_v3_against_oracle(orc):
    # V3 shapes, three batches of 256 tokens with the bias stepping between them;
    # the last batch's output on sampled tokens against the oracle (routed with
    # the bias after two updates)
    from fine_grained_fp8_bias_b300.layer import MoELayer
    cfg = wl.V3_PREFILL.with_(T=256)
    gamma = cfg.gamma
    L = MoELayer.from_config(cfg, "cuda")
    batches = [wl.tokens(cfg, "cuda", step=k) for k in range(3)]
    outs = L.forward_pipelined(batches, gamma, reserve_sms=16)
    torch.cuda.synchronize()
    assert L.pipelined_status() == 0
    bias = wl.bias(cfg).numpy().copy()
    cent = wl.centroids(cfg).numpy()
    for k, u in enumerate(batches):
        ub = bits(u.cpu())
        r = route_threaded(orc, ub, cent, bias, cfg.K)
        bad = routing_agreement(outs[k]["idx"].cpu().numpy(), outs[k]["gate"].cpu().numpy(), r,
                                bias=bias)
        idx_o = r["idx"].copy()
        idx_o[bad] = outs[k]["idx"].cpu().numpy()[bad]
        counts = np.bincount(idx_o.ravel(), minlength=cfg.E).astype(np.int32)
        assert np.array_equal(counts, outs[k]["counts"].cpu().numpy())
        if k == len(batches) - 1:
            toks = [t for t in (0, 1, 100, 255) if t not in set(bad.tolist())]
            need = set(range(cfg.E, cfg.E + cfg.S)) | {int(e) for t in toks for e in r["idx"][t]}
            W = oracle_weights_threaded(orc, cfg, need)
            ref = layer_forward_threaded(orc, ub, r["idx"], r["gate"], W, cfg, toks)
            got = outs[k]["h"].cpu().numpy()[toks]
            assert rel_fro(got, ref) <= REL_FRO and float(np.abs(got - ref).max()) <= MAX_ABS
        bias = orc.update_bias(counts, bias, cfg.T, cfg.K, gamma)
    assert np.array_equal(L.bias.cpu().numpy(), bias)
