"""The grouped GEMMs' bounded waits: when a pipeline wait runs out the kernel
records MOE_ERR_TIMEOUT in the call's status word, stops, waits for its copies
and MMAs in flight, releases its tensor memory and returns, and the context
stays usable.  The failure is made on purpose without any fault: the test
switch moe_set_pipeline_stall keeps the producer from issuing loads, so the
first stage is never filled, and moe_set_pipeline_wait_limit shortens the
waits to about half a millisecond.  A normal call on the same stream right
after must be correct (bit-exact on exact-integer operands)."""
import numpy as np
import pytest
import torch

from tests.test_gpu_gemm import groups, int_operands, oracle_grouped, bf16_round

pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = -5


@pytest.fixture(scope="module")
def L():
    from fine_grained_fp8_bias_b300 import lib
    return lib


def call_down(L, qa, sa, go, qw, sw, M, small, status):
    dev = "cuda"
    out = torch.full((M, qw.shape[1]), 7.0, dtype=torch.bfloat16, device=dev)
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    fn = L.moe_grouped_gemm_fp8_small if small else L.moe_grouped_gemm_fp8
    fn(L.MOE_GEMM_DOWN, T(qa), T(sa.T), T(go), T(qw), None, T(sw), None, out=out, status=status)
    return out


@pytest.mark.parametrize("small", [False, True], ids=["large", "small"])
def test_pipeline_wait_runs_out_and_the_next_call_is_correct(L, orc, small):
    sizes = [130, 7, 0, 33]
    go, M = groups(sizes)
    qa, sa, qw, sw = int_operands(orc, M, len(sizes), 256, 512, seed=61)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    prev_limit = L.set_pipeline_wait_limit(1_000_000)       # ~0.5 ms of SM clock
    prev_stall = L.set_pipeline_stall(True)
    try:
        call_down(L, qa, sa, go, qw, sw, M, small, status)
    finally:
        L.set_pipeline_stall(prev_stall)
        L.set_pipeline_wait_limit(prev_limit)
    # the kernel returned (the synchronize inside the status check completes)
    # and reported the timeout; the check clears the word
    assert L.moe_check_device_status(status) == MOE_ERR_TIMEOUT
    assert L.moe_check_device_status(status) == 0
    # the next call on the same stream runs normally
    out = call_down(L, qa, sa, go, qw, sw, M, small, status)
    assert L.moe_check_device_status(status) == 0
    ref = oracle_grouped(orc, qa, sa, go, qw, sw)
    assert np.array_equal(out.float().cpu().numpy()[: go[-1]], bf16_round(ref))


def test_layer_forward_reports_a_timeout_then_recovers(orc):
    # the same through moe_forward: the status word of the layer's workspace
    from fine_grained_fp8_bias_b300 import lib as L
    from fine_grained_fp8_bias_b300 import workloads as wl
    from fine_grained_fp8_bias_b300.layer import MoELayer
    cfg = wl.TINY
    layer = MoELayer.from_config(cfg, "cuda")
    u = wl.tokens(cfg, "cuda")
    ref = layer.forward(u)
    h_ref = ref["h"].clone()
    assert layer.status() == 0
    prev_limit = L.set_pipeline_wait_limit(1_000_000)
    prev_stall = L.set_pipeline_stall(True)
    try:
        layer.forward(u)
    finally:
        L.set_pipeline_stall(prev_stall)
        L.set_pipeline_wait_limit(prev_limit)
    assert layer.status() == MOE_ERR_TIMEOUT
    again = layer.forward(u)
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(again["h"], h_ref)
