"""Failure detection without a GPU fault: a bounded device-side wait that can
never be satisfied expires after the host-set limit, the forward reports
MOE_ERR_TIMEOUT through the status words, and the next normal forward on the
same device meets the oracle.  The unreachable waits come from the library's
test hook (a dependency counter target one above the units that exist, or a
grid barrier waiting for one CTA more than the grid has); nothing faults, traps
or spins without a bound."""
import numpy as np
import pytest
import torch

import moe_synth as ms
import oracle
import mxfp4_mixture_experts_gemv_gb300 as moe
from tests import moe_cases as mc

pytestmark = pytest.mark.gpu

LIMIT_NS = 1_000_000  # 1 ms: far above any healthy wait, far below the default 2 s


def _forward_with_held_waits(shape, which, seed):
    inp = ms.make_layer(shape, seed=seed)
    dev = inp.to("cuda")
    dims, packed = mc.pack(dev)
    ws = moe.alloc_workspace(dims, shape.T, shape.k)
    out = torch.full_like(dev.x, float("nan"))
    moe.set_wait_limit_ns(LIMIT_NS)
    moe.debug_hold_waits(which)
    try:
        moe.forward(dims, dev.x, dev.router_w, dev.router_b, packed, shape.k, out=out, workspace=ws)
        st = moe.device_status(ws)
    finally:
        moe.debug_hold_waits(0)
        moe.set_wait_limit_ns(0)
    assert moe.wait_limit_ns() == 2_000_000_000
    return inp, dev, packed, st


def _normal_forward_meets_the_oracle(inp, dev, packed):
    run = mc.run_gpu(dev, packed)  # asserts MOE_OK status
    s = inp.shape
    ref = oracle.moe_forward(inp.x, inp.router_w, inp.router_b, inp.gate_up_blocks, inp.gate_up_scales,
                             inp.gate_up_bias, inp.down_blocks, inp.down_scales, inp.down_bias, k=s.k)
    mc.compare_out(mc.bf16_to_f64(run.out), ref["out"], "after timeout", bf16_rounding=True)


@pytest.mark.parametrize("T", [4, 20, 64, 300],
                         ids=["cluster_route", "grid_route", "tensor_core_route", "tensor_core_route_128_row_tiles"])
def test_held_down_units_time_out_and_the_device_stays_usable(T):
    shape = ms.LayerShape(T=T, H=256, I=256, E=8, k=2)
    inp, dev, packed, st = _forward_with_held_waits(shape, moe.HOLD_DOWN_UNITS, seed=30 + T)
    assert st == 7, moe.STATUS_NAMES.get(st, st)  # MOE_ERR_TIMEOUT
    msg = moe.lib().moe_last_error().decode()
    assert "device wait expired" in msg
    _normal_forward_meets_the_oracle(inp, dev, packed)


@pytest.mark.parametrize("T", [20, 4], ids=["grid_route_barrier", "cluster_route_flags"])
def test_held_routing_barrier_times_out_and_the_device_stays_usable(T):
    """T = 20: the small-batch routing grid waits at its barrier for one CTA more
    than it has.  T = 4: the expert kernel waits for one more cluster-routing CTA
    than published its grouped rows (the flag it follows the running routing by)."""
    shape = ms.LayerShape(T=T, H=256, I=256, E=8, k=2)
    inp, dev, packed, st = _forward_with_held_waits(shape, moe.HOLD_ROUTING_BARRIER, seed=41 + T)
    assert st == 7, moe.STATUS_NAMES.get(st, st)
    assert "device wait expired" in moe.lib().moe_last_error().decode()
    _normal_forward_meets_the_oracle(inp, dev, packed)

