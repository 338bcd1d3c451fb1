"""The allocation-free entry point (moe_forward_static_scratch).

Some callers cannot allocate device memory (their device memory belongs to a
host runtime that forbids or budgets cudaMalloc, or an allocator call in their
launch path would synchronise the device).  For them the library keeps the
forward's scratch in a fixed-size array of its own device image.  These tests
check that entry point against the regular moe_forward on two calls in a row,
and that a call too large for the array is refused on the host.

The file is named so pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import moe_synth as ms
import mxfp4_mixture_experts_gemv_gb300 as moe
from mxfp4_mixture_experts_gemv_gb300 import build as moe_build
from tests import moe_cases as mc


def test_static_scratch_rejects_calls_larger_than_the_array():
    moe_build.build()
    L = moe.lib()
    dims = moe.LayerDims(128, 2880, 2880)
    T = 4096  # needs far more than MOE_STATIC_SCRATCH_BYTES
    assert moe.workspace_size(dims, T, 4) > moe.STATIC_SCRATCH_BYTES
    fake = 1 << 20  # never dereferenced: the size check comes first
    st = L.moe_forward_static_scratch(dims.c(), fake, T, fake, fake, fake, 4, fake, None)
    assert st == 4 and b"static scratch" in L.moe_last_error()


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [ms.LayerShape(T=8, H=256, I=256, E=8, k=2),
                                   ms.LayerShape(T=4, H=2880, I=2880, E=128, k=4)],
                         ids=["tiny", "gpt_oss_decode_t4"])
def test_static_scratch_matches_workspace_forward_twice(shape):
    dev = ms.make_layer(shape, seed=21).to("cuda")
    dims, packed = mc.pack(dev)
    for call in range(2):  # two calls in a row share (and reuse) the static array
        x = ms.make_tokens(100 + call, shape.T, shape.H).cuda()
        want = moe.forward(dims, x, dev.router_w, dev.router_b, packed, shape.k)
        got = moe.forward_static_scratch(dims, x, dev.router_w, dev.router_b, packed, shape.k)
        torch.cuda.synchronize()
        g, w = mc.bf16_to_f64(got), mc.bf16_to_f64(want)
        mc.compare_out(g, w, f"static scratch call {call}")
        assert np.array_equal(g, w), f"call {call}: differs from moe_forward"
