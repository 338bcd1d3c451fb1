"""The allocation-free entry point (moe_forward_static_scratch).

Some callers cannot allocate device memory (their device memory belongs to a
host runtime that forbids or budgets cudaMalloc, or an allocator call in their
launch path would synchronise the device).  For them the library keeps the
forward's scratch in a fixed-size array of its own device image.  These tests
check that entry point against the regular moe_forward on calls in a row
(including calls that switch between routing paths on the shared array), that
its status words are readable, and that bad calls are refused on the host with
moe_forward's own errors.

The file is named so pytest collects it last.
"""
import re
import os

import numpy as np
import pytest
import torch

import moe_synth as ms
import mxfp4_mixture_experts_gemv_gb300 as moe
from mxfp4_mixture_experts_gemv_gb300 import build as moe_build
from tests import moe_cases as mc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 1 << 20  # never dereferenced: every check here comes before any device work


def _header_scratch_bytes():
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        m = re.search(r"#define MOE_STATIC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", f.read())
    return int(m.group(1)) << int(m.group(2))


def test_static_scratch_size_matches_the_header():
    moe_build.build()
    assert moe.static_scratch_bytes() == _header_scratch_bytes()


def test_static_scratch_rejects_calls_larger_than_the_array():
    moe_build.build()
    L = moe.lib()
    dims = moe.LayerDims(128, 2880, 2880)
    T = 4096  # needs far more than MOE_STATIC_SCRATCH_BYTES
    assert moe.workspace_size(dims, T, 4) > moe.static_scratch_bytes()
    st = L.moe_forward_static_scratch(dims.c(), FAKE, T, FAKE, FAKE, FAKE, 4, FAKE, None)
    assert st == 4 and b"static scratch" in L.moe_last_error()
    # the largest documented call fits: gpt-oss shapes at T = 128, top-4
    assert moe.workspace_size(dims, 128, 4) <= moe.static_scratch_bytes()


@pytest.mark.parametrize("dims,T,k,want", [
    (moe.LayerDims(128, 2880, 2880), 4096, 9, 1),   # top_k > 8: an argument error, not a size error
    (moe.LayerDims(128, 2880, 2880), 4, 0, 1),
    (moe.LayerDims(128, 2880, 2880), -1, 4, 1),
    (moe.LayerDims(128, 2880, 2881), 4, 4, 2),      # H and I must be multiples of 32 / 64
    (moe.LayerDims(0, 2880, 2880), 4, 4, 1),
    (moe.LayerDims(300, 2880, 2880), 4, 4, 2),
])
def test_static_scratch_reports_argument_errors_like_moe_forward(dims, T, k, want):
    moe_build.build()
    L = moe.lib()
    st = L.moe_forward_static_scratch(dims.c(), FAKE, T, FAKE, FAKE, FAKE, k, FAKE, None)
    msg = L.moe_last_error()
    st2 = L.moe_forward(dims.c(), FAKE, T, FAKE, FAKE, FAKE, k, FAKE, FAKE, 1 << 40, None)
    assert st == want and st2 == want, (st, st2, msg)
    assert msg == L.moe_last_error()


def test_static_scratch_zero_tokens_is_a_noop():
    moe_build.build()
    L = moe.lib()
    dims = moe.LayerDims(128, 2880, 2880)
    assert L.moe_forward_static_scratch(dims.c(), None, 0, None, None, None, 4, None, None) == 0


def _check_twice(shape, seq):
    dev = ms.make_layer(shape, seed=21).to("cuda")
    dims, packed = mc.pack(dev)
    for call, T in enumerate(seq):
        x = ms.make_tokens(100 + call, T, shape.H).cuda()
        want = moe.forward(dims, x, dev.router_w, dev.router_b, packed, shape.k)
        got = moe.forward_static_scratch(dims, x, dev.router_w, dev.router_b, packed, shape.k)
        torch.cuda.synchronize()
        assert moe.static_scratch_status() == moe.MOE_OK
        g, w = mc.bf16_to_f64(got), mc.bf16_to_f64(want)
        mc.compare_out(g, w, f"static scratch call {call} (T={T})")
        assert np.array_equal(g, w), f"call {call} (T={T}): differs from moe_forward"


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [ms.LayerShape(T=8, H=256, I=256, E=8, k=2),
                                   ms.LayerShape(T=4, H=2880, I=2880, E=128, k=4)],
                         ids=["tiny", "gpt_oss_decode_t4"])
def test_static_scratch_matches_workspace_forward_twice(shape):
    _check_twice(shape, [shape.T, shape.T])  # two calls in a row share (and reuse) the static array


@pytest.mark.gpu
def test_static_scratch_switches_routing_paths_on_the_shared_array():
    """gpt-oss shapes: T = 32 (grid routing, cleared by a memset), T = 4 (cluster
    routing, which clears its own counters), T = 128 (tensor-core routing, the
    documented maximum), then T = 32 again, on the array the previous call left."""
    _check_twice(ms.LayerShape(T=128, H=2880, I=2880, E=128, k=4), [32, 4, 128, 32])
