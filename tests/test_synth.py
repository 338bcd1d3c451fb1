"""The seeded input generator: published splitmix64 outputs, slicing, distributions."""
import math

import numpy as np
import torch

import moe_synth as ms


def _splitmix64_py(state, n):
    """Plain-integer splitmix64 (Steele, Lea, Flood 2014), for cross-checking the torch lanes."""
    out = []
    M = (1 << 64) - 1
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & M
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M
        out.append(z ^ (z >> 31))
    return out


def test_splitmix64_published_sequence_from_zero():
    # first outputs of splitmix64 seeded with 0, as published with the reference C code
    assert _splitmix64_py(0, 3) == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_torch_lanes_equal_integer_splitmix64():
    for seed, stream in [(0, 1), (7, 300), (123456789, 47)]:
        key = ms.stream_key(seed, stream) & ((1 << 64) - 1)
        ref = _splitmix64_py(key, 50)
        got = [int(v) & ((1 << 64) - 1) for v in ms.hashes(seed, stream, 0, 50)]
        assert got == ref


def test_slices_are_consistent():
    full = ms.rand_bytes(3, 4, 0, 1000)
    for a, n in [(0, 1), (5, 17), (8, 8), (123, 400), (999, 1)]:
        assert torch.equal(ms.rand_bytes(3, 4, a, n), full[a:a + n])
    g = ms.rand_normal_bf16(3, 6, 0, 500, 0.5)
    assert torch.equal(ms.rand_normal_bf16(3, 6, 100, 50, 0.5), g[100:150])
    gub, gus, gubias, db, ds, dbias = ms.make_expert_weights(1, 64, 32, 4)
    sub = ms.make_expert_weights(1, 64, 32, 4, experts=[2])
    for full_t, sub_t in zip((gub, gus, gubias, db, ds, dbias), sub):
        assert torch.equal(full_t[2:3], sub_t)


def test_distributions():
    n = 200000
    z = ms.rand_normal_bf16(0, 1, 0, n, 1.0).double()
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    s = ms.rand_scales(0, 5, 0, n)
    assert int(s.min()) == 118 and int(s.max()) == 124
    counts = torch.bincount(s.long() - 118, minlength=7).double() / n
    assert (counts - 1 / 7).abs().max() < 0.01
    b = ms.rand_bytes(0, 4, 0, n)
    nib = torch.cat([b & 0xF, b >> 4]).long()
    assert ((torch.bincount(nib, minlength=16).double() / (2 * n)) - 1 / 16).abs().max() < 0.005


def test_router_skew_and_shapes():
    shape = ms.LayerShape(T=3, H=64, I=32, E=20, k=4)
    a = ms.make_layer(shape, seed=2)
    b = ms.make_layer(shape, seed=2, hot_experts=16, hot_bias=1.0)
    assert a.x.shape == (3, 64) and a.router_w.shape == (20, 64)
    assert a.gate_up_blocks.shape == (20, 64, 2, 16) and a.down_scales.shape == (20, 64, 1)
    d = (b.router_b.double() - a.router_b.double())
    assert torch.allclose(d[:16], torch.ones(16, dtype=torch.float64), atol=0.01)
    assert (d[16:] == 0).all()
    assert abs(a.router_w.double().std() - 1 / math.sqrt(64)) < 0.01
