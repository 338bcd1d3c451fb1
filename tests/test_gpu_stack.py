"""The stacked-layer workload, x <- x + moe(rmsnorm(x)): the residual/RMSNorm
kernel, and a chain of gpt-oss-shaped layers against the oracle's own chain."""
import numpy as np
import pytest
import torch

import moe_synth as ms
import oracle
import mxfp4_mixture_experts_gemv_gb300 as moe
from tests import moe_cases as mc

pytestmark = pytest.mark.gpu

# Bound on the relative Frobenius drift of chained layers (layer 0 uses the layer tolerance).
DRIFT_REL = 5e-2


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _widen(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_residual_rmsnorm_matches_oracle():
    T, H = 33, 2880
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(T, H, generator=g, dtype=torch.float64) * 3).float()
    prev = torch.randn(T, H, generator=g).to(torch.bfloat16)
    xr = x.clone().cuda()
    hidden = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    moe.residual_rmsnorm(xr, prev.cuda(), hidden)
    torch.cuda.synchronize()
    want_x = x.double().numpy() + _widen(_bits(prev))
    np.testing.assert_allclose(xr.cpu().double().numpy(), want_x, rtol=2 ** -23, atol=0)
    want_h = _widen(oracle.rmsnorm_bf16(want_x, 1e-5))
    got_h = _widen(_bits(hidden))
    # same bf16 grid: equal, or one bf16 step apart where the fp32 and fp64 norms round differently
    d = np.abs(got_h - want_h)
    assert (d <= 2.0 ** -7 * np.abs(want_h)).all()
    assert (d > 0).mean() < 0.01
    # no previous output: only the norm
    moe.residual_rmsnorm(xr, None, hidden)
    torch.cuda.synchronize()
    assert np.abs(_widen(_bits(hidden)) - want_h).max() <= 2.0 ** -7 * np.abs(want_h).max()


def test_three_layer_stack_matches_oracle_chain():
    H = I = 2880
    E, k, T, n_layers = 128, 4, 3, 3
    dims = moe.LayerDims(E, H, I)
    x0 = ms.make_tokens(0, T, H)
    # GPU chain
    xr = x0.float().cuda()
    hidden = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    outs, cpu_layers = [], []
    out = None
    for l in range(n_layers):
        w = ms.make_expert_weights(0, H, I, E, layer=l, device="cuda")
        packed = moe.pack_weights(dims, *w)
        rw, rb = ms.make_router(0, H, E, layer=l)
        cpu_layers.append((rw, rb, [t.cpu() for t in w]))
        moe.residual_rmsnorm(xr, out, hidden)
        out = moe.forward(dims, hidden, rw.cuda(), rb.cuda(), packed, k)
        outs.append(out.clone())
        torch.cuda.synchronize()
        del w, packed
    moe.residual_rmsnorm(xr, out, hidden)
    torch.cuda.synchronize()
    # oracle chain: the same recurrence with each layer's output rounded to bf16,
    # the layer's output format
    xo = _widen(_bits(x0))
    prev = None
    for l, (rw, rb, w) in enumerate(cpu_layers):
        if prev is not None:
            xo = xo + _widen(prev)
        h_bits = oracle.rmsnorm_bf16(xo, 1e-5)
        r = oracle.moe_forward(h_bits.view(np.uint16), rw, rb, *w, k=k)
        prev = oracle.bf16_round_array(r["out"])
        got = mc.bf16_to_f64(outs[l])
        if l == 0:
            # the first layer sees identical inputs: the layer tolerance holds
            mc.compare_out(got, r["out"], "layer 0", bf16_rounding=True)
        else:
            # later layers see inputs that already differ by the earlier layers' rounding
            # (about a quarter of the bf16 inputs one step apart), which the MXFP8
            # re-quantisation of x turns into code changes: only a bounded drift holds
            rel = np.linalg.norm(got - r["out"]) / np.linalg.norm(r["out"])
            print(f"layer {l}: relative drift {rel:.3g}")
            assert np.isfinite(got).all() and rel <= DRIFT_REL, f"layer {l}: drift {rel:.3g}"
    xo = xo + _widen(prev)
    rel = np.linalg.norm(xr.cpu().double().numpy() - xo) / np.linalg.norm(xo)
    print(f"residual after {n_layers} layers: relative drift {rel:.3g}")
    assert rel <= DRIFT_REL
