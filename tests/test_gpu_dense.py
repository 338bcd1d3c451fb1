"""Dense MXFP4 linears (attention projections and LM head) through the C ABI
against the oracle: the BF16 -> MXFP4 weight quantiser bit-exact, and the
forward on both paths (CUDA cores for a few tokens, tensor cores) within the
layer tolerance, including a 64-row tail weight tile and a padded K."""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import moe_synth as ms
import oracle
import mxfp4_mixture_experts_gemv_gb300 as moe
from tests import moe_cases as mc

pytestmark = pytest.mark.gpu


def _weights(N, K, seed, std=0.05):
    g = torch.Generator().manual_seed(seed)
    w = (torch.randn(N, K, generator=g, dtype=torch.float64) * std).to(torch.bfloat16)
    b = (torch.randn(N, generator=g, dtype=torch.float64) * 0.02).to(torch.bfloat16)
    return w, b


def _oracle_rows(x, blocks, scales, bias, rows):
    """The oracle dense linear on the listed rows of x, one row per host thread."""
    with cf.ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as ex:
        parts = list(ex.map(lambda t: oracle.dense_linear(x[t:t + 1], blocks, scales, bias), rows))
    return np.concatenate(parts, axis=0)


@pytest.mark.parametrize("N,K", [(384, 256), (320, 288), (64, 32)])
def test_dense_weight_quantiser_matches_the_oracle(N, K):
    w, _ = _weights(N, K, seed=N + K)
    blocks, scales = moe.dense_quantize_weights(w.cuda())
    want_b, want_s = oracle.quantize_mxfp4_weights(w.float().double().numpy())
    np.testing.assert_array_equal(blocks.cpu().numpy(), want_b)
    np.testing.assert_array_equal(scales.cpu().numpy(), want_s)


@pytest.mark.parametrize("path", ["auto", "cuda_cores", "weights_m"])
@pytest.mark.parametrize("N,K,T", [(384, 256, 1), (320, 288, 3), (384, 256, 4), (320, 288, 40), (448, 512, 300)])
def test_dense_forward_matches_the_oracle(N, K, T, path):
    if path == "cuda_cores" and T > 4:
        pytest.skip("the CUDA-core path takes at most 4 tokens")
    w, b = _weights(N, K, seed=7 * N + T)
    x = ms.make_tokens(31, T, K)
    blocks, scales = moe.dense_quantize_weights(w.cuda())
    packed = moe.dense_pack(blocks, scales, b.cuda())
    moe.set_plan(0, "auto", path)
    try:
        out = moe.dense_forward(N, K, x.cuda(), packed)
        torch.cuda.synchronize()
    finally:
        moe.set_plan(0, "auto")
    ref = oracle.dense_linear(x, blocks.cpu(), scales.cpu(), b)
    mc.compare_out(mc.bf16_to_f64(out), ref, f"dense {N}x{K} T={T} {path}", bf16_rounding=True)


@pytest.mark.parametrize("N,K,T,path", [(5120, 2880, 4, "auto"), (2880, 4096, 4, "auto"), (5120, 2880, 64, "auto"),
                                         (2880, 4096, 200, "auto"), (5120, 2880, 4, "cuda_cores"),
                                         (2880, 4096, 2, "cuda_cores")],
                         ids=["qkv_t4", "o_t4", "qkv_t64", "o_t200", "qkv_t4_cuda_cores", "o_t2_cuda_cores"])
def test_dense_gpt_oss_projection_shapes(N, K, T, path):
    """gpt-oss-120b's attention projections (hidden 2880, 64 query and 8 KV heads of
    64: QKV 5120 outputs, O 2880 outputs from 4096), outputs of a token sample; the
    CUDA-core cases split K over up to 14 chunks per weight tile and sum them in order."""
    w, b = _weights(N, K, seed=N ^ K)
    x = ms.make_tokens(32, T, K)
    blocks, scales = moe.dense_quantize_weights(w.cuda())
    packed = moe.dense_pack(blocks, scales, b.cuda())
    moe.set_plan(0, "auto", path)
    try:
        out = mc.bf16_to_f64(moe.dense_forward(N, K, x.cuda(), packed))
    finally:
        moe.set_plan(0, "auto")
    rows = sorted(set(np.linspace(0, T - 1, min(T, 8)).astype(int).tolist()))
    ref = _oracle_rows(x, blocks.cpu(), scales.cpu(), b, rows)
    mc.compare_out(out[rows], ref, f"dense {N}x{K} T={T}")


def test_dense_lm_head_shape_t1():
    """The LM head (201,088 outputs from 2880) for one token on the CUDA-core path;
    every output against the oracle."""
    N, K = 201088, 2880
    g = torch.Generator(device="cuda").manual_seed(5)
    w = (torch.randn(N, K, generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    blocks, scales = moe.dense_quantize_weights(w)
    del w
    packed = moe.dense_pack(blocks, scales, None)
    x = ms.make_tokens(33, 1, K)
    out = mc.bf16_to_f64(moe.dense_forward(N, K, x.cuda(), packed))
    bc, sc = blocks.cpu(), scales.cpu()
    cuts = np.linspace(0, N, 17).astype(int)
    with cf.ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as ex:
        parts = list(ex.map(lambda ab: oracle.dense_linear(x, bc[ab[0]:ab[1]], sc[ab[0]:ab[1]]), zip(cuts[:-1], cuts[1:])))
    mc.compare_out(out, np.concatenate(parts, axis=1), "lm head T=1")

