"""GPU parity: the CUDA path through the C ABI against the CPU oracle, stage by
stage (router ids and weights, MXFP8 codes of x, grouping, hq) and end to end."""
import numpy as np
import pytest
import torch

import moe_synth as ms
import oracle
import mxfp4_mixture_experts_gemv_gb300 as moe
from tests import moe_cases as mc

pytestmark = pytest.mark.gpu

# Small shapes that the oracle finishes in well under a second but that span
# several weight tiles, ragged token tiles and the padded contraction tails.
SMALL_CASES = {
    "tiny_T8_k2": (ms.LayerShape(T=8, H=256, I=256, E=8, k=2), 0),
    "T1_k1": (ms.LayerShape(T=1, H=256, I=256, E=8, k=1), 3),
    "ragged_T37_k4": (ms.LayerShape(T=37, H=256, I=256, E=8, k=4), 4),
    "many_tiles_T300": (ms.LayerShape(T=300, H=256, I=128, E=8, k=2), 5),
    "tails_H288_I192": (ms.LayerShape(T=50, H=288, I=192, E=6, k=3), 6),
    "k8_E16": (ms.LayerShape(T=20, H=128, I=64, E=16, k=8), 7),
    # a few tokens (cluster routing): experts not a multiple of the cluster, k = 8, E = 200
    "cluster_E6_tails": (ms.LayerShape(T=5, H=288, I=192, E=6, k=3), 10),
    "cluster_k8_E200": (ms.LayerShape(T=3, H=128, I=64, E=200, k=8), 11),
    # batched decode (grid routing) with padded contraction tails
    "grid_T12_tails": (ms.LayerShape(T=12, H=288, I=192, E=6, k=3), 12),
    # tensor-core router split along H (4 and 3 CTAs per token tile), one and two tiles
    "router_split_T40_H1024": (ms.LayerShape(T=40, H=1024, I=128, E=8, k=2), 13),
    "router_split_T150_E24": (ms.LayerShape(T=150, H=768, I=64, E=24, k=3), 14),
    # tensor-core router with more than 128 experts (MMA N = 256), k = 8
    "router_E200_k8": (ms.LayerShape(T=40, H=256, I=64, E=200, k=8), 15),
    # degenerate routing: one expert (every weight is 1), and k = E (every token takes
    # every expert), on the small-batch, cluster and tensor-core routing paths
    "single_expert_T20": (ms.LayerShape(T=20, H=128, I=64, E=1, k=1), 16),
    "single_expert_T40": (ms.LayerShape(T=40, H=256, I=64, E=1, k=1), 17),
    "k_equals_E_T6": (ms.LayerShape(T=6, H=128, I=64, E=2, k=2), 18),
    "k_equals_E_T70": (ms.LayerShape(T=70, H=256, I=128, E=2, k=2), 19),
}


def _full_check(inp_cpu, run, strict=True):
    s = inp_cpu.shape
    ref = oracle.moe_forward(inp_cpu.x, inp_cpu.router_w, inp_cpu.router_b, inp_cpu.gate_up_blocks,
                             inp_cpu.gate_up_scales, inp_cpu.gate_up_bias, inp_cpu.down_blocks,
                             inp_cpu.down_scales, inp_cpu.down_bias, k=s.k, intermediates=True,
                             act_format=run.act_format)
    ties = mc.check_routing(run, inp_cpu.x, inp_cpu.router_w, inp_cpu.router_b, ref["logits"])
    assert not ties, f"near-tie tokens {sorted(ties)}"
    mc.check_quantised_x(run, ref["xq"], ref["xs"])
    cnt, off, sr, inv = mc.check_grouping(run, s.T)
    mc.check_gathered(run, s.T, sr, ref["xq"], ref["xs"])
    allow, flips = mc.check_intermediate(run, ref, inp_cpu, inv)
    got = mc.bf16_to_f64(run.out)
    mc.compare_out(got, ref["out"], "out", allow=allow, bf16_rounding=not strict)
    return ref


@pytest.mark.parametrize("act_format", ["mxfp8", "mxfp4", "nvfp4"])
@pytest.mark.parametrize("name", list(SMALL_CASES))
def test_small_layer_parity(name, act_format):
    shape, seed = SMALL_CASES[name]
    if act_format == "nvfp4" and (shape.H % 64 or shape.I % 64):
        pytest.skip("NVFP4 packing needs H and I multiples of 64")
    inp = ms.make_layer(shape, seed=seed)
    dev = inp.to("cuda")
    _, packed = mc.pack(dev, nvfp4=act_format == "nvfp4")
    run = mc.run_gpu(dev, packed, act_format=act_format)
    _full_check(inp, run, strict=False)


def _untile(flat, E, rows_stored, Kp):
    """Tile-contiguous data ([E][m][kt][rows_m][64 B]) back to [E][rows_stored][Kp/2] bytes."""
    kt_n = Kp // 128
    out = np.zeros((E, rows_stored, Kp // 2), np.uint8)
    pos = 0
    for e in range(E):
        for m in range(0, rows_stored, 128):
            rows_m = min(128, rows_stored - m)
            for kt in range(kt_n):
                n = rows_m * 64
                out[e, m:m + rows_m, kt * 64:(kt + 1) * 64] = flat[pos:pos + n].reshape(rows_m, 64)
                pos += n
    assert pos == flat.size
    return out


def test_pack_is_a_bijection_with_deterministic_padding():
    shape = ms.LayerShape(T=1, H=288, I=192, E=3, k=1)
    inp = ms.make_layer(shape, seed=9)
    dev = inp.to("cuda")
    _, packed = mc.pack(dev)
    pk = packed.cpu().numpy()
    E, H, I = shape.E, shape.H, shape.I
    Hp, Ip = 384, 256
    Hs = 320  # down rows stored: H rounded up to 64
    hdr = pk[:64].view(np.uint32)
    assert hdr[0] == 0x4D584645 and hdr[1] == 2 and tuple(hdr[2:5]) == (E, H, I)
    assert tuple(hdr[11:13]) == (2 * I, Hs)
    offs = pk[56:112].view(np.uint64)
    gu_data, gu_sf, gu_b, d_data, d_sf, d_b, total = (int(o) for o in offs)
    assert total == moe.packed_size(moe.LayerDims(E, H, I))
    # gate_up rows: tile t = gate rows 64t.., then up rows I+64t..
    src_row = np.array([(64 * (r // 128) + r % 128) if r % 128 < 64 else (I + 64 * (r // 128) + r % 128 - 64)
                        for r in range(2 * I)])
    gub = inp.gate_up_blocks.numpy().reshape(E, 2 * I, H // 2)
    got = _untile(pk[gu_data:gu_data + E * 2 * I * Hp // 2], E, 2 * I, Hp)
    np.testing.assert_array_equal(got[:, :, :H // 2], gub[:, src_row])
    assert (got[:, :, H // 2:] == 0).all()
    db = inp.down_blocks.numpy().reshape(E, H, I // 2)
    got = _untile(pk[d_data:d_data + E * Hs * Ip // 2], E, Hs, Ip)
    np.testing.assert_array_equal(got[:, :H, :I // 2], db)
    assert (got[:, :, I // 2:] == 0).all() and (got[:, H:, :] == 0).all()

    def atoms(base, rows, nb, kt, src):
        mt = (rows + 127) // 128
        a = pk[base:base + E * mt * kt * 512].reshape(E, mt, kt, 512)
        full = np.full((E, mt * 128, kt * 4), 127, np.uint8)
        j = np.arange(512)
        r = (j >> 4) + 32 * ((j & 15) >> 2)
        kb = j & 3
        for m in range(mt):
            for kk in range(kt):
                full[:, m * 128 + r, kk * 4 + kb] = a[:, m, kk, j]
        assert (full[:, :rows, :nb] == src).all()
        assert (full[:, rows:, :] == 127).all() and (full[:, :, nb:] == 127).all()

    atoms(gu_sf, 2 * I, H // 32, Hp // 128, inp.gate_up_scales.numpy()[:, src_row])
    atoms(d_sf, H, I // 32, Ip // 128, inp.down_scales.numpy())
    bias = pk[gu_b:gu_b + E * 2 * I * 4].view(np.float32).reshape(E, 2 * I)
    np.testing.assert_array_equal(bias, inp.gate_up_bias.float().numpy()[:, src_row])
    bias = pk[d_b:d_b + E * H * 4].view(np.float32).reshape(E, H)
    np.testing.assert_array_equal(bias, inp.down_bias.float().numpy())


@pytest.mark.parametrize("T", [4, 20, 64], ids=["cluster_route", "grid_route", "tensor_core_route"])
def test_deterministic_and_independent_of_workspace_contents(T):
    shape = ms.LayerShape(T=T, H=256, I=256, E=8, k=4)
    inp = ms.make_layer(shape, seed=11).to("cuda")
    _, packed = mc.pack(inp)
    a = mc.run_gpu(inp, packed, poison=0x00)
    b = mc.run_gpu(inp, packed, poison=0xFF)
    c = mc.run_gpu(inp, packed, poison=0x7F)
    for r in (b, c):
        assert torch.equal(a.out.view(torch.int16), r.out.view(torch.int16))
        for name, shp in [("topk_ids", (T * 4,)), ("sorted_rows", (T * 4,)), ("inv_pos", (T * 4,))]:
            assert torch.equal(a.section(name, shp, torch.int32), r.section(name, shp, torch.int32))


def test_zero_tokens_is_a_noop():
    shape = ms.LayerShape(T=4, H=256, I=256, E=8, k=2)
    inp = ms.make_layer(shape, seed=1).to("cuda")
    dims, packed = mc.pack(inp)
    out = torch.full((0, 256), 1.0, dtype=torch.bfloat16, device="cuda")
    ws = moe.alloc_workspace(dims, 1, 2)
    moe.forward(dims, inp.x[:0], inp.router_w, inp.router_b, packed, 2, out=out, workspace=ws)
    torch.cuda.synchronize()


# ----------------------------------------------------------------------- gpt-oss-shaped layer
@pytest.fixture(scope="module")
def gpt_layer():
    H = I = 2880
    E = 128
    w = ms.make_expert_weights(0, H, I, E, device="cuda")
    dims = moe.LayerDims(E, H, I)
    packed = moe.pack_weights(dims, *w)
    cpu = [t.cpu() for t in w]
    return dims, packed, w, cpu


_NV_PACKED = {}


def _nvfp4_packed(gpt_layer):
    """The gpt-oss layer's weights converted to NVFP4 (packed once per module)."""
    dims, packed, w, cpu = gpt_layer
    key = packed.data_ptr()
    if key not in _NV_PACKED:
        _NV_PACKED.clear()
        _NV_PACKED[key] = moe.pack_weights(dims, *w, nvfp4=True)
    return _NV_PACKED[key]


def _gpt_inputs(gpt_layer, T, hot=0, hot_bias=0.0):
    dims, packed, w, cpu = gpt_layer
    shape = ms.LayerShape(T=T, H=dims.H, I=dims.I, E=dims.E, k=4)
    x = ms.make_tokens(0, T, dims.H)
    rw, rb = ms.make_router(0, dims.H, dims.E, hot_experts=hot, hot_bias=hot_bias)
    cpu_inp = ms.LayerInputs(shape, x, rw, rb, *cpu)
    dev_inp = ms.LayerInputs(shape, x.cuda(), rw.cuda(), rb.cuda(), *w)
    return cpu_inp, dev_inp, packed


@pytest.mark.parametrize("act_format", ["mxfp8", "mxfp4", "nvfp4"])
@pytest.mark.parametrize("T,hot", [(4, 0), (32, 16)], ids=["decode_t4", "decode_t32_skewed"])
def test_gpt_oss_decode_parity(gpt_layer, T, hot, act_format):
    cpu_inp, dev_inp, packed = _gpt_inputs(gpt_layer, T, hot, 1.0 if hot else 0.0)
    if act_format == "nvfp4":
        packed = _nvfp4_packed(gpt_layer)
    run = mc.run_gpu(dev_inp, packed, act_format=act_format)
    _full_check(cpu_inp, run)


@pytest.mark.parametrize("act_format", ["mxfp8", "mxfp4", "nvfp4"])
def test_gpt_oss_prefill_sampled_parity(gpt_layer, act_format):
    """T = 2048 with the launch configuration of the benchmark; all ids and the
    whole grouping are checked, the output on a sample of tokens."""
    T = 2048
    cpu_inp, dev_inp, packed = _gpt_inputs(gpt_layer, T)
    if act_format == "nvfp4":
        packed = _nvfp4_packed(gpt_layer)
    run = mc.run_gpu(dev_inp, packed, act_format=act_format)
    logits, ids_ref, _ = oracle.route(cpu_inp.x, cpu_inp.router_w, cpu_inp.router_b, 4)
    ties = mc.check_routing(run, cpu_inp.x, cpu_inp.router_w, cpu_inp.router_b, logits)
    cnt, off, sr, inv = mc.check_grouping(run, T)
    # sample: spread tokens plus the tokens of the most loaded expert's last tile
    e_max = int(np.argmax(cnt))
    last = [int(sr[p]) // 4 for p in range(off[e_max + 1] - 3, off[e_max + 1])]
    sample = sorted(set(list(range(0, T, 257)) + last + [T - 1]) - ties)
    sub = cpu_inp.x[sample]
    ref = oracle.moe_forward(sub, cpu_inp.router_w, cpu_inp.router_b, *cpu_inp_weights(cpu_inp), k=4,
                             intermediates=True, act_format=act_format)
    allow, _ = mc.check_intermediate(run, ref, cpu_inp, inv.reshape(T, 4)[sample])
    got = mc.bf16_to_f64(run.out)[sample]
    mc.compare_out(got, ref["out"], "prefill sample", allow=allow)


def cpu_inp_weights(c):
    return (c.gate_up_blocks, c.gate_up_scales, c.gate_up_bias, c.down_blocks, c.down_scales, c.down_bias)


# ----------------------------------------------------------------------- plans
@pytest.mark.parametrize("T,tile_rows,route,expert", [
    (6, 8, "cluster", "auto"), (6, 32, "cluster", "auto"), (6, 16, "grid", "auto"), (6, 64, "tensor_core", "auto"),
    (20, 8, "grid", "auto"), (20, 64, "grid", "auto"), (20, 16, "tensor_core", "auto"),
    (20, 128, "tensor_core", "weights_m"), (20, 128, "grid", "tokens_m"),
    (70, 32, "tensor_core", "auto"), (70, 8, "tensor_core", "auto"),
    (300, 128, "auto", "weights_m"), (300, 128, "auto", "tokens_m"),
])
def test_forced_plans_meet_the_oracle(T, tile_rows, route, expert):
    """Every tile height on every routing path that fits, and both expert kernels
    on 128-row tiles: the plan changes launch shapes only, never the result beyond
    the layer tolerance."""
    shape = ms.LayerShape(T=T, H=256, I=128, E=8, k=4)
    inp = ms.make_layer(shape, seed=50 + T)
    dev = inp.to("cuda")
    _, packed = mc.pack(dev)
    moe.set_plan(tile_rows, route, expert)
    try:
        run = mc.run_gpu(dev, packed)
        assert run.layout.tile_rows == tile_rows
        _full_check(inp, run, strict=False)
    finally:
        moe.set_plan(0, "auto")


@pytest.mark.parametrize("act_format", ["mxfp8", "mxfp4", "nvfp4"])
@pytest.mark.parametrize("expert", ["weights_m", "tokens_m"])
def test_both_expert_kernels_on_ragged_tails(expert, act_format):
    """Ragged shapes: a 64-row down tail tile, three gate_up tiles (one pair and a
    single), 128-row token tiles with a ragged last tile; MXFP8, MXFP4 and NVFP4
    activations (kind::mxf8f6f4, kind::mxf4, kind::mxf4nvf4).  H = 288 and I = 192
    (NVFP4 packing needs multiples of 64: H = 320 there)."""
    shape = ms.LayerShape(T=90, H=320 if act_format == "nvfp4" else 288, I=192, E=6, k=3)
    inp = ms.make_layer(shape, seed=61)
    dev = inp.to("cuda")
    _, packed = mc.pack(dev, nvfp4=act_format == "nvfp4")
    moe.set_plan(128, "auto", expert)
    try:
        run = mc.run_gpu(dev, packed, act_format=act_format)
        _full_check(inp, run, strict=False)
    finally:
        moe.set_plan(0, "auto")


@pytest.mark.parametrize("act_format", ["mxfp4", "nvfp4"])
@pytest.mark.parametrize("T", [20, 300])
def test_tokens_on_m_kernel_with_fp4_activations(T, act_format):
    """The tokens-on-M kernel in its kind::mxf4 and kind::mxf4nvf4 forms (both
    operands packed, eight stages) on 128-row token tiles."""
    shape = ms.LayerShape(T=T, H=256, I=128, E=8, k=4)
    inp = ms.make_layer(shape, seed=70 + T)
    dev = inp.to("cuda")
    _, packed = mc.pack(dev, nvfp4=act_format == "nvfp4")
    moe.set_plan(128, "auto", "tokens_m")
    try:
        run = mc.run_gpu(dev, packed, act_format=act_format)
        assert run.layout.tile_rows == 128
        _full_check(inp, run, strict=False)
    finally:
        moe.set_plan(0, "auto")


def test_forced_route_that_does_not_fit_is_refused():
    shape = ms.LayerShape(T=40, H=256, I=128, E=8, k=4)
    dev = ms.make_layer(shape, seed=1).to("cuda")
    dims, packed = mc.pack(dev)
    moe.set_plan(0, "grid")  # the grid routing kernel holds at most 32 tokens
    try:
        with pytest.raises(moe.MoeError, match="UNSUPPORTED_SHAPE"):
            moe.forward(dims, dev.x, dev.router_w, dev.router_b, packed, 4)
    finally:
        moe.set_plan(0, "auto")


@pytest.mark.parametrize("T,act_format", [(8, "mxfp8"), (9, "mxfp8"), (32, "mxfp8"), (33, "mxfp8"), (128, "mxfp8"),
                                          (129, "mxfp8"), (224, "mxfp8"), (225, "mxfp8"), (512, "mxfp8"),
                                          (1024, "mxfp8"), (2048, "mxfp8"), (224, "mxfp4"), (225, "mxfp4"),
                                          (1024, "mxfp4")])
def test_gpt_oss_parity_at_the_plan_cutoffs(gpt_layer, T, act_format):
    """Either side of every automatic cutoff: cluster / grid routing at 8, grid /
    tensor-core routing at 32, token tiles of 8 / 16 rows at 128, and 16-row tiles
    (weights-on-M kernel) / 128-row tiles (tokens-on-M kernel) at 224 (7 / 8 rows
    per expert on average), for MXFP8 and MXFP4 activations; then the tokens-on-M
    kernel at 512, 1024 and 2048.  Routing, grouping and the gathered rows are
    checked for every token, the output on up to 24 tokens (the oracle runs one
    token per host thread)."""
    cpu_inp, dev_inp, packed = _gpt_inputs(gpt_layer, T)
    run = mc.run_gpu(dev_inp, packed, act_format=act_format)
    logits, _, _ = oracle.route(cpu_inp.x, cpu_inp.router_w, cpu_inp.router_b, 4)
    ties = mc.check_routing(run, cpu_inp.x, cpu_inp.router_w, cpu_inp.router_b, logits)
    cnt, off, sr, inv = mc.check_grouping(run, T)
    if act_format == "mxfp8":
        xq, xs = oracle.mxfp8_quantize(mc.bf16_to_f64(cpu_inp.x))
        mc.check_quantised_x(run, xq, xs)
        mc.check_gathered(run, T, sr, xq, xs)
    e_max = int(np.argmax(cnt))
    last = [int(sr[p]) // 4 for p in range(max(off[e_max], off[e_max + 1] - 4), off[e_max + 1])]
    spread = np.linspace(0, T - 1, min(T, 20)).astype(int).tolist()
    sample = sorted(set(spread + last) - ties)
    ref = mc.oracle_tokens_parallel(cpu_inp, sample, act_format)
    allow, _ = mc.check_intermediate(run, ref, cpu_inp, inv.reshape(T, 4)[sample])
    mc.compare_out(mc.bf16_to_f64(run.out)[sample], ref["out"], f"T={T} {act_format}", allow=allow)


def test_nvfp4_pack_matches_the_oracle_conversion():
    """The NVFP4 repacker, unpacked from its tiles and scale atoms, equals the oracle's
    conversion of the MXFP4 checkpoint (codes and E4M3 scales of every row, bit-exact),
    and it records each projection's amax, from which both sides take the global scale."""
    shape = ms.LayerShape(T=1, H=256, I=192, E=3, k=1)
    inp = ms.make_layer(shape, seed=23)
    dev = inp.to("cuda")
    _, packed = mc.pack(dev, nvfp4=True)
    pk = packed.cpu().numpy()
    E, H, I = shape.E, shape.H, shape.I
    assert pk[52:56].view(np.int32)[0] == 1  # weight format: NVFP4
    offs = pk[56:112].view(np.uint64)
    gu_data, gu_sf, gu_b, d_data, d_sf, d_b, total = (int(o) for o in offs)
    assert total == moe.lib().moe_packed_size_nvfp4(moe.LayerDims(E, H, I).c())
    amax = pk[512:520].view(np.float32).astype(np.float64)
    assert amax[0] == oracle.mxfp4_amax(inp.gate_up_blocks, inp.gate_up_scales)
    assert amax[1] == oracle.mxfp4_amax(inp.down_blocks, inp.down_scales)

    def check(data_off, sf_off, rows, rows_stored, K, blocks, scales, src_row):
        kt_n, mt_n = (K + 127) // 128, (rows_stored + 127) // 128
        gs = oracle.nvfp4_global_scale(oracle.mxfp4_amax(blocks, scales))
        flat = pk[data_off:data_off + E * rows_stored * kt_n * 64]
        sfa = pk[sf_off:sf_off + E * mt_n * kt_n * 2 * 512].reshape(E, mt_n, kt_n, 2, 512)
        untiled = _untile(flat, E, rows_stored, kt_n * 128)
        for e in range(E):
            want_c, want_s = oracle.convert_mxfp4_to_nvfp4(blocks[e], scales[e], gs)
            got = np.empty((rows_stored, kt_n * 128), np.uint8)
            got[:, 0::2] = untiled[e] & 15
            got[:, 1::2] = untiled[e] >> 4
            r = np.arange(rows)
            np.testing.assert_array_equal(got[r, :K], want_c[src_row(r)])
            assert (got[:, K:] == 0).all() and (got[rows:] == 0).all()
            q = np.arange(K // 16)
            byte = ((r % 32) * 16 + ((r % 128) // 32) * 4)[:, None] + (q % 4)[None, :]
            s = sfa[e, (r // 128)[:, None], (q // 8)[None, :], ((q // 4) % 2)[None, :], byte]
            np.testing.assert_array_equal(s, want_s[src_row(r)])

    gu_src = np.vectorize(lambda pr: (64 * (pr // 128) + pr % 128) if pr % 128 < 64 else (I + 64 * (pr // 128) + pr % 128 - 64))
    check(gu_data, gu_sf, 2 * I, 2 * I, H, inp.gate_up_blocks.numpy(), inp.gate_up_scales.numpy(), gu_src)
    check(d_data, d_sf, H, 256, I, inp.down_blocks.numpy(), inp.down_scales.numpy(), lambda r: r)


def test_formats_alternate_on_one_packed_address():
    """The same device address packed as MXFP4, then NVFP4, then MXFP4 again (the
    caching allocator hands freed buffers back): each forward must use the layout
    of the buffer it is given, not descriptors cached for the previous one."""
    shape = ms.LayerShape(T=5, H=128, I=64, E=6, k=2)
    inp = ms.make_layer(shape, seed=44)
    dev = inp.to("cuda")
    dims = moe.LayerDims(shape.E, shape.H, shape.I)
    n = max(moe.packed_size(dims), moe.lib().moe_packed_size_nvfp4(dims.c()))
    buf = moe._alloc_aligned(n, "cuda")
    for fmt in ("mxfp8", "nvfp4", "mxfp4", "nvfp4"):
        w = (dev.gate_up_blocks, dev.gate_up_scales, dev.gate_up_bias, dev.down_blocks, dev.down_scales, dev.down_bias)
        packed = moe.pack_weights(dims, *w, packed=buf, nvfp4=fmt == "nvfp4")
        run = mc.run_gpu(dev, packed, act_format=fmt)
        _full_check(inp, run, strict=False)
