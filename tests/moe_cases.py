"""Shared helpers of the GPU parity tests: build a case, run the C ABI, run the
oracle, and compare stage by stage."""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import math
import os

import numpy as np
import torch

import moe_synth as ms
import oracle
import mxfp4_mixture_experts_gemv_gb300 as moe

# Output tolerances of the layer (fp32 GPU path with one bf16 rounding vs the
# fp64 oracle): max |d| <= 2e-2 * rms(ref) and ||d||_F / ||ref||_F <= 5e-3.
MAX_ABS_OVER_RMS = 2e-2
REL_FRO = 5e-3
TOPK_W_ATOL = 1e-6


@dataclasses.dataclass
class GpuForward:
    dims: moe.LayerDims
    k: int
    out: torch.Tensor
    ws: torch.Tensor
    layout: moe.WorkspaceLayout
    act_format: str = "mxfp8"

    @property
    def fp4(self) -> bool:
        return self.act_format in ("mxfp4", "nvfp4")

    @property
    def nv(self) -> bool:
        return self.act_format == "nvfp4"

    @property
    def block(self) -> int:
        """Elements per activation scale: 16 for NVFP4, 32 for the MX formats."""
        return 16 if self.nv else 32

    def atom_scales(self, section, rows_of, n_rows, K, n_blocks=None):
        """Scale codes of the listed grouped rows from a scale-atom section: [rows, blocks].
        MX formats: one atom per 128-element k-tile, byte (n%32)*16 + (n/32)*4 + block%4;
        NVFP4: two atoms per k-tile, atom (block/4)%2 of k-tile block/8."""
        L = self.layout
        kt = (K + 127) // 128
        atoms = self.section(section, (L.max_tiles, kt, 2, 512) if self.nv else (L.max_tiles, kt, 512),
                             torch.uint8).numpy()
        tiles = self.section("tiles", (4 + 4 * L.max_tiles,), torch.int32).numpy()
        td = tiles[4:4 + 4 * tiles[0]].reshape(-1, 4)
        pos = np.asarray(rows_of, np.int64)
        b = np.searchsorted(td[:, 1], pos, side="right") - 1
        n = pos - td[b, 1]
        nb = n_blocks if n_blocks is not None else (8 if self.nv else 4) * kt
        kb = np.arange(nb)
        byte = ((n % 32) * 16 + (n // 32) * 4)[:, None] + (kb % 4)[None, :]
        if self.nv:
            return atoms[b[:, None], (kb // 8)[None, :], ((kb // 4) % 2)[None, :], byte]
        return atoms[b[:, None], (kb // 4)[None, :], byte]

    def scale_values(self, codes):
        """Scale multipliers of scale codes: 2^(code - 127) (E8M0) or the E4M3 value."""
        if self.nv:
            return _code_table(False)[codes]
        return np.ldexp(1.0, codes.astype(np.int64) - 127)

    def codes(self, name, rows, cols):
        """Activation codes of a workspace section, one code per element: E4M3 bytes,
        or E2M1 nibbles unpacked (two per byte, the even element in the low nibble)."""
        if not self.fp4:
            return self.section(name, (rows, cols), torch.uint8).numpy()
        return unpack_e2m1(self.section(name, (rows, cols // 2), torch.uint8).numpy())

    def section(self, name, shape, dtype):
        return moe.view(self.ws, getattr(self.layout, name), shape, dtype).cpu()


def pack(inp: ms.LayerInputs, nvfp4: bool = False):
    s = inp.shape
    dims = moe.LayerDims(s.E, s.H, s.I)
    packed = moe.pack_weights(dims, inp.gate_up_blocks, inp.gate_up_scales, inp.gate_up_bias,
                              inp.down_blocks, inp.down_scales, inp.down_bias, nvfp4=nvfp4)
    return dims, packed


def unpack_e2m1(a: np.ndarray) -> np.ndarray:
    out = np.empty(a.shape[:-1] + (2 * a.shape[-1],), np.uint8)
    out[..., 0::2] = a & 0xF
    out[..., 1::2] = a >> 4
    return out


def zero_codes_equal(codes: np.ndarray, fp4: bool) -> np.ndarray:
    """The negative-zero code read as the positive one: both encode zero, and which
    of the two a rounding of a tiny negative value gives is not part of the format."""
    c = codes.copy()
    c[c == (0x8 if fp4 else 0x80)] = 0
    return c


def run_gpu(inp: ms.LayerInputs, packed, x=None, poison: int | None = None, act_format: str = "mxfp8") -> GpuForward:
    s = inp.shape
    dims = moe.LayerDims(s.E, s.H, s.I)
    x = inp.x if x is None else x
    T = x.shape[0]
    ws = moe.alloc_workspace(dims, T, s.k, x.device)
    if poison is not None:
        ws.fill_(poison)
    out = torch.full_like(x, float("nan"))
    moe.forward(dims, x, inp.router_w, inp.router_b, packed, s.k, out=out, workspace=ws, act_format=act_format)
    st = moe.device_status(ws)
    assert st == moe.MOE_OK, moe.STATUS_NAMES.get(st, st)
    return GpuForward(dims, s.k, out, ws, moe.workspace_layout(dims, T, s.k, act_format), act_format)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().double().numpy()


def _widen(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_routing(run: GpuForward, x_cpu, wr_cpu, br_cpu, logits_ref: np.ndarray):
    """Router ids: equal to the oracle's, or a valid selection under fp32 near-ties.

    Returns the set of tokens whose ids differ (accepted near-ties)."""
    T, E = logits_ref.shape
    k = run.k
    ids = run.section("topk_ids", (T, k), torch.int32).numpy()
    w = run.section("topk_w", (T, k), torch.float32).numpy().astype(np.float64)
    xf = _widen(x_cpu.view(torch.int16).numpy().view(np.uint16))
    wf = _widen(wr_cpu.view(torch.int16).numpy().view(np.uint16))
    bf = _widen(br_cpu.view(torch.int16).numpy().view(np.uint16))
    l32 = logits_ref.astype(np.float32)
    # GPU logits within the fp32 dot-product error bound of the exact ones
    gl = run.section("logits", (T, E), torch.float32).numpy().astype(np.float64)
    absdot = np.abs(xf) @ np.abs(wf).T
    bound = H_gamma(xf.shape[1]) * absdot + 2.0 ** -23 * (np.abs(logits_ref) + np.abs(bf))
    assert (np.abs(gl - logits_ref) <= bound).all(), f"logits off by {np.abs(gl - logits_ref).max():.3g}"
    # the oracle's selection: experts by fp32 logit descending, lower index first on ties
    want = np.argsort(-l32, axis=1, kind="stable")[:, :k]
    ties = set()
    for t in np.nonzero((ids != want).any(axis=1))[0]:
        # accept only a selection that fp32 rounding can explain
        assert len(set(ids[t].tolist())) == k, f"token {t}: repeated expert ids {ids[t]}"
        err = H_gamma(xf.shape[1]) * absdot[t] + 2 ** -23 * np.abs(logits_ref[t]) + np.abs(bf) * 2 ** -24
        sel = ids[t]
        rest = np.setdiff1d(np.arange(E), sel)
        lo_sel = min(logits_ref[t, e] + err[e] for e in sel)
        hi_rest = max(logits_ref[t, e] - err[e] for e in rest)
        assert lo_sel >= hi_rest, f"token {t}: ids {ids[t]} vs oracle {want[t]} beyond fp32 error"
        for a, b in zip(sel, sel[1:]):
            assert logits_ref[t, a] + err[a] >= logits_ref[t, b] - err[b], f"token {t}: order"
        ties.add(int(t))
    # weights: a logit error d moves a softmax weight by at most 0.5 * max|d| (its
    # Jacobian row sums to 2 w (1 - w) <= 0.5), plus fp32 rounding
    sel_l = np.take_along_axis(logits_ref, ids.astype(np.int64), axis=1)
    ref_w = np.exp(sel_l - sel_l[:, :1])
    ref_w /= ref_w.sum(axis=1, keepdims=True)
    dl = np.abs(np.take_along_axis(gl, ids.astype(np.int64), axis=1) - sel_l).max(axis=1)
    over = np.abs(w - ref_w) > (0.5 * dl + TOPK_W_ATOL)[:, None]
    assert not over.any(), f"routing weights of token {np.argwhere(over)[0][0]} off"
    return ties


def H_gamma(n: int) -> float:
    u = 2.0 ** -24
    return n * u / (1 - n * u)


def check_quantised_x(run: GpuForward, xq_ref, xs_ref):
    T, H = xq_ref.shape
    xq = run.codes("xq", T, H)
    xs = run.section("xs", (T, H // run.block), torch.uint8).numpy()
    np.testing.assert_array_equal(zero_codes_equal(xq, run.fp4), zero_codes_equal(xq_ref, run.fp4))
    np.testing.assert_array_equal(xs, xs_ref)


def check_gathered(run: GpuForward, T: int, sr: np.ndarray, xq_ref: np.ndarray, xs_ref: np.ndarray):
    """The grouped MXFP8 rows, bit-exact: row p holds the oracle's codes of token
    sorted_rows[p] // k, and its scale-atom entry the token's block scales (127 on
    the padding blocks past H/32)."""
    H, k = run.dims.H, run.k
    L = run.layout
    TK = T * k
    xp = run.codes("xp", TK, H)
    np.testing.assert_array_equal(zero_codes_equal(xp, run.fp4), zero_codes_equal(xq_ref[sr // k], run.fp4))
    sc = run.atom_scales("xp_sf", np.arange(TK), TK, H)
    # padding blocks past H: the neutral E8M0 scale, or the zero E4M3 scale
    want = np.full(sc.shape, 0 if run.nv else 127, np.uint8)
    want[:, :H // run.block] = xs_ref[sr // k]
    np.testing.assert_array_equal(sc, want)


def check_grouping(run: GpuForward, T: int):
    E, k = run.dims.E, run.k
    ids = run.section("topk_ids", (T, k), torch.int32).numpy()
    cnt, off, sr, inv = oracle.permute(ids, E)
    np.testing.assert_array_equal(run.section("counts", (E,), torch.int32).numpy(), cnt)
    np.testing.assert_array_equal(run.section("offsets", (E + 1,), torch.int32).numpy(), off)
    np.testing.assert_array_equal(run.section("sorted_rows", (T * k,), torch.int32).numpy(), sr)
    np.testing.assert_array_equal(run.section("inv_pos", (T * k,), torch.int32).numpy(), inv.reshape(-1))
    # tile list: every expert's rows covered in order by tiles of at most tile_rows
    L = run.layout
    tiles = run.section("tiles", (4 + 4 * L.max_tiles,), torch.int32).numpy()
    n = tiles[0]
    td = tiles[4:4 + 4 * n].reshape(n, 4)
    want = []
    for e in range(E):
        for r0 in range(0, cnt[e], L.tile_rows):
            want.append((e, off[e] + r0, min(L.tile_rows, cnt[e] - r0)))
    assert [tuple(r[:3]) for r in td] == want
    return cnt, off, sr, inv


def compare_out(got: np.ndarray, want: np.ndarray, what="", allow=None, bf16_rounding=False):
    """Layer tolerances: max |d| <= 2e-2 * rms(ref) and relative Frobenius <= 5e-3.

    ``allow`` [T] adds, per token, the exact bound of validated MXFP8 near-midpoint
    flips of the intermediate (see check_intermediate).  ``bf16_rounding`` adds, per
    element, the largest error of rounding the reference to the bf16 output format
    with round-to-nearest-even (half a bf16 step, at most 2^-9 |ref|); used for the
    small edge-case shapes whose few outputs can sit many rms above the mean,
    where that rounding alone can exceed 2e-2 * rms."""
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    d = got - want
    rms = float(np.sqrt(np.mean(want ** 2)))
    rel = float(np.linalg.norm(d) / np.linalg.norm(want))
    lim = np.full(want.shape, MAX_ABS_OVER_RMS * rms)
    if allow is not None:
        lim += np.asarray(allow)[:, None]
    if bf16_rounding:
        lim += 2.0 ** -9 * np.abs(want)
    over = np.abs(d) > lim
    per_tok = np.abs(d).max(axis=1)
    if over.any():
        t, c = np.argwhere(over)[0]
        raise AssertionError(f"{what}: |d| {abs(d[t, c]):.4g} at token {t} col {c} > limit {lim[t, c]:.4g} "
                             f"(ref {want[t, c]:.4g}, rms {rms:.4g}, rel {rel:.3g})")
    assert rel <= REL_FRO, f"{what}: rel Frobenius {rel:.4g} > {REL_FRO}"
    # a broken FP4 GEMM shows up as rows whose every element is equal
    if got.shape[1] > 1:
        assert (np.ptp(got, axis=1) > 0).all(), f"{what}: constant output row"
    return float(per_tok.max()) / rms, rel


_TABLES = {}


def e4m3_values():
    return _code_table(False)


def _code_table(fp4: bool):
    """Value of every activation code from the oracle's decoders (E2M1 or E4M3)."""
    if fp4 not in _TABLES:
        n, f = (16, oracle.e2m1_value) if fp4 else (256, oracle.e4m3_value)
        _TABLES[fp4] = np.array([f(c) for c in range(n)])
    return _TABLES[fp4]


def gpu_hq(run: GpuForward, T: int, inv: np.ndarray):
    """GPU intermediate codes and scale codes per (token, slot): [T,k,I], [T,k,I/32]."""
    I, k = run.dims.I, run.k
    L = run.layout
    TK = run.out.shape[0] * k
    hq = run.codes("hq", TK, I)
    pos = inv.reshape(-1).astype(np.int64)
    sc = run.atom_scales("hq_sf", pos, TK, I, n_blocks=I // run.block)
    return hq[pos].reshape(-1, k, I), sc.reshape(-1, k, I // run.block)


def check_intermediate(run: GpuForward, ref: dict, inp_cpu: ms.LayerInputs, inv: np.ndarray, tokens=None,
                       rel_mid=2e-4):
    """Compare the GPU's MXFP8 intermediate with the oracle's for every (token, slot).

    Codes may differ only where the two codes are neighbours in the format's value
    grid and the oracle's h (fp32) lies within ``rel_mid`` of the rounding midpoint
    between them (or the block amax within ``rel_mid`` of the power of two where
    the shared exponent changes): both codes are then correct results of the same
    quantisation, taken from sums accumulated in a different order.  Returns the
    per-token bound such flips put on the output (sum over slots of
    w * sum |delta hq_i| * max_c |Wd[c][i]|) and the flip count."""
    T, k, I = ref["hq"].shape
    e4 = _code_table(run.fp4)
    mag = 0x7 if run.fp4 else 0x7F
    gq, gs = gpu_hq(run, T, inv)
    rq, rs = ref["hq"], ref["hs"]
    B = run.block
    gv = e4[gq] * np.repeat(run.scale_values(gs), B, axis=-1)
    rv = e4[rq] * np.repeat(run.scale_values(rs), B, axis=-1)
    h = ref["h"]
    allow = np.zeros(T)
    flips = 0
    colmax = {}
    for t, j in zip(*np.nonzero((gv != rv).any(axis=-1))):
        e = int(ref["ids"][t, j])
        bad = np.nonzero(gv[t, j] != rv[t, j])[0]
        for blk in np.unique(bad // B):
            sl = slice(B * blk, B * blk + B)
            if gs[t, j, blk] != rs[t, j, blk]:
                amax = np.abs(h[t, j, sl]).max()
                if run.nv:
                    # the E4M3 block scale flips where amax / 6 sits at the midpoint of two scale values
                    mid_s = 0.5 * (e4m3_values()[int(gs[t, j, blk])] + e4m3_values()[int(rs[t, j, blk])])
                    assert abs(amax / 6 - mid_s) <= rel_mid * amax / 6, f"pair {(t, j)} block {blk}: scale differs away from a midpoint"
                else:
                    edge = 2.0 ** np.round(np.log2(amax))
                    assert abs(amax - edge) <= rel_mid * amax, f"pair {(t, j)} block {blk}: scale differs away from a power of two"
            else:
                for i in bad[(bad >= B * blk) & (bad < B * blk + B)]:
                    mid = 0.5 * (gv[t, j, i] + rv[t, j, i])
                    a, b = int(gq[t, j, i]), int(rq[t, j, i])
                    # neighbours: magnitudes one code apart with the same sign, or either side of zero
                    same_sign = (a & ~mag) == (b & ~mag) or (a & mag) == 0 or (b & mag) == 0
                    assert same_sign and abs((a & mag) - (b & mag)) == 1, \
                        f"pair {(t, j)} elem {i}: codes not adjacent ({gv[t, j, i]} vs {rv[t, j, i]})"
                    assert abs(h[t, j, i] - mid) <= rel_mid * abs(h[t, j, i]), \
                        f"pair {(t, j)} elem {i}: h={h[t, j, i]!r} not at the midpoint {mid!r}"
        if e not in colmax:
            wd = oracle.dequant_mxfp4(inp_cpu.down_blocks[e], inp_cpu.down_scales[e])
            if run.nv:  # the NVFP4 weights: the MXFP4 ones re-quantised, within one block-scale unit
                gsd = oracle.nvfp4_global_scale(oracle.mxfp4_amax(inp_cpu.down_blocks, inp_cpu.down_scales))
                wd = oracle.nvfp4_dequant(*oracle.convert_mxfp4_to_nvfp4(inp_cpu.down_blocks[e], inp_cpu.down_scales[e],
                                                                          gsd), gsd)
            colmax[e] = np.abs(wd).max(axis=0)
        allow[t] += ref["w"][t, j] * float((np.abs(gv[t, j] - rv[t, j]) * colmax[e]).sum())
        flips += bad.size
    total = T * k * I
    assert flips <= max(4, 0.002 * total), f"intermediate flips {flips}/{total}"
    return allow, flips


def oracle_tokens_parallel(inp: ms.LayerInputs, tokens, act_format: str = "mxfp8"):
    """The oracle layer on the listed tokens, one single-threaded oracle call per
    token on every host core (its calls release the interpreter lock); the
    results stacked as one call would return them (with intermediates)."""
    w = (inp.gate_up_blocks, inp.gate_up_scales, inp.gate_up_bias, inp.down_blocks, inp.down_scales,
         inp.down_bias)

    def one(t):
        return oracle.moe_forward(inp.x[t:t + 1], inp.router_w, inp.router_b, *w, k=inp.shape.k,
                                  intermediates=True, act_format=act_format)

    with cf.ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as ex:
        refs = list(ex.map(one, tokens))
    return {key: np.concatenate([r[key] for r in refs], axis=0) for key in refs[0]}
