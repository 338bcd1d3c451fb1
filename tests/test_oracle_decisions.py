"""The oracle takes two decisions in fp32, the precision the kernels decide in:
the top-k order compares logits rounded to fp32, and the intermediate h is rounded
to fp32 before its MXFP8 quantisation.  The plain definition decides both in fp64.
These pins show that the two readings part only where the fp64 values straddle
one fp32 rounding step, and never elsewhere:

* routing: experts whose fp64 logits differ but round to the same fp32 value may
  swap places (lower index first); every other position is the same;
* h: an MXFP8 code can differ only where rounding h to fp32 moves it onto or
  across an E4M3 rounding midpoint of its block (or the block's amax across a
  power of two).
"""
import numpy as np
import pytest

import oracle


def _bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bit patterns (through fp32, then round to nearest even): input generator."""
    f = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
    r = ((f + 0x7FFF + ((f >> 16) & 1)) >> 16).astype(np.uint16)
    return r


def _fp64_order(l: np.ndarray, k: int) -> np.ndarray:
    """Top-k by fp64 logit descending, lower index first on exact ties."""
    E = l.shape[-1]
    return np.stack([np.lexsort((np.arange(E), -row))[:k] for row in l]).astype(np.int32)


def test_route_fp32_order_differs_from_fp64_only_at_fp32_ties():
    rng = np.random.default_rng(11)
    T, H, E, k = 96, 64, 16, 4
    base = rng.normal(0, 0.5, (E // 2, H))
    wr = np.repeat(base, 2, axis=0)
    # expert 2i+1 = expert 2i but for one bf16 step in element 0, either direction
    wr_bits = _bf16_bits(wr)
    step = rng.choice([-1, 1], E // 2).astype(np.int32)
    wr_bits[1::2, 0] = (wr_bits[1::2, 0].astype(np.int32) + step).astype(np.uint16)
    br_bits = np.repeat(_bf16_bits(rng.normal(0, 0.1, E // 2)), 2)
    x = rng.normal(0, 1, (T, H))
    x[:, 0] = rng.choice([-1.0, 1.0], T) * 2.0 ** -40  # pair logits differ by ~1e-14: far below one fp32 ulp
    x_bits = _bf16_bits(x)
    logits, ids, _ = oracle.route(x_bits, wr_bits, br_bits, k)
    ids64 = _fp64_order(logits, k)
    l32 = logits.astype(np.float32)
    differ = ids != ids64
    assert differ.any(), "the planted near-ties should reorder some tokens"
    for t, j in zip(*np.nonzero(differ)):
        a, b = ids[t, j], ids64[t, j]
        assert l32[t, a] == l32[t, b] and logits[t, a] != logits[t, b], (t, j, a, b)
        tie = [jj for jj in range(k) if l32[t, ids[t, jj]] == l32[t, a]]
        assert list(ids[t, tie]) == sorted(ids[t, tie]), "an fp32 tie keeps the lower index first"
    # the same selection as a set wherever the k-th and (k+1)-th fp32 logits are distinct
    srt = -np.sort(-l32, axis=1)
    clear = srt[:, k - 1] != srt[:, k]
    assert (np.sort(ids[clear], axis=1) == np.sort(ids64[clear], axis=1)).all()

    # without planted ties the two readings agree everywhere
    wr2 = _bf16_bits(rng.normal(0, 0.5, (E, H)))
    x2 = _bf16_bits(rng.normal(0, 1, (T, H)))
    logits2, ids2, _ = oracle.route(x2, wr2, br_bits, k)
    assert (ids2 == _fp64_order(logits2, k)).all()


def _e4m3_table():
    return np.array([oracle.e4m3_value(c) for c in range(256)])


def test_h_rounding_changes_mxfp8_codes_only_at_midpoints():
    """Planted: one block with amax exactly 1 (shared exponent -8 either way) whose
    other elements sit a hair (2^-30 relative) off an E4M3 rounding midpoint.  Rounding to
    fp32 lands them on the midpoint, where round-half-even decides; fp64 rounds
    toward the hair's side.  Exactly the elements whose two choices differ change."""
    tab = _e4m3_table()
    rng = np.random.default_rng(3)
    pos = np.array(sorted(v for v in set(tab[:0x7F]) if v > 0))  # positive finite E4M3 values
    v = np.zeros(32)
    v[0] = 1.0  # amax: shared exponent floor(log2 1) - 8 = -8
    expect_diff = np.zeros(32, bool)
    scale = 2.0 ** -8
    for i in range(1, 32):
        j = rng.integers(0, len(pos) - 1)
        lo, hi = pos[j], pos[j + 1]
        if hi * scale >= 1.0:
            lo, hi = pos[0], pos[1]
        mid = (lo + hi) / 2 * scale
        hair = rng.choice([-1.0, 1.0]) * mid * 2.0 ** -30  # well inside half an fp32 ulp
        sign = rng.choice([-1.0, 1.0])
        v[i] = sign * (mid + hair)
        assert np.float32(v[i]) == sign * mid  # fp32 lands on the midpoint
        # fp64 rounds toward the hair; the midpoint itself goes to the even code
        away = hi if hair > 0 else lo
        lo_code = int(np.nonzero(tab == lo)[0][0])
        even = lo if lo_code % 2 == 0 else hi
        expect_diff[i] = away != even
    q64, s64 = oracle.mxfp8_quantize(v)
    q32, s32 = oracle.mxfp8_quantize(v.astype(np.float32).astype(np.float64))
    assert s64[0] == s32[0] == 127 - 8
    assert ((q64 != q32) == expect_diff).all()
    assert expect_diff.any() and not expect_diff.all()


def test_oracle_h_is_the_fp32_rounding_of_the_fp64_product_and_codes_follow_it():
    """On a random expert: h equals fp32(silu(g_gate) * g_up) from the oracle's own
    fp64 g, and the codes of fp32(h) and of the fp64 h agree except where an
    E4M3 midpoint (or a power-of-two amax) lies between the two values."""
    rng = np.random.default_rng(5)
    H = I = 64
    gub = rng.integers(0, 256, (2 * I, H // 32, 16), dtype=np.uint8)
    gus = rng.integers(118, 124, (2 * I, H // 32), dtype=np.uint8)
    db = rng.integers(0, 256, (H, I // 32, 16), dtype=np.uint8)
    ds = rng.integers(118, 124, (H, I // 32), dtype=np.uint8)
    gubias = _bf16_bits(rng.normal(0, 0.05, 2 * I))
    dbias = _bf16_bits(rng.normal(0, 0.05, H))
    tab = _e4m3_table()
    checked = 0
    for r in range(24):
        xq, xs = oracle.mxfp8_quantize(rng.normal(0, 1, H))
        o = oracle.expert_mlp(xq, xs, gub, gus, gubias, db, ds, dbias)
        g = o["g"]
        gate, up = g[:I], g[I:]
        h64 = gate / (1.0 + np.exp(-gate)) * up
        h32 = h64.astype(np.float32).astype(np.float64)
        # numpy's exp may differ from the C library's in the last fp64 bit, which can
        # move the fp32 rounding by at most one fp32 step
        assert np.allclose(o["h"], h32, rtol=2.0 ** -23, atol=0)
        assert np.array_equal(o["h"], o["h"].astype(np.float32).astype(np.float64))
        q_or, s_or = oracle.mxfp8_quantize(o["h"])
        assert np.array_equal(q_or, o["hq"]) and np.array_equal(s_or, o["hs"])
        q64, s64 = oracle.mxfp8_quantize(h64)
        for b in range(I // 32):
            blk = slice(32 * b, 32 * b + 32)
            if s64[b] != o["hs"][b]:
                a64, a32 = np.abs(h64[blk]).max(), np.abs(o["h"][blk]).max()
                assert np.floor(np.log2(a64)) != np.floor(np.log2(a32))  # amax crossed a power of two
                continue
            sc = 2.0 ** (int(s64[b]) - 127)
            for i in np.nonzero(q64[blk] != o["hq"][blk])[0]:
                va, vb = tab[q64[blk][i]], tab[o["hq"][blk][i]]
                mid = (va + vb) / 2 * sc
                lo, hi = sorted((h64[blk][i], o["h"][blk][i]))
                assert lo <= mid <= hi, (r, b, i)
            checked += 32
    assert checked == 24 * I
