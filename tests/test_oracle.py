"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test ties one oracle routine to something independent of it: values the
MXFP4 page prints (tests/golden), a library routine (torch's float8_e4m3fn
cast, numpy matmul / stable argsort, scipy softmax / expit), a closed form
worked out by hand, or brute force on tiny inputs.
"""
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                a, b = line.split()
                rows.append((int(a), float(b)))
    return rows


def _bf16_bits(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# --- number formats ------------------------------------------------------------------------
def test_e2m1_codes_match_page_value_set():
    table = dict(_golden("e2m1_values.txt"))
    for code in range(16):
        v = oracle.e2m1_value(code)
        assert v == table[code] and math.copysign(1, v) == math.copysign(1, table[code])
    page_set = {0.0, 0.5, -0.5, 1.0, -1.0, 1.5, -1.5, 2.0, -2.0, 3.0, -3.0, 4.0, -4.0, 6.0, -6.0}
    assert {oracle.e2m1_value(c) for c in range(16)} == page_set


def test_all_256_bytes_decode_low_nibble_first():
    table = dict(_golden("e2m1_values.txt"))
    # 16 rows x one 32-element block; row r holds bytes 16r .. 16r+15, scale 127 (x1)
    blocks = np.arange(256, dtype=np.uint8).reshape(16, 1, 16)
    scales = np.full((16, 1), 127, np.uint8)
    W = oracle.dequant_mxfp4(blocks, scales)
    for byte in range(256):
        r, j = divmod(byte, 16)
        assert W[r, 2 * j] == table[byte & 0xF]
        assert W[r, 2 * j + 1] == table[byte >> 4]


def test_e8m0_scale_matches_page():
    for code, value in _golden("e8m0_scale.txt"):
        v = oracle.e8m0_value(code)
        if math.isnan(value):
            assert math.isnan(v)
        else:
            assert v == value


def test_dequant_applies_block_scale_per_32_elements():
    # byte 0x22 = two elements of code 2 (1.0); block b gets scale 120 + b
    blocks = np.full((2, 3, 16), 0x22, np.uint8)
    scales = np.array([[120, 121, 122], [127, 130, 0]], np.uint8)
    W = oracle.dequant_mxfp4(blocks, scales)
    for r in range(2):
        for c in range(96):
            assert W[r, c] == 2.0 ** (int(scales[r, c // 32]) - 127)


def test_e4m3_decode_matches_torch_float8_e4m3fn():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = oracle.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c], c
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_cast_on_float32_values():
    rng = np.random.default_rng(1)
    mags = np.exp(rng.uniform(math.log(2.0 ** -12), math.log(460.0), 20000))
    v = (mags * rng.choice([-1.0, 1.0], mags.size)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(a)) for a in v], np.uint8)
    np.testing.assert_array_equal(got, ref)


def test_e4m3_encode_midpoints_ties_to_even_and_saturates():
    finite = [c for c in range(0x7F)]  # positive codes, increasing values
    vals = [oracle.e4m3_value(c) for c in finite]
    assert all(a < b for a, b in zip(vals, vals[1:]))
    for c in range(len(vals) - 1):
        mid = 0.5 * (vals[c] + vals[c + 1])
        want = c if c % 2 == 0 else c + 1  # even mantissa code wins the tie
        assert oracle.e4m3_encode(mid) == want
        assert oracle.e4m3_encode(-mid) == 0x80 | want
        assert oracle.e4m3_encode(vals[c]) == c
    for big in (448.0, 449.0, 464.0, 1e6, float("inf")):
        assert oracle.e4m3_encode(big) == 0x7E
        assert oracle.e4m3_encode(-big) == 0xFE


def test_bf16_round_matches_torch_and_ties_to_even():
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(5000) * np.exp(rng.uniform(-20, 20, 5000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_round(float(a)) for a in v], np.uint16)
    np.testing.assert_array_equal(got, ref)
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to the even significand (1.0)
    assert oracle.bf16_round(1.0 + 2.0 ** -8) == 0x3F80
    assert oracle.bf16_round(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # just above the midpoint rounds up (a double a float32 cast would flatten)
    assert oracle.bf16_round(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81


# --- MXFP8 block quantisation ---------------------------------------------------------------
def test_mxfp8_hand_examples():
    # block of all 1.0: amax 1 = 2^0 -> shared exponent 0 - 8 = -8 (code 119);
    # 1.0 / 2^-8 = 256 = 2^8 -> E4M3 exponent field 8+7 = 15, mantissa 0 -> 0x78
    q, s = oracle.mxfp8_quantize(np.ones(32))
    assert s[0] == 119 and (q == 0x78).all()
    # amax 3 -> exponent 1 - 8 = -7 (code 120); 3 * 128 = 384 = 1.5 * 2^8 -> 0x7C;
    # 0.5 * 128 = 64 = 2^6 -> 0x68; -1 * 128 = -128 -> 0xF0
    v = np.zeros(32)
    v[0], v[1], v[2] = 3.0, 0.5, -1.0
    q, s = oracle.mxfp8_quantize(v)
    assert s[0] == 120 and q[0] == 0x7C and q[1] == 0x68 and q[2] == 0xF0 and q[3] == 0
    # amax just under 2: 1.999 * 256 = 511.7 exceeds 448 and saturates (the clamp case)
    v = np.full(32, 1.999)
    q, s = oracle.mxfp8_quantize(v)
    assert s[0] == 119 and (q == 0x7E).all()
    # all-zero block -> smallest scale code, zero elements
    q, s = oracle.mxfp8_quantize(np.zeros(32))
    assert s[0] == 0 and (q == 0).all()


def _mx_values(q, s):
    e4 = np.array([oracle.e4m3_value(c) for c in range(256)])
    return e4[q] * np.ldexp(1.0, s.astype(np.int64) - 127).repeat(32, axis=-1)


def test_mxfp8_elements_match_torch_cast_and_are_idempotent():
    rng = np.random.default_rng(3)
    v = rng.standard_normal((64, 32)) * np.exp(rng.uniform(-6, 6, (64, 1)))
    v = v.astype(np.float32).astype(np.float64)
    q, s = oracle.mxfp8_quantize(v)
    scale = np.ldexp(1.0, s.astype(np.int64) - 127)  # [64, 1]
    ref = torch.from_numpy(np.clip(v / scale, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(q, ref)
    # the block's largest magnitude lands in the top binade [256, 512) before the clamp
    amax = np.abs(v).max(axis=1)
    assert ((amax / scale[:, 0] >= 256) & (amax / scale[:, 0] < 512)).all()
    q2, s2 = oracle.mxfp8_quantize(_mx_values(q, s))
    np.testing.assert_array_equal(q2, q)
    np.testing.assert_array_equal(s2, s)


# --- MXFP4 activations (the FP4 x FP4 variant) ----------------------------------------------
def test_e2m1_encode_round_trips_the_page_value_set():
    for code, value in _golden("e2m1_values.txt"):
        assert oracle.e2m1_encode(value) == code


def test_e2m1_encode_midpoints_tie_to_even_mantissa_and_saturate():
    # midpoints between neighbouring magnitudes go to the code whose mantissa bit
    # (bit 0) is clear: 0 (0), 1.0 (2), 2.0 (4), 4.0 (6)
    for v, code in [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6)]:
        assert oracle.e2m1_encode(v) == code, v
        assert oracle.e2m1_encode(-v) == code | 8, -v
    # just off a midpoint: the nearer magnitude
    for v, code in [(0.26, 1), (0.74, 1), (1.26, 3), (2.51, 5), (5.01, 7), (4.99, 6)]:
        assert oracle.e2m1_encode(v) == code, v
    # beyond the largest magnitude: saturate to 6; a tiny negative keeps its sign
    for v in (6.0, 6.5, 7.99, 1e30, math.inf):
        assert oracle.e2m1_encode(v) == 7 and oracle.e2m1_encode(-v) == 15
    assert oracle.e2m1_encode(-1e-30) == 8


def test_e2m1_encode_is_the_nearest_page_value_off_midpoints():
    mags = np.array(sorted({abs(v) for _, v in _golden("e2m1_values.txt")}))
    codes = {abs(v): c for c, v in _golden("e2m1_values.txt") if c < 8}
    rng = np.random.default_rng(11)
    v = rng.uniform(-7.5, 7.5, 4000)
    mids = (mags[1:] + mags[:-1]) / 2
    v = v[np.abs(np.abs(v)[:, None] - mids[None, :]).min(axis=1) > 1e-6]
    for x in v:
        m = mags[np.abs(mags - min(abs(x), 6.0)).argmin()]
        assert oracle.e2m1_encode(x) == codes[m] | (8 if x < 0 else 0), x


def _mx4_values(q, s):
    e2 = np.array([oracle.e2m1_value(c) for c in range(16)])
    return e2[q] * np.ldexp(1.0, s.astype(np.int64) - 127).repeat(32, axis=-1)


def test_mxfp4_hand_examples():
    # amax 6 = 1.5 * 2^2 -> shared exponent 2 - 2 = 0 (code 127); 6 -> code 7, -1.5 -> 11
    v = np.zeros(32)
    v[0], v[1] = 6.0, -1.5
    q, s = oracle.mxfp4_quantize(v)
    assert s[0] == 127 and q[0] == 7 and q[1] == 11 and (q[2:] == 0).all()
    # amax 12 -> exponent 3 - 2 = 1 (code 128): 12 / 2 = 6 -> 7; 5 / 2 = 2.5 ties to 2.0 -> 4
    v[0], v[1] = 12.0, 5.0
    q, s = oracle.mxfp4_quantize(v)
    assert s[0] == 128 and q[0] == 7 and q[1] == 4
    # amax 0.75 -> exponent -1 - 2 = -3 (code 124): 0.75 * 8 = 6 -> 7
    q, s = oracle.mxfp4_quantize(np.full(32, 0.75))
    assert s[0] == 124 and (q == 7).all()
    # amax 7 -> exponent 0: 7 exceeds 6 and saturates (the clamp case)
    q, s = oracle.mxfp4_quantize(np.full(32, 7.0))
    assert s[0] == 127 and (q == 7).all()
    # all-zero block -> smallest scale code, zero codes
    q, s = oracle.mxfp4_quantize(np.zeros(32))
    assert s[0] == 0 and (q == 0).all()


def test_mxfp4_block_lands_in_the_top_binade_and_is_idempotent():
    rng = np.random.default_rng(12)
    v = rng.standard_normal((64, 32)) * np.exp(rng.uniform(-6, 6, (64, 1)))
    q, s = oracle.mxfp4_quantize(v)
    scale = np.ldexp(1.0, s.astype(np.int64) - 127)
    amax = np.abs(v).max(axis=1)
    assert ((amax / scale[:, 0] >= 4) & (amax / scale[:, 0] < 8)).all()
    # so the block's largest code is 4 or 6
    top = np.abs(_mx4_values(q, s) / scale.repeat(32, axis=1)).max(axis=1)
    assert set(np.unique(top)) <= {4.0, 6.0}
    q2, s2 = oracle.mxfp4_quantize(_mx4_values(q, s))
    np.testing.assert_array_equal(q2, q)
    np.testing.assert_array_equal(s2, s)


def test_fp4_activation_layer_matches_dequantised_dense_path():
    """The layer with x and h quantised to MXFP4, against numpy matmuls on the
    pinned dequantiser, the pinned MXFP4 quantiser and the pinned router."""
    rng = np.random.default_rng(13)
    T, H, I, E, k = 5, 64, 64, 4, 2
    x, wr, br = _tiny_router(T, H, E, seed=14)
    ex = [_rand_expert(H, I, rng) for _ in range(E)]
    gub, gus, gubias, db, ds, dbias = (np.stack([e[i] for e in ex]) for i in range(6))
    r = oracle.moe_forward(x, wr, br, gub, gus, gubias, db, ds, dbias, k=k, intermediates=True,
                           act_format="mxfp4")
    _, ids, w = oracle.route(x, wr, br, k)
    np.testing.assert_array_equal(r["ids"], ids)
    xq, xs = oracle.mxfp4_quantize(_widen(x))
    np.testing.assert_array_equal(r["xq"], xq)
    np.testing.assert_array_equal(r["xs"], xs)
    out = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            g = oracle.dequant_mxfp4(gub[e], gus[e]) @ _mx4_values(xq[t], xs[t]) + _widen(gubias[e])
            h = (g[:I] * scipy.special.expit(g[:I]) * g[I:]).astype(np.float32).astype(np.float64)
            np.testing.assert_allclose(r["h"][t, j], h, rtol=1e-6, atol=1e-30)
            hq, hs = oracle.mxfp4_quantize(r["h"][t, j])
            np.testing.assert_array_equal(r["hq"][t, j], hq)
            y = oracle.dequant_mxfp4(db[e], ds[e]) @ _mx4_values(hq, hs) + _widen(dbias[e])
            out[t] += w[t, j] * y
    np.testing.assert_allclose(r["out"], out, rtol=1e-12, atol=1e-12 * np.abs(out).max())
    # and the MXFP8 layer is unchanged by the format switch
    r8 = oracle.moe_forward(x, wr, br, gub, gus, gubias, db, ds, dbias, k=k)
    r8b = oracle.moe_forward(x, wr, br, gub, gus, gubias, db, ds, dbias, k=k, act_format="mxfp8")
    np.testing.assert_array_equal(r8["out"], r8b["out"])
    assert np.abs(r8["out"] - r["out"]).max() > 0


# --- routing -------------------------------------------------------------------------------
def _tiny_router(T=16, H=64, E=8, seed=5):
    rng = np.random.default_rng(seed)
    x = _bf16_bits(rng.standard_normal((T, H)))
    wr = _bf16_bits(rng.standard_normal((E, H)) / math.sqrt(H))
    br = _bf16_bits(rng.standard_normal(E) * 0.01)
    return x, wr, br


def _widen(bits):
    return bits.astype(np.uint32).__lshift__(16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("k", [1, 2, 4])
def test_route_against_numpy(k):
    x, wr, br = _tiny_router()
    logits, ids, w = oracle.route(x, wr, br, k)
    ref_logits = _widen(x) @ _widen(wr).T + _widen(br)
    np.testing.assert_allclose(logits, ref_logits, rtol=1e-12, atol=1e-12)
    l32 = ref_logits.astype(np.float32)
    for t in range(x.shape[0]):
        order = np.lexsort((np.arange(l32.shape[1]), -l32[t]))  # logit desc, index asc
        np.testing.assert_array_equal(ids[t], order[:k])
        ref_w = scipy.special.softmax(ref_logits[t, order[:k]])
        np.testing.assert_allclose(w[t], ref_w, rtol=1e-13, atol=0)
        assert abs(w[t].sum() - 1.0) <= 1e-12
    if k == 1:
        assert (w == 1.0).all()


def test_route_ties_go_to_lower_expert():
    H, E = 32, 6
    x = _bf16_bits(np.ones((1, H)))
    wr = _bf16_bits(np.zeros((E, H)))
    br = _bf16_bits(np.array([0.0, 2.0, 1.0, 2.0, 1.0, 2.0]))
    _, ids, w = oracle.route(x, wr, br, 4)
    assert ids[0].tolist() == [1, 3, 5, 2]
    # softmax of [2, 2, 2, 1]: 1/(3 + e^-1) for the tied top three
    top = 1.0 / (3.0 + math.exp(-1.0))
    np.testing.assert_allclose(w[0], [top, top, top, math.exp(-1.0) * top], rtol=1e-15)


# --- permutation ---------------------------------------------------------------------------
@pytest.mark.parametrize("T,k,E", [(1, 1, 4), (7, 2, 8), (64, 4, 128), (3, 4, 4)])
def test_permute_against_numpy_stable_argsort(T, k, E):
    rng = np.random.default_rng(T * 131 + k)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    cnt, off, sr, inv = oracle.permute(ids, E)
    flat = ids.reshape(-1)
    np.testing.assert_array_equal(cnt, np.bincount(flat, minlength=E))
    assert off[0] == 0 and off[E] == T * k
    np.testing.assert_array_equal(np.diff(off), cnt)
    np.testing.assert_array_equal(sr, np.argsort(flat, kind="stable"))
    np.testing.assert_array_equal(sr[inv.reshape(-1)], np.arange(T * k))


# --- expert MLP ----------------------------------------------------------------------------
def _rand_expert(H, I, rng):
    gub = rng.integers(0, 256, (2 * I, H // 32, 16), dtype=np.uint8)
    gus = rng.integers(118, 125, (2 * I, H // 32), dtype=np.uint8)
    gubias = _bf16_bits(rng.standard_normal(2 * I) * 0.02)
    db = rng.integers(0, 256, (H, I // 32, 16), dtype=np.uint8)
    ds = rng.integers(118, 125, (H, I // 32), dtype=np.uint8)
    dbias = _bf16_bits(rng.standard_normal(H) * 0.02)
    return gub, gus, gubias, db, ds, dbias


def test_expert_mlp_matches_dequantised_dense_path():
    rng = np.random.default_rng(7)
    H, I = 96, 64
    gub, gus, gubias, db, ds, dbias = _rand_expert(H, I, rng)
    x = _widen(_bf16_bits(rng.standard_normal(H)))
    xq, xs = oracle.mxfp8_quantize(x)
    r = oracle.expert_mlp(xq, xs, gub, gus, gubias, db, ds, dbias)
    xv = _mx_values(xq, xs)
    g_ref = oracle.dequant_mxfp4(gub, gus) @ xv + _widen(gubias)
    np.testing.assert_allclose(r["g"], g_ref, rtol=1e-12, atol=1e-12 * np.abs(g_ref).max())
    gate, up = g_ref[:I], g_ref[I:]
    h_ref = gate * scipy.special.expit(gate) * up
    np.testing.assert_allclose(r["h"], h_ref.astype(np.float32), rtol=1e-6, atol=0)
    hq, hs = oracle.mxfp8_quantize(r["h"])
    np.testing.assert_array_equal(hq, r["hq"])
    np.testing.assert_array_equal(hs, r["hs"])
    y_ref = oracle.dequant_mxfp4(db, ds) @ _mx_values(hq, hs) + _widen(dbias)
    np.testing.assert_allclose(r["y"], y_ref, rtol=1e-12, atol=1e-12 * np.abs(y_ref).max())


def test_silu_matches_scipy():
    for z in np.linspace(-30, 30, 241):
        assert abs(oracle.silu(z) - z * scipy.special.expit(z)) <= 1e-15 * max(1.0, abs(z))


def _closed_form_layer():
    """H = I = 32, E = 2, k = 1.  Worked by hand:

    x = all ones (bf16) -> MXFP8 scale code 119, element 0x78, value exactly 1.
    router: Wr = 0, br = [0, 1] -> expert 1 chosen with weight 1.
    expert 1 gate rows: byte 0x22 (two codes 2 = 1.0), scale 127 -> W = 1 -> g = 32 + 0.25
    expert 1 up rows:   byte 0x11 (code 1 = 0.5), scale 128 (x2) -> W = 1 -> g = 32 - 0.25
      (biases 0.25 and -0.25)
    h = silu(32.25) * 31.75; e^-32.25 < 2^-46, so in fp32 h = 32.25 * 31.75 = 1023.9375
    MXFP8 of h: amax 1023.9375 in [2^9, 2^10) -> exponent 9 - 8 = 1 (code 128);
      1023.9375 / 2 = 511.97 > 448 -> saturates to 448 -> value 896.
    down row c: byte 0xAA (code 10 = -1.0), scale 120 + (c % 3) -> W = -2^(c%3 - 7);
      y_c = 32 * 896 * -2^(c%3 - 7) + bd_c = -224 * 2^(c%3) + 0.5
    out = 1 * y.
    """
    H = I = 32
    E = 2
    x = _bf16_bits(np.ones((1, H)))
    wr = _bf16_bits(np.zeros((E, H)))
    br = _bf16_bits(np.array([0.0, 1.0]))
    gub = np.zeros((E, 2 * I, 1, 16), np.uint8)
    gus = np.full((E, 2 * I, 1), 127, np.uint8)
    gubias = np.zeros((E, 2 * I), np.uint16)
    db = np.zeros((E, H, 1, 16), np.uint8)
    ds = np.full((E, H, 1), 127, np.uint8)
    dbias = np.zeros((E, H), np.uint16)
    gub[1, :I] = 0x22
    gub[1, I:] = 0x11
    gus[1, I:] = 128
    gubias[1, :I] = _bf16_bits([0.25] * I)
    gubias[1, I:] = _bf16_bits([-0.25] * I)
    db[1] = 0xAA
    ds[1, :, 0] = [120 + (c % 3) for c in range(H)]
    dbias[1] = _bf16_bits([0.5] * H)
    # expert 0 holds a different layer entirely (must not be used)
    gub[0] = 0x77
    db[0] = 0x77
    expected = np.array([-224.0 * 2 ** (c % 3) + 0.5 for c in range(H)])
    return (x, wr, br, gub, gus, gubias, db, ds, dbias), expected


def test_layer_closed_form():
    args, expected = _closed_form_layer()
    r = oracle.moe_forward(*args, k=1)
    assert r["ids"][0, 0] == 1 and r["w"][0, 0] == 1.0
    np.testing.assert_array_equal(r["out"][0], expected)


def test_zero_gate_gives_down_bias():
    rng = np.random.default_rng(11)
    H, I = 64, 64
    gub, gus, gubias, db, ds, dbias = _rand_expert(H, I, rng)
    gub[:I] = 0                      # every gate weight is +0
    gubias[:I] = 0                   # and so is the gate bias -> silu(0) = 0 -> h = 0
    x = _widen(_bf16_bits(rng.standard_normal(H)))
    xq, xs = oracle.mxfp8_quantize(x)
    r = oracle.expert_mlp(xq, xs, gub, gus, gubias, db, ds, dbias)
    assert (r["h"] == 0).all()
    np.testing.assert_array_equal(r["y"], _widen(dbias))


def test_layer_equals_brute_force_over_all_experts():
    rng = np.random.default_rng(13)
    T, H, I, E, k = 6, 64, 32, 4, 2
    x, wr, br = _tiny_router(T, H, E, seed=17)
    experts = [_rand_expert(H, I, rng) for _ in range(E)]
    stack = [np.stack([ex[i] for ex in experts]) for i in range(6)]
    r = oracle.moe_forward(x, wr, br, *stack, k=k)
    logits = _widen(x) @ _widen(wr).T + _widen(br)
    for t in range(T):
        xq, xs = oracle.mxfp8_quantize(_widen(x[t]))
        np.testing.assert_array_equal(xq, r["xq"][t])
        np.testing.assert_array_equal(xs, r["xs"][t])
        ys = np.stack([oracle.expert_mlp(xq, xs, *experts[e])["y"] for e in range(E)])
        order = np.lexsort((np.arange(E), -logits[t].astype(np.float32)))[:k]
        w = scipy.special.softmax(logits[t, order])
        ref = (w[:, None] * ys[order]).sum(0)
        np.testing.assert_allclose(r["out"][t], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_rmsnorm_closed_form():
    x = np.full((2, 64), 3.0)
    x[1] = -0.5
    out = oracle.rmsnorm_bf16(x, 1e-5)
    for t, c in enumerate([3.0, -0.5]):
        want = oracle.bf16_round(c / math.sqrt(c * c + 1e-5))
        assert (out[t] == want).all()


# ----------------------------------------------------------------------- dense MXFP4 linears
def _e2m1_table():
    return np.array([v for _, v in sorted(_golden("e2m1_values.txt"))])


def test_pack_e2m1_round_trips_through_the_dequantiser():
    """Codes packed into the checkpoint blocks decode (by the pinned dequantiser) to the
    page's value of each code times its block scale, element by element."""
    rng = np.random.default_rng(5)
    rows, K = 6, 96
    codes = rng.integers(0, 16, (rows, K)).astype(np.uint8)
    scales = rng.integers(118, 131, (rows, K // 32)).astype(np.uint8)
    W = oracle.dequant_mxfp4(oracle.pack_e2m1(codes), scales)
    want = _e2m1_table()[codes] * np.exp2(np.repeat(scales.astype(np.int64), 32, axis=1) - 127.0)
    np.testing.assert_array_equal(W, want)


def test_quantize_mxfp4_weights_hand_block_and_idempotence():
    """A hand-worked block (amax 6 -> shared exponent 0, codes from the page's table),
    idempotence on values the format holds, and the error bound of the top binade:
    at most 2^(s+1) per element (the 4..6 gap halved, or saturation from below 8)."""
    blk = np.zeros((1, 32))
    blk[0, :6] = [6.0, 3.0, -1.5, 0.5, 0.25, 0.75]
    b, s = oracle.quantize_mxfp4_weights(blk)
    assert s[0, 0] == 127
    by = b[0, 0]
    lo = by[0] & 0xF, by[0] >> 4, by[1] & 0xF, by[1] >> 4, by[2] & 0xF, by[2] >> 4
    assert lo == (7, 5, 11, 1, 0, 2)  # 0.25 and 0.75 are midpoints: ties go to the even code
    rng = np.random.default_rng(6)
    W = rng.normal(0, 0.3, (8, 128))
    b1, s1 = oracle.quantize_mxfp4_weights(W)
    W1 = oracle.dequant_mxfp4(b1, s1)
    b2, s2 = oracle.quantize_mxfp4_weights(W1)
    np.testing.assert_array_equal(b1, b2)
    np.testing.assert_array_equal(s1, s2)
    step = np.exp2(np.repeat(s1.astype(np.int64), 32, axis=1) - 127.0 + 1)
    assert (np.abs(W - W1) <= step).all()


@pytest.mark.parametrize("act_format", ["mxfp8", "mxfp4"])
def test_dense_linear_matches_dequantised_matmul(act_format):
    """The dense linear against numpy: the pinned activation quantiser and weight
    dequantiser, then a library matmul and the bias."""
    rng = np.random.default_rng(7)
    T, K, N = 3, 96, 40
    x = torch.from_numpy(rng.normal(0, 1, (T, K))).to(torch.bfloat16)
    b, s = oracle.quantize_mxfp4_weights(rng.normal(0, 0.2, (N, K)))
    bias = torch.from_numpy(rng.normal(0, 0.1, N)).to(torch.bfloat16)
    got = oracle.dense_linear(x, b, s, bias, act_format=act_format)
    xf = x.float().double().numpy()
    if act_format == "mxfp8":
        q, qs = oracle.mxfp8_quantize(xf)
        xv = np.array([oracle.e4m3_value(c) for c in range(256)])[q]
    else:
        q, qs = oracle.mxfp4_quantize(xf)
        xv = _e2m1_table()[q]
    xv = xv * np.exp2(np.repeat(qs.astype(np.int64), 32, axis=1) - 127.0)
    want = xv @ oracle.dequant_mxfp4(b, s).T + bias.float().double().numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    assert np.allclose(oracle.dense_linear(x, b, s, None, act_format=act_format), want - bias.float().double().numpy(),
                       rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------- NVFP4
def test_nvfp4_global_scale_closed_form():
    # amax / (6 * 448): a tensor whose amax is 6 * 448 needs no global scaling
    assert oracle.nvfp4_global_scale(2688.0) == 1.0
    assert oracle.nvfp4_global_scale(5376.0) == 2.0
    assert oracle.nvfp4_global_scale(0.0) == 1.0
    assert oracle.nvfp4_global_scale(1.0) == float(np.float32(1.0) / np.float32(2688.0))


def test_nvfp4_hand_blocks():
    """Scale = E4M3(amax / 6); elements E2M1(v / scale), ties to even, saturating at 6."""
    v = np.zeros(16)
    v[:7] = [6.0, -3.0, 1.5, 0.25, 0.75, 2.5, 5.0]
    q, s = oracle.nvfp4_quantize(v)
    assert s[0] == 0x38  # E4M3 1.0
    assert tuple(q[:7]) == (7, 13, 3, 0, 2, 4, 6)  # 0.25->0, 0.75->1.0, 2.5->2, 5->4 (ties to even)
    v2 = np.zeros(16)
    v2[0] = 7.0  # 7/6 = 1.1667 rounds to E4M3 1.125; 7/1.125 = 6.2 saturates to 6
    q, s = oracle.nvfp4_quantize(v2)
    assert oracle.e4m3_value(int(s[0])) == 1.125 and q[0] == 7
    q, s = oracle.nvfp4_quantize(np.zeros(16))  # an all-zero block: zero scale, zero codes
    assert s[0] == 0 and (q == 0).all()
    # a global scale divides the block scale's argument
    q, s = oracle.nvfp4_quantize(v * 4.0, gs=4.0)
    assert s[0] == 0x38 and tuple(q[:7]) == (7, 13, 3, 0, 2, 4, 6)


def test_nvfp4_scale_matches_torch_cast_and_error_bound():
    """The block scale code is torch's float8_e4m3fn cast of the fp32 amax / (6 gs)
    (a library routine), and every element lies within one scale unit of its value
    (the largest E2M1 gap, 4..6, halved; or saturation from at most 6 (1 + 1/16))."""
    rng = np.random.default_rng(8)
    v = rng.normal(0, 2.0, (32, 64)) * np.exp2(rng.integers(-6, 6, (32, 1)))
    gs = oracle.nvfp4_global_scale(np.abs(v).max())
    q, s = oracle.nvfp4_quantize(v, gs)
    amax = np.abs(v).reshape(32, 4, 16).max(axis=2)
    t = torch.from_numpy(amax.astype(np.float32)) / torch.tensor(6.0 * np.float32(gs), dtype=torch.float32)
    want = t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(s, want)
    deq = oracle.nvfp4_dequant(q, s, gs)
    sv = np.repeat(np.array([oracle.e4m3_value(c) for c in range(256)])[s], 16, axis=1) * gs
    assert (np.abs(v - deq) <= sv * (1 + 1e-12)).all()


def test_expert_mlp_nvfp4_matches_dequantised_dense_path():
    """One expert with NVFP4 weights and activations against numpy: dequantised
    operands, library matmuls, scipy's expit for the SiLU; the intermediate is
    quantised by the pinned NVFP4 quantiser."""
    rng = np.random.default_rng(9)
    H, I = 64, 32
    x = rng.normal(0, 1, H)
    xq, xs = oracle.nvfp4_quantize(x)
    wgu = rng.normal(0, 0.2, (2 * I, H))
    wd = rng.normal(0, 0.2, (H, I))
    gsg = oracle.nvfp4_global_scale(np.abs(wgu).max())
    gsd = oracle.nvfp4_global_scale(np.abs(wd).max())
    guq, gus = oracle.nvfp4_quantize(wgu, gsg)
    dq, dsc = oracle.nvfp4_quantize(wd, gsd)
    gub = torch.from_numpy(rng.normal(0, 0.02, 2 * I)).to(torch.bfloat16)
    db = torch.from_numpy(rng.normal(0, 0.02, H)).to(torch.bfloat16)
    r = oracle.expert_mlp_nvfp4(xq, xs, guq, gus, gsg, gub, dq, dsc, gsd, db)
    g = oracle.nvfp4_dequant(xq, xs, 1.0) @ oracle.nvfp4_dequant(guq, gus, gsg).T + gub.float().double().numpy()
    h = (g[:I] * scipy.special.expit(g[:I]) * g[I:]).astype(np.float32).astype(np.float64)
    np.testing.assert_allclose(r["h"], h, rtol=1e-6, atol=1e-9)
    hq, hs = oracle.nvfp4_quantize(r["h"])
    np.testing.assert_array_equal(r["hq"], hq)
    y = oracle.nvfp4_dequant(hq, hs, 1.0) @ oracle.nvfp4_dequant(dq, dsc, gsd).T + db.float().double().numpy()
    np.testing.assert_allclose(r["y"], y, rtol=1e-12, atol=1e-12)


def test_nvfp4_layer_matches_its_steps_and_brute_force():
    """The NVFP4 layer against its pinned steps composed in numpy: the conversion
    of every used expert (dequantise MXFP4, global scale from the projection's
    amax over all experts, NVFP4 quantisation), the NVFP4 expert MLP, and the
    routing-weighted sum; and the projections' amax against a dense dequantisation."""
    import moe_synth as ms
    shape = ms.LayerShape(T=5, H=64, I=64, E=4, k=2)
    inp = ms.make_layer(shape, seed=12)
    w = (inp.gate_up_blocks, inp.gate_up_scales, inp.gate_up_bias, inp.down_blocks, inp.down_scales, inp.down_bias)
    r = oracle.moe_forward(inp.x, inp.router_w, inp.router_b, *w, k=2, intermediates=True, act_format="nvfp4")
    amax_gu = np.abs(oracle.dequant_mxfp4(inp.gate_up_blocks.reshape(-1, 2, 16), inp.gate_up_scales.reshape(-1, 2))).max()
    assert oracle.mxfp4_amax(inp.gate_up_blocks, inp.gate_up_scales) == amax_gu
    gs_gu = oracle.nvfp4_global_scale(amax_gu)
    gs_d = oracle.nvfp4_global_scale(oracle.mxfp4_amax(inp.down_blocks, inp.down_scales))
    _, ids, wts = oracle.route(inp.x, inp.router_w, inp.router_b, 2)
    np.testing.assert_array_equal(r["ids"], ids)
    want = np.zeros((5, 64))
    for t in range(5):
        xq, xs = oracle.nvfp4_quantize(inp.x[t].float().double().numpy())
        np.testing.assert_array_equal(r["xq"][t], xq)
        for j in range(2):
            e = int(ids[t, j])
            gc, gsc = oracle.convert_mxfp4_to_nvfp4(inp.gate_up_blocks[e], inp.gate_up_scales[e], gs_gu)
            q2, s2 = oracle.nvfp4_quantize(oracle.dequant_mxfp4(inp.gate_up_blocks[e], inp.gate_up_scales[e]), gs_gu)
            np.testing.assert_array_equal(gc, q2)
            np.testing.assert_array_equal(gsc, s2)
            dc, dsc = oracle.convert_mxfp4_to_nvfp4(inp.down_blocks[e], inp.down_scales[e], gs_d)
            m = oracle.expert_mlp_nvfp4(xq, xs, gc, gsc, gs_gu, inp.gate_up_bias[e], dc, dsc, gs_d, inp.down_bias[e])
            np.testing.assert_array_equal(r["hq"][t, j], m["hq"])
            want[t] += wts[t, j] * m["y"]
    np.testing.assert_allclose(r["out"], want, rtol=1e-12, atol=1e-12)
