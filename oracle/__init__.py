"""ctypes binding of the CPU oracle (``moe_oracle.cpp``).

TEST INFRASTRUCTURE ONLY: imported by tests/, the smoke check and the
benchmark's CPU-baseline leg.  The CUDA library never imports this package.

The shared object is compiled from source with the host compiler on first use
(or by the top-level ``build()``), with floating-point contraction off so the
fp64 results are the same on x86-64 and AArch64 hosts.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into a shared object next to its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            d, i32, i64, p = ctypes.c_double, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
            L.oracle_e2m1_value.restype = d
            L.oracle_e2m1_value.argtypes = [ctypes.c_int]
            L.oracle_e8m0_value.restype = d
            L.oracle_e8m0_value.argtypes = [ctypes.c_int]
            L.oracle_e4m3_value.restype = d
            L.oracle_e4m3_value.argtypes = [ctypes.c_int]
            L.oracle_e4m3_encode.restype = ctypes.c_int
            L.oracle_e4m3_encode.argtypes = [d]
            L.oracle_e2m1_encode.restype = ctypes.c_int
            L.oracle_e2m1_encode.argtypes = [d]
            L.oracle_mxfp4_quantize.restype = None
            L.oracle_mxfp4_quantize.argtypes = [p, i64, p, p]
            L.oracle_expert_mlp_fmt.restype = None
            L.oracle_expert_mlp_fmt.argtypes = [p, p, i64, i64, p, p, p, p, p, p, p, p, p, p, p, i32]
            L.oracle_bf16_value.restype = d
            L.oracle_bf16_value.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_round.restype = ctypes.c_uint16
            L.oracle_bf16_round.argtypes = [d]
            L.oracle_silu.restype = d
            L.oracle_silu.argtypes = [d]
            L.oracle_dequant_mxfp4.restype = None
            L.oracle_dequant_mxfp4.argtypes = [p, p, i64, i64, p]
            L.oracle_mxfp8_quantize.restype = None
            L.oracle_mxfp8_quantize.argtypes = [p, i64, p, p]
            L.oracle_route.restype = None
            L.oracle_route.argtypes = [p, p, p, i64, i64, i64, i32, p, p, p]
            L.oracle_permute.restype = None
            L.oracle_permute.argtypes = [p, i64, i32, i32, p, p, p, p]
            L.oracle_expert_mlp.restype = None
            L.oracle_expert_mlp.argtypes = [p, p, i64, i64, p, p, p, p, p, p, p, p, p, p, p]
            L.oracle_moe_forward.restype = None
            L.oracle_moe_forward.argtypes = [p, i64, i64, i64, i64, i32, p, p, p, p, p, p, p, p,
                                             p, p, p, p, p, p, p, p, p]
            L.oracle_moe_forward_fmt.restype = None
            L.oracle_moe_forward_fmt.argtypes = [p, i64, i64, i64, i64, i32, p, p, p, p, p, p, p, p,
                                             p, p, p, p, p, p, p, p, p, i32]
            L.oracle_pack_e2m1.restype = None
            L.oracle_pack_e2m1.argtypes = [p, i64, i64, p]
            L.oracle_quantize_mxfp4_weights.restype = None
            L.oracle_quantize_mxfp4_weights.argtypes = [p, i64, i64, p, p]
            L.oracle_dense_linear.restype = None
            L.oracle_dense_linear.argtypes = [p, i64, i64, i64, p, p, p, p, i32]
            L.oracle_nvfp4_global_scale.restype = d
            L.oracle_nvfp4_global_scale.argtypes = [d]
            L.oracle_nvfp4_quantize.restype = None
            L.oracle_nvfp4_quantize.argtypes = [p, i64, d, p, p]
            L.oracle_nvfp4_value.restype = d
            L.oracle_nvfp4_value.argtypes = [ctypes.c_int, ctypes.c_int, d]
            L.oracle_expert_mlp_nvfp4.restype = None
            L.oracle_expert_mlp_nvfp4.argtypes = [p, p, i64, i64, p, p, d, p, p, p, d, p, p, p, p, p]
            L.oracle_convert_mxfp4_to_nvfp4.restype = None
            L.oracle_convert_mxfp4_to_nvfp4.argtypes = [p, p, i64, i64, d, p, p]
            L.oracle_mxfp4_amax.restype = d
            L.oracle_mxfp4_amax.argtypes = [p, p, i64, i64]
            L.oracle_moe_forward_nvfp4.restype = None
            L.oracle_moe_forward_nvfp4.argtypes = [p, i64, i64, i64, i64, i32, p, p, p, p, p, p, p, p,
                                                   p, p, p, p, p, p, p, p, p]
            L.oracle_rmsnorm_bf16.restype = None
            L.oracle_rmsnorm_bf16.argtypes = [p, i64, i64, d, p]
            _lib = L
    return _lib


def _np(a, dtype):
    """Contiguous numpy view of a CPU torch tensor or array, with the given dtype."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if a.dtype == torch.bfloat16:
                a = a.view(torch.int16)
            a = a.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        a = a.view(dtype) if a.dtype.itemsize == np.dtype(dtype).itemsize else a.astype(dtype)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data


# --- scalar codecs -------------------------------------------------------------------------
def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(code)


def e8m0_value(code: int) -> float:
    return lib().oracle_e8m0_value(code)


def e4m3_value(code: int) -> float:
    return lib().oracle_e4m3_value(code)


def e4m3_encode(v: float) -> int:
    return lib().oracle_e4m3_encode(float(v))


def e2m1_encode(v: float) -> int:
    return lib().oracle_e2m1_encode(float(v))


def bf16_value(bits: int) -> float:
    return lib().oracle_bf16_value(bits)


def bf16_round(v: float) -> int:
    return lib().oracle_bf16_round(float(v))


def silu(z: float) -> float:
    return lib().oracle_silu(float(z))


# --- array routines ------------------------------------------------------------------------
def dequant_mxfp4(blocks, scales) -> np.ndarray:
    """[rows, K/32, 16] uint8 + [rows, K/32] uint8 -> fp64 [rows, K]."""
    b = _np(blocks, np.uint8)
    s = _np(scales, np.uint8)
    rows, nb = s.shape[-2], s.shape[-1]
    W = np.empty((rows, nb * 32), np.float64)
    lib().oracle_dequant_mxfp4(_ptr(b), _ptr(s), rows, nb * 32, _ptr(W))
    return W


def mxfp8_quantize(v):
    """fp64 values (last dim a multiple of 32) -> (e4m3 codes uint8, e8m0 scale codes uint8)."""
    a = _np(v, np.float64)
    q = np.empty(a.shape, np.uint8)
    s = np.empty(a.shape[:-1] + (a.shape[-1] // 32,), np.uint8)
    lib().oracle_mxfp8_quantize(_ptr(a), a.size, _ptr(q), _ptr(s))
    return q, s


def mxfp4_quantize(v):
    """fp64 values (last dim a multiple of 32) -> (e2m1 codes uint8, one per byte; e8m0 scale codes uint8)."""
    a = _np(v, np.float64)
    q = np.empty(a.shape, np.uint8)
    s = np.empty(a.shape[:-1] + (a.shape[-1] // 32,), np.uint8)
    lib().oracle_mxfp4_quantize(_ptr(a), a.size, _ptr(q), _ptr(s))
    return q, s


_ACT = {"mxfp8": 0, "mxfp4": 1}


def route(x, router_w, router_b, k: int):
    """-> (logits fp64 [T,E], ids int32 [T,k], w fp64 [T,k])."""
    xx = _np(x, np.uint16)
    wr = _np(router_w, np.uint16)
    br = _np(router_b, np.uint16)
    T, H = xx.shape
    E = wr.shape[0]
    logits = np.empty((T, E), np.float64)
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    lib().oracle_route(_ptr(xx), _ptr(wr), _ptr(br), T, H, E, k, _ptr(logits), _ptr(ids), _ptr(w))
    return logits, ids, w


def permute(ids, E: int):
    """-> (cnt [E], off [E+1], sorted_rows [T*k], inv_pos [T,k]), all int32."""
    a = _np(ids, np.int32)
    T, k = a.shape
    cnt = np.empty(E, np.int32)
    off = np.empty(E + 1, np.int32)
    sr = np.empty(T * k, np.int32)
    inv = np.empty((T, k), np.int32)
    lib().oracle_permute(_ptr(a), T, k, E, _ptr(cnt), _ptr(off), _ptr(sr), _ptr(inv))
    return cnt, off, sr, inv


def expert_mlp(xq, xs, gu_blocks, gu_scales, gu_bias, d_blocks, d_scales, d_bias, act_format: str = "mxfp8"):
    """One expert on one quantised row -> dict(g, h, hq, hs, y); act_format "mxfp8" or "mxfp4"."""
    xq = _np(xq, np.uint8)
    xs = _np(xs, np.uint8)
    gub, gus, gubias = _np(gu_blocks, np.uint8), _np(gu_scales, np.uint8), _np(gu_bias, np.uint16)
    db, ds, dbias = _np(d_blocks, np.uint8), _np(d_scales, np.uint8), _np(d_bias, np.uint16)
    H = xq.shape[-1]
    I = gus.shape[0] // 2
    g = np.empty(2 * I, np.float64)
    h = np.empty(I, np.float64)
    hq = np.empty(I, np.uint8)
    hs = np.empty(I // 32, np.uint8)
    y = np.empty(H, np.float64)
    lib().oracle_expert_mlp_fmt(_ptr(xq), _ptr(xs), H, I, _ptr(gub), _ptr(gus), _ptr(gubias),
                                _ptr(db), _ptr(ds), _ptr(dbias), _ptr(g), _ptr(h), _ptr(hq), _ptr(hs),
                                _ptr(y), _ACT[act_format])
    return dict(g=g, h=h, hq=hq, hs=hs, y=y)


def mxfp4_amax(blocks, scales) -> float:
    """Largest magnitude of an MXFP4 tensor (checkpoint layout, any leading dims)."""
    b = _np(blocks, np.uint8)
    s = _np(scales, np.uint8)
    nb = s.shape[-1]
    rows = s.size // nb
    return lib().oracle_mxfp4_amax(_ptr(b), _ptr(s), rows, nb * 32)


def convert_mxfp4_to_nvfp4(blocks, scales, gs: float):
    """MXFP4 rows [rows, K/32, 16] + [rows, K/32] -> NVFP4 (codes [rows, K] one per byte,
    E4M3 scale codes [rows, K/16]) with global scale gs."""
    b = _np(blocks, np.uint8)
    s = _np(scales, np.uint8)
    rows, nb = s.shape[-2], s.shape[-1]
    K = nb * 32
    codes = np.empty((rows, K), np.uint8)
    sc = np.empty((rows, K // 16), np.uint8)
    lib().oracle_convert_mxfp4_to_nvfp4(_ptr(b), _ptr(s), rows, K, float(gs), _ptr(codes), _ptr(sc))
    return codes, sc


def moe_forward(x, router_w, router_b, gu_blocks, gu_scales, gu_bias, d_blocks, d_scales, d_bias,
                k: int, intermediates: bool = False, act_format: str = "mxfp8"):
    """The whole layer -> dict(out fp64 [T,H], logits, ids, w, xq, xs[, h, hq, hs]).

    act_format "mxfp8" (the layer as built) or "mxfp4" (activations x and h
    quantised to MXFP4, the FP4 x FP4 variant)."""
    xx = _np(x, np.uint16)
    wr, br = _np(router_w, np.uint16), _np(router_b, np.uint16)
    gub, gus, gubias = _np(gu_blocks, np.uint8), _np(gu_scales, np.uint8), _np(gu_bias, np.uint16)
    db, ds, dbias = _np(d_blocks, np.uint8), _np(d_scales, np.uint8), _np(d_bias, np.uint16)
    T, H = xx.shape
    E = wr.shape[0]
    I = gus.shape[1] // 2
    if act_format == "nvfp4":
        return _moe_forward_nvfp4(xx, wr, br, gub, gus, gubias, db, ds, dbias, T, H, I, E, k, intermediates)
    out = np.empty((T, H), np.float64)
    logits = np.empty((T, E), np.float64)
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    xq = np.empty((T, H), np.uint8)
    xs = np.empty((T, H // 32), np.uint8)
    h = hq = hs = None
    if intermediates:
        h = np.empty((T, k, I), np.float64)
        hq = np.empty((T, k, I), np.uint8)
        hs = np.empty((T, k, I // 32), np.uint8)
    lib().oracle_moe_forward_fmt(_ptr(xx), T, H, I, E, k, _ptr(wr), _ptr(br), _ptr(gub), _ptr(gus),
                                 _ptr(gubias), _ptr(db), _ptr(ds), _ptr(dbias), _ptr(out),
                                 _ptr(logits), _ptr(ids), _ptr(w), _ptr(xq), _ptr(xs), _ptr(h),
                                 _ptr(hq), _ptr(hs), _ACT[act_format])
    r = dict(out=out, logits=logits, ids=ids, w=w, xq=xq, xs=xs)
    if intermediates:
        r.update(h=h, hq=hq, hs=hs)
    return r


def bf16_round_array(v) -> np.ndarray:
    """fp64 array -> bf16 bit patterns (one RNE rounding per element)."""
    a = _np(v, np.float64)
    L = lib()
    return np.array([L.oracle_bf16_round(float(x)) for x in a.reshape(-1)], np.uint16).reshape(a.shape)


def rmsnorm_bf16(x, eps: float = 1e-5) -> np.ndarray:
    """fp64 [T,H] -> bf16 bits uint16 [T,H]."""
    a = _np(x, np.float64)
    T, H = a.shape
    out = np.empty((T, H), np.uint16)
    lib().oracle_rmsnorm_bf16(_ptr(a), T, H, eps, _ptr(out))
    return out


# --- dense MXFP4 linears -------------------------------------------------------------
def pack_e2m1(codes) -> np.ndarray:
    """E2M1 codes one per byte [rows, K] -> checkpoint blocks [rows, K/32, 16]."""
    c = _np(codes, np.uint8)
    rows, K = c.shape
    out = np.empty((rows, K // 32, 16), np.uint8)
    lib().oracle_pack_e2m1(_ptr(c), rows, K, _ptr(out))
    return out


def quantize_mxfp4_weights(w):
    """fp64 [rows, K] -> (blocks [rows, K/32, 16], scales [rows, K/32]) in the checkpoint layout."""
    a = _np(w, np.float64)
    rows, K = a.shape
    blocks = np.empty((rows, K // 32, 16), np.uint8)
    scales = np.empty((rows, K // 32), np.uint8)
    lib().oracle_quantize_mxfp4_weights(_ptr(a), rows, K, _ptr(blocks), _ptr(scales))
    return blocks, scales


def dense_linear(x, blocks, scales, bias=None, act_format: str = "mxfp8") -> np.ndarray:
    """bf16 x [T, K] against MXFP4 W [N, K] (+ bf16 bias [N]) -> fp64 [T, N]."""
    xx = _np(x, np.uint16)
    b = _np(blocks, np.uint8)
    sc = _np(scales, np.uint8)
    bb = None if bias is None else _np(bias, np.uint16)
    T, K = xx.shape
    N = sc.shape[0]
    out = np.empty((T, N), np.float64)
    lib().oracle_dense_linear(_ptr(xx), T, K, N, _ptr(b), _ptr(sc), _ptr(bb), _ptr(out), _ACT[act_format])
    return out


# --- NVFP4 -----------------------------------------------------------------------------
def nvfp4_global_scale(amax: float) -> float:
    return lib().oracle_nvfp4_global_scale(float(amax))


def nvfp4_quantize(v, gs: float = 1.0):
    """fp64 values (last dim a multiple of 16) -> (E2M1 codes one per byte, E4M3 scale codes per 16)."""
    a = _np(v, np.float64)
    q = np.empty(a.shape, np.uint8)
    s = np.empty(a.shape[:-1] + (a.shape[-1] // 16,), np.uint8)
    lib().oracle_nvfp4_quantize(_ptr(a), a.size, float(gs), _ptr(q), _ptr(s))
    return q, s


def nvfp4_value(code: int, scale_code: int, gs: float = 1.0) -> float:
    return lib().oracle_nvfp4_value(code, scale_code, float(gs))


def nvfp4_dequant(codes, scale_codes, gs: float) -> np.ndarray:
    """codes [..., K] (one per byte) and scale codes [..., K/16] -> fp64 values."""
    c = _np(codes, np.uint8)
    s = _np(scale_codes, np.uint8)
    e2 = np.array([e2m1_value(i) for i in range(16)])
    e4 = np.array([e4m3_value(i) for i in range(256)])
    return e2[c] * np.repeat(e4[s], 16, axis=-1) * gs


def expert_mlp_nvfp4(xq, xs, gu_codes, gu_sc, gu_gs, gu_bias, d_codes, d_sc, d_gs, d_bias):
    """One expert on one NVFP4 activation row with NVFP4 weights -> dict(h, hq, hs, y)."""
    xq = _np(xq, np.uint8)
    xs = _np(xs, np.uint8)
    guc, gus, gub = _np(gu_codes, np.uint8), _np(gu_sc, np.uint8), _np(gu_bias, np.uint16)
    dc, ds, db = _np(d_codes, np.uint8), _np(d_sc, np.uint8), _np(d_bias, np.uint16)
    H = xq.shape[-1]
    I = guc.shape[0] // 2
    h = np.empty(I, np.float64)
    hq = np.empty(I, np.uint8)
    hs = np.empty(I // 16, np.uint8)
    y = np.empty(H, np.float64)
    lib().oracle_expert_mlp_nvfp4(_ptr(xq), _ptr(xs), H, I, _ptr(guc), _ptr(gus), float(gu_gs), _ptr(gub),
                                  _ptr(dc), _ptr(ds), float(d_gs), _ptr(db), _ptr(h), _ptr(hq), _ptr(hs), _ptr(y))
    return dict(h=h, hq=hq, hs=hs, y=y)


def _moe_forward_nvfp4(xx, wr, br, gub, gus, gubias, db, ds, dbias, T, H, I, E, k, intermediates):
    out = np.empty((T, H), np.float64)
    logits = np.empty((T, E), np.float64)
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    xq = np.empty((T, H), np.uint8)
    xs = np.empty((T, H // 16), np.uint8)
    h = hq = hs = None
    if intermediates:
        h = np.empty((T, k, I), np.float64)
        hq = np.empty((T, k, I), np.uint8)
        hs = np.empty((T, k, I // 16), np.uint8)
    lib().oracle_moe_forward_nvfp4(_ptr(xx), T, H, I, E, k, _ptr(wr), _ptr(br), _ptr(gub), _ptr(gus),
                                   _ptr(gubias), _ptr(db), _ptr(ds), _ptr(dbias), _ptr(out), _ptr(logits),
                                   _ptr(ids), _ptr(w), _ptr(xq), _ptr(xs), _ptr(h), _ptr(hq), _ptr(hs))
    r = dict(out=out, logits=logits, ids=ids, w=w, xq=xq, xs=xs)
    if intermediates:
        r.update(h=h, hq=hq, hs=hs)
    return r
