"""The C ABI without a GPU: the library loads, exports every declared symbol,
computes sizes, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import mxfp4_mixture_experts_gemv_gb300 as moe
from mxfp4_mixture_experts_gemv_gb300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    moe_build.build()
    return moe.lib()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_declarations_match_binding():
    assert _declared_functions() == sorted(moe.EXPORTED)


def test_library_exports_every_declared_symbol(L):
    for name in _declared_functions():
        assert hasattr(L, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", moe.LIB_PATH], capture_output=True, text=True).stdout
    for name in _declared_functions():
        assert re.search(rf"\bT {name}$", out, re.M), name


def test_version(L):
    assert L.moe_version() & 0xFFFF == 2


GPT = moe.LayerDims(E=128, H=2880, I=2880)


def test_packed_size_layout():
    # data rows padded to 2944 elements (1472 bytes), scale atoms of 512 bytes per
    # 128 rows x 128 columns, fp32 biases, each section 1024-aligned after a 1 KB header
    def r(x):
        return (x + 1023) // 1024 * 1024
    gu_data = 128 * 5760 * 1472   # tile-contiguous, K padded to 2944
    gu_sf = 128 * 45 * 23 * 512
    gu_b = 128 * 5760 * 4
    d_data = 128 * 2880 * 1472    # 2880 rows = 22 full tiles + one 64-row tile
    d_sf = 128 * 23 * 23 * 512
    d_b = 128 * 2880 * 4
    want = 1024 + sum(r(x) for x in (gu_data, gu_sf, gu_b, d_data, d_sf, d_b))
    assert moe.packed_size(GPT) == want
    assert moe.packed_size(moe.LayerDims(8, 100, 256)) == 0   # H not a multiple of 32
    assert moe.packed_size(moe.LayerDims(8, 256, 96)) == 0    # I not a multiple of 64
    assert moe.packed_size(moe.LayerDims(300, 256, 256)) == 0  # E > 256


def test_workspace_layout_sections_are_disjoint_and_aligned():
    for T in (1, 4, 32, 128, 129, 256, 512, 1000, 1024, 2048, 8192):
        lay = moe.workspace_layout(GPT, T, 4)
        names = [f[0] for f in moe.WorkspaceLayout._fields_[:-3] if f[0] != "zero_bytes"]
        assert lay.zero_bytes == lay.logits  # status and counters lead the workspace
        offs = [getattr(lay, n) for n in names]
        assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
        assert lay.total == moe.workspace_size(GPT, T, 4)
        # the measured table: 128-row tiles (tokens-on-M) from 8 rows per expert on
        # average (T >= 225 here), below that twice the average rounded up to a power of
        # two from 8 (8 rows up to T = 128)
        avg = -(-T * 4 // 128)
        want = 128 if avg >= 8 else 8 if T <= 128 else 16
        assert lay.tile_rows == want
        # MXFP4 follows the same table; NVFP4 keeps the weights-on-M table; the
        # offsets are the same for every format
        want_nv = 8 if T <= 128 else 16 if T <= 256 else 32 if T <= 512 else 64 if T <= 1024 else 128
        for fmt, w in (("mxfp4", want), ("nvfp4", want_nv)):
            l4 = moe.workspace_layout(GPT, T, 4, fmt)
            assert l4.tile_rows == w
            assert [getattr(l4, n) for n in names] == offs and l4.total == lay.total
            assert l4.max_tiles >= T * 4 // l4.tile_rows + min(T * 4, 128)
        # enough tiles for any routing: every expert's partial tile plus full tiles
        assert lay.max_tiles >= T * 4 // lay.tile_rows + min(T * 4, 128)


FAKE = 1 << 20  # never dereferenced: every call below fails validation first


def _fwd(L, dims=GPT, hidden=FAKE, T=4, rw=FAKE, rb=FAKE, packed=FAKE, k=4, out=FAKE, ws=FAKE,
         ws_bytes=1 << 40):
    return L.moe_forward(dims.c(), hidden, T, rw, rb, packed, k, out, ws, ws_bytes, None)


def test_forward_rejects_bad_arguments_on_host(L):
    assert _fwd(L, k=0) == 1 and b"top_k" in L.moe_last_error()
    assert _fwd(L, k=9) == 1
    assert _fwd(L, dims=moe.LayerDims(4, 64, 128), k=5) == 1        # k > E
    assert _fwd(L, T=-1) == 1
    assert _fwd(L, dims=moe.LayerDims(128, 2888, 2880)) == 2         # H % 32
    assert _fwd(L, dims=moe.LayerDims(128, 2880, 2880 + 32)) == 2    # I % 64
    assert _fwd(L, dims=moe.LayerDims(257, 2880, 2880)) == 2
    assert _fwd(L, hidden=0) == 1
    assert _fwd(L, out=0) == 1
    assert _fwd(L, hidden=FAKE + 8) == 3
    assert _fwd(L, ws=FAKE + 16) == 3
    assert _fwd(L, packed=FAKE + 128) == 3
    need = moe.workspace_size(GPT, 4, 4)
    assert _fwd(L, ws_bytes=need - 1) == 4 and b"workspace" in L.moe_last_error()
    assert _fwd(L, T=0) == 0  # no-op, nothing launched
    assert _fwd(L, T=1 << 24) == 2  # T*k*H beyond 32-bit indexing


def test_pack_rejects_bad_arguments_on_host(L):
    w = moe.Weights(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)
    n = moe.packed_size(GPT)
    assert L.moe_pack_weights(GPT.c(), None, FAKE, n, None) == 1
    assert L.moe_pack_weights(GPT.c(), ctypes.byref(w), FAKE + 64, n, None) == 3
    assert L.moe_pack_weights(GPT.c(), ctypes.byref(w), FAKE, n - 1, None) == 5
    w2 = moe.Weights(FAKE + 4, FAKE, FAKE, FAKE, FAKE, FAKE)
    assert L.moe_pack_weights(GPT.c(), ctypes.byref(w2), FAKE, n, None) == 3
    w3 = moe.Weights(FAKE, 0, FAKE, FAKE, FAKE, FAKE)
    assert L.moe_pack_weights(GPT.c(), ctypes.byref(w3), FAKE, n, None) == 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU failure path")
def test_forward_fails_loudly_without_a_gpu(L):
    # valid arguments on a host with no CUDA device: the library reports a CUDA
    # error instead of computing anything on the CPU
    assert _fwd(L) == 6
    assert b"cudaError" in L.moe_last_error()


def test_residual_rmsnorm_rejects_bad_arguments_on_host(L):
    assert L.moe_residual_rmsnorm(FAKE, None, 4, 2882, 1e-5, FAKE, None) == 1    # H % 4
    assert L.moe_residual_rmsnorm(FAKE, None, 4, 2880, 0.0, FAKE, None) == 1     # eps must be > 0
    assert L.moe_residual_rmsnorm(0, None, 4, 2880, 1e-5, FAKE, None) == 1       # null residual
    assert L.moe_residual_rmsnorm(FAKE + 8, None, 4, 2880, 1e-5, FAKE, None) == 3
    assert L.moe_residual_rmsnorm(FAKE, None, 0, 2880, 1e-5, FAKE, None) == 0    # T = 0: no-op


def test_wait_limit_and_hold_mask_are_checked_on_host(L):
    assert L.moe_set_wait_limit_ns(10) == 1             # below 1 us
    assert L.moe_set_wait_limit_ns(61_000_000_000) == 1  # above 60 s
    assert L.moe_set_wait_limit_ns(5_000_000) == 0 and L.moe_get_wait_limit_ns() == 5_000_000
    assert L.moe_set_wait_limit_ns(0) == 0 and L.moe_get_wait_limit_ns() == 2_000_000_000
    assert L.moe_debug_hold_waits(8) == 1
    assert L.moe_debug_hold_waits(moe.HOLD_DOWN_UNITS | moe.HOLD_ROUTING_BARRIER) == 0
    assert L.moe_debug_hold_waits(0) == 0


def test_plan_override_is_checked_and_sizes_follow_it(L):
    assert L.moe_set_plan(12, 0, 0) == 1           # not a tile height the kernels have
    assert L.moe_set_plan(0, 7, 0) == 1            # unknown routing path
    assert L.moe_set_plan(0, 0, 4) == 1            # unknown expert kernel
    base = moe.workspace_layout(GPT, 1024, 4)
    assert base.tile_rows == 128
    try:
        moe.set_plan(8, "tensor_core")
        lay = moe.workspace_layout(GPT, 1024, 4)
        assert lay.tile_rows == 8 and lay.max_tiles > base.max_tiles
        assert moe.workspace_size(GPT, 1024, 4) == lay.total
    finally:
        moe.set_plan(0, "auto")
    assert moe.workspace_layout(GPT, 1024, 4).tile_rows == 128


def test_forward_act_rejects_unknown_formats(L):
    assert L.moe_forward_act(GPT.c(), 3, FAKE, 4, FAKE, FAKE, FAKE, 4, FAKE, FAKE, 1 << 40, None) == 1
    assert b"activation format" in L.moe_last_error()


def test_dense_sizes_and_host_checks(L):
    # packed: 1 KiB header, then 64-byte rows per 128-wide k-tile (K padded to 128),
    # 512-byte scale atoms per (128-row, 128-wide) tile, fp32 biases; 1 KiB sections
    N, K = 320, 288
    kt, mt = 3, 3
    up = lambda b: (b + 1023) // 1024 * 1024
    want = 1024 + up(N * kt * 64) + up(mt * kt * 512) + up(N * 4)
    assert L.moe_dense_packed_size(N, K) == want
    assert L.moe_dense_packed_size(100, 256) == 0    # N a multiple of 64
    assert L.moe_dense_packed_size(128, 250) == 0    # K a multiple of 32
    assert L.moe_dense_workspace_size(128, 256, -1) == 0
    assert L.moe_dense_quantize_weights(128, 250, FAKE, FAKE, FAKE, None) == 2
    assert L.moe_dense_quantize_weights(128, 256, None, FAKE, FAKE, None) == 1
    assert L.moe_dense_quantize_weights(128, 256, FAKE + 2, FAKE, FAKE, None) == 3
    n = L.moe_dense_packed_size(128, 256)
    assert L.moe_dense_pack(100, 256, FAKE, FAKE, None, FAKE, n, None) == 2
    assert L.moe_dense_pack(128, 256, None, FAKE, None, FAKE, n, None) == 1
    assert L.moe_dense_pack(128, 256, FAKE, FAKE, None, FAKE + 64, n, None) == 3
    assert L.moe_dense_pack(128, 256, FAKE, FAKE, None, FAKE, n - 1, None) == 5
    ws = L.moe_dense_workspace_size(128, 256, 4)
    assert ws > 0
    fwd = lambda **kw: L.moe_dense_forward(kw.get("N", 128), 256, kw.get("x", FAKE), kw.get("T", 4), kw.get("pk", FAKE),
                                           kw.get("out", FAKE), kw.get("ws", FAKE), kw.get("ws_bytes", ws), None)
    assert fwd(N=100) == 2
    assert fwd(T=-1) == 1
    assert fwd(T=0) == 0                             # no-op
    assert fwd(x=0) == 1 and fwd(out=0) == 1
    assert fwd(x=FAKE + 8) == 3 and fwd(pk=FAKE + 16) == 3
    assert fwd(ws_bytes=ws - 1) == 4
    try:
        moe.set_plan(0, "auto", "cuda_cores")
        assert fwd(T=5, ws_bytes=1 << 30) == 2 and b"at most 4 tokens" in L.moe_last_error()
    finally:
        moe.set_plan(0, "auto")


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU failure path")
def test_dense_forward_fails_loudly_without_a_gpu(L):
    ws = L.moe_dense_workspace_size(128, 256, 4)
    assert L.moe_dense_forward(128, 256, FAKE, 4, FAKE, FAKE, FAKE, ws, None) == 6
    assert b"cudaError" in L.moe_last_error()


def test_workspace_sections_hold_every_formats_tiles():
    """For random layer shapes and token counts, each activation format's tile height
    and tile capacity fit the shared section offsets: the tile list, the gate_up
    counters and both scale-atom sections are sized for the largest tile count any
    format can produce (every expert's partial tile plus the full tiles)."""
    import random
    rng = random.Random(7)
    for _ in range(300):
        E = rng.choice([1, 2, 3, 8, 32, 128, 200, 256])
        k = rng.randint(1, min(8, E))
        H = 32 * rng.randint(1, 100)
        I = 64 * rng.randint(1, 50)
        T = rng.choice([0, 1, rng.randint(1, 64), rng.randint(1, 3000), rng.randint(1, 20000)])
        dims = moe.LayerDims(E, H, I)
        lays = {f: moe.workspace_layout(dims, T, k, f) for f in ("mxfp8", "mxfp4", "nvfp4")}
        base = lays["mxfp8"]
        kth, kti = -(-H // 128), -(-I // 128)
        TK = T * k
        for f, l in lays.items():
            for name, _ in moe.WorkspaceLayout._fields_[:-2]:
                if name not in ("max_tiles", "tile_rows"):
                    assert getattr(l, name) == getattr(base, name), (f, name)
            assert l.tile_rows in (8, 16, 32, 64, 128)
            assert l.max_tiles >= TK // l.tile_rows + min(TK, E), (f, E, k, T)
            assert l.done_tok - l.done_gu >= 4 * l.max_tiles
            assert l.xp - l.tiles >= (4 + 4 * l.max_tiles) * 4
            assert l.hq - l.xp_sf >= l.max_tiles * kth * 2 * 512
            assert l.y - l.hq_sf >= l.max_tiles * kti * 2 * 512
