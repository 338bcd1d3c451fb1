"""Python binding of the GB300 MXFP4 mixture-of-experts layer.

Argument marshalling only: every step of the layer runs in the CUDA kernels of
``libmoe_gb300.so`` (see ``include/moe.h``).  torch supplies device memory and
the current stream.  There is no fallback: if the shared library is missing or
a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_OK = 0
STATUS_NAMES = {
    0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE", 3: "MOE_ERR_ALIGNMENT",
    4: "MOE_ERR_WORKSPACE_TOO_SMALL", 5: "MOE_ERR_BAD_PACKED_HEADER", 6: "MOE_ERR_CUDA",
    7: "MOE_ERR_TIMEOUT",
}

# Every symbol the C ABI exports (include/moe.h).
EXPORTED = ["moe_packed_size", "moe_pack_weights", "moe_packed_size_nvfp4", "moe_pack_weights_nvfp4",
            "moe_workspace_size", "moe_workspace_layout_get", "moe_workspace_layout_act",
            "moe_forward", "moe_forward_act", "moe_forward_static_scratch", "moe_static_scratch_status", "moe_static_scratch_bytes",
            "moe_get_device_status", "moe_set_wait_limit_ns", "moe_get_wait_limit_ns",
            "moe_debug_hold_waits", "moe_set_plan", "moe_profile_begin", "moe_profile_end", "moe_residual_rmsnorm",
            "moe_dense_packed_size", "moe_dense_quantize_weights", "moe_dense_pack", "moe_dense_workspace_size",
            "moe_dense_forward", "moe_last_error", "moe_version"]
STAGES = ["routing", "expert_mlp"]


class MoeError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("gate_up_blocks", "gate_up_scales", "gate_up_bias",
                                                "down_blocks", "down_scales", "down_bias")]


class WorkspaceLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "status", "done_gu", "done_tok", "grid_bar", "zero_bytes", "logits", "topk_ids", "topk_w", "xq", "xs", "counts", "offsets", "sorted_rows",
        "inv_pos", "tiles", "xp", "xp_sf", "hq", "hq_sf", "y", "total")] + [
        ("max_tiles", ctypes.c_int32), ("tile_rows", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load the shared library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run __graft_entry__.build() (or "
                               "python -m mxfp4_mixture_experts_gemv_gb300.build) first")
        L = ctypes.CDLL(LIB_PATH)
        sz, st, vp, i32 = ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p, ctypes.c_int32
        L.moe_packed_size.restype = sz
        L.moe_packed_size.argtypes = [Dims]
        L.moe_pack_weights.restype = st
        L.moe_pack_weights.argtypes = [Dims, ctypes.POINTER(Weights), vp, sz, vp]
        L.moe_packed_size_nvfp4.restype = sz
        L.moe_packed_size_nvfp4.argtypes = [Dims]
        L.moe_pack_weights_nvfp4.restype = st
        L.moe_pack_weights_nvfp4.argtypes = [Dims, ctypes.POINTER(Weights), vp, sz, vp]
        L.moe_workspace_size.restype = sz
        L.moe_workspace_size.argtypes = [Dims, i32, i32]
        L.moe_workspace_layout_get.restype = st
        L.moe_workspace_layout_get.argtypes = [Dims, i32, i32, ctypes.POINTER(WorkspaceLayout)]
        L.moe_workspace_layout_act.restype = st
        L.moe_workspace_layout_act.argtypes = [Dims, i32, i32, i32, ctypes.POINTER(WorkspaceLayout)]
        L.moe_forward.restype = st
        L.moe_forward.argtypes = [Dims, vp, i32, vp, vp, vp, i32, vp, vp, sz, vp]
        L.moe_forward_act.restype = st
        L.moe_forward_act.argtypes = [Dims, i32, vp, i32, vp, vp, vp, i32, vp, vp, sz, vp]
        L.moe_forward_static_scratch.restype = st
        L.moe_forward_static_scratch.argtypes = [Dims, vp, i32, vp, vp, vp, i32, vp, vp]
        L.moe_static_scratch_status.restype = st
        L.moe_static_scratch_status.argtypes = [vp]
        L.moe_static_scratch_bytes.restype = sz
        L.moe_static_scratch_bytes.argtypes = []
        L.moe_get_device_status.restype = st
        L.moe_get_device_status.argtypes = [vp, vp]
        L.moe_set_wait_limit_ns.restype = st
        L.moe_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        L.moe_get_wait_limit_ns.restype = ctypes.c_uint64
        L.moe_get_wait_limit_ns.argtypes = []
        L.moe_set_plan.restype = st
        L.moe_set_plan.argtypes = [i32, i32, i32]
        L.moe_debug_hold_waits.restype = st
        L.moe_debug_hold_waits.argtypes = [i32]
        L.moe_residual_rmsnorm.restype = st
        L.moe_residual_rmsnorm.argtypes = [vp, vp, i32, i32, ctypes.c_float, vp, vp]
        L.moe_profile_begin.restype = st
        L.moe_profile_begin.argtypes = [i32]
        L.moe_profile_end.restype = st
        L.moe_profile_end.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int32)]
        L.moe_dense_packed_size.restype = sz
        L.moe_dense_packed_size.argtypes = [i32, i32]
        L.moe_dense_quantize_weights.restype = st
        L.moe_dense_quantize_weights.argtypes = [i32, i32, vp, vp, vp, vp]
        L.moe_dense_pack.restype = st
        L.moe_dense_pack.argtypes = [i32, i32, vp, vp, vp, vp, sz, vp]
        L.moe_dense_workspace_size.restype = sz
        L.moe_dense_workspace_size.argtypes = [i32, i32, i32]
        L.moe_dense_forward.restype = st
        L.moe_dense_forward.argtypes = [i32, i32, vp, i32, vp, vp, vp, sz, vp]
        L.moe_last_error.restype = ctypes.c_char_p
        L.moe_last_error.argtypes = []
        L.moe_version.restype = ctypes.c_uint32
        L.moe_version.argtypes = []
        _lib = L
    return _lib


def _check(status: int):
    if status != MOE_OK:
        raise MoeError(status, lib().moe_last_error().decode())


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dev_ptr(t: torch.Tensor, name: str, dtype=None) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


@dataclasses.dataclass(frozen=True)
class LayerDims:
    E: int
    H: int
    I: int

    def c(self) -> Dims:
        return Dims(self.E, self.H, self.I)


def packed_size(dims: LayerDims) -> int:
    return lib().moe_packed_size(dims.c())


def workspace_size(dims: LayerDims, T: int, top_k: int) -> int:
    return lib().moe_workspace_size(dims.c(), T, top_k)


def workspace_layout(dims: LayerDims, T: int, top_k: int, act_format: str = "mxfp8") -> WorkspaceLayout:
    """Section offsets of the workspace (the same for every activation format) and
    the tile height / tile capacity the forward in ``act_format`` uses."""
    out = WorkspaceLayout()
    _check(lib().moe_workspace_layout_act(dims.c(), T, top_k, ACT_FORMATS[act_format], ctypes.byref(out)))
    return out


def _alloc_aligned(nbytes: int, device) -> torch.Tensor:
    """uint8 device buffer whose data pointer is 256-byte aligned."""
    buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % 256
    return buf[off:off + nbytes]


def pack_weights(dims: LayerDims, gate_up_blocks, gate_up_scales, gate_up_bias, down_blocks,
                 down_scales, down_bias, packed: torch.Tensor | None = None, stream=None,
                 nvfp4: bool = False) -> torch.Tensor:
    """Repack checkpoint-layout MXFP4 expert weights (CUDA tensors) into the forward layout
    (converted to NVFP4 with nvfp4=True, for the NVFP4 forward)."""
    L = lib()
    size_fn, pack_fn = (L.moe_packed_size_nvfp4, L.moe_pack_weights_nvfp4) if nvfp4 else (L.moe_packed_size,
                                                                                        L.moe_pack_weights)
    n = size_fn(dims.c())
    if n == 0:
        _check(pack_fn(dims.c(), None, None, 0, None))
    if packed is None:
        packed = _alloc_aligned(n, gate_up_blocks.device)
    w = Weights(_dev_ptr(gate_up_blocks, "gate_up_blocks", torch.uint8),
                _dev_ptr(gate_up_scales, "gate_up_scales", torch.uint8),
                _dev_ptr(gate_up_bias, "gate_up_bias", torch.bfloat16),
                _dev_ptr(down_blocks, "down_blocks", torch.uint8),
                _dev_ptr(down_scales, "down_scales", torch.uint8),
                _dev_ptr(down_bias, "down_bias", torch.bfloat16))
    _check(pack_fn(dims.c(), ctypes.byref(w), _dev_ptr(packed, "packed"), packed.numel() * packed.element_size(),
                   _stream(stream)))
    return packed


def alloc_workspace(dims: LayerDims, T: int, top_k: int, device="cuda") -> torch.Tensor:
    return _alloc_aligned(max(workspace_size(dims, T, top_k), 256), device)


ACT_FORMATS = {"mxfp8": 0, "mxfp4": 1, "nvfp4": 2}


def forward(dims: LayerDims, hidden: torch.Tensor, router_w: torch.Tensor, router_b: torch.Tensor,
            packed: torch.Tensor, top_k: int, out: torch.Tensor | None = None,
            workspace: torch.Tensor | None = None, stream=None, act_format: str = "mxfp8") -> torch.Tensor:
    """One MoE layer: bf16 hidden [T, H] -> bf16 out [T, H].

    act_format "mxfp8" (moe_forward) or "mxfp4" (moe_forward_act, FP4 x FP4)."""
    T = hidden.shape[0]
    if out is None:
        out = torch.empty_like(hidden)
    if workspace is None:
        workspace = alloc_workspace(dims, T, top_k, hidden.device)
    args = (_dev_ptr(hidden, "hidden", torch.bfloat16), T, _dev_ptr(router_w, "router_w", torch.bfloat16),
            _dev_ptr(router_b, "router_b", torch.bfloat16), _dev_ptr(packed, "packed"), top_k,
            _dev_ptr(out, "out", torch.bfloat16), _dev_ptr(workspace, "workspace"),
            workspace.numel() * workspace.element_size(), _stream(stream))
    if act_format == "mxfp8":
        _check(lib().moe_forward(dims.c(), *args))
    else:
        _check(lib().moe_forward_act(dims.c(), ACT_FORMATS[act_format], *args))
    return out


def static_scratch_bytes() -> int:
    """Size of the library's static scratch array (MOE_STATIC_SCRATCH_BYTES as built)."""
    return lib().moe_static_scratch_bytes()


def forward_static_scratch(dims: LayerDims, hidden: torch.Tensor, router_w: torch.Tensor,
                           router_b: torch.Tensor, packed: torch.Tensor, top_k: int,
                           out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The layer forward through the allocation-free entry point (library-owned scratch)."""
    if out is None:
        out = torch.empty_like(hidden)
    _check(lib().moe_forward_static_scratch(dims.c(), _dev_ptr(hidden, "hidden", torch.bfloat16), hidden.shape[0],
                                            _dev_ptr(router_w, "router_w", torch.bfloat16),
                                            _dev_ptr(router_b, "router_b", torch.bfloat16),
                                            _dev_ptr(packed, "packed"), top_k,
                                            _dev_ptr(out, "out", torch.bfloat16), _stream(stream)))
    return out


def residual_rmsnorm(x_res: torch.Tensor, layer_out: torch.Tensor | None, hidden: torch.Tensor,
                     eps: float = 1e-5, stream=None):
    """x_res (fp32 [T, H]) += layer_out (bf16, optional); hidden (bf16) = rmsnorm(x_res)."""
    T, H = x_res.shape
    _check(lib().moe_residual_rmsnorm(_dev_ptr(x_res, "x_res", torch.float32),
                                      None if layer_out is None else _dev_ptr(layer_out, "layer_out", torch.bfloat16),
                                      T, H, eps, _dev_ptr(hidden, "hidden", torch.bfloat16), _stream(stream)))
    return hidden


def profile_begin(max_calls: int):
    """Arm per-stage event timing for the next ``max_calls`` forward calls."""
    _check(lib().moe_profile_begin(max_calls))


def profile_end() -> tuple[dict, int]:
    """-> ({stage: summed ms}, calls recorded)."""
    ms = (ctypes.c_double * 8)()
    calls = ctypes.c_int32()
    _check(lib().moe_profile_end(ms, ctypes.byref(calls)))
    return {name: ms[i] for i, name in enumerate(STAGES)}, calls.value


def device_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise and return the status of the last forward that used ``workspace``."""
    return lib().moe_get_device_status(_dev_ptr(workspace, "workspace"), _stream(stream))


def static_scratch_status(stream=None) -> int:
    """Synchronise and return the status of the last allocation-free forward on this device."""
    return lib().moe_static_scratch_status(_stream(stream))


def set_wait_limit_ns(ns: int):
    """Limit of every bounded device-side wait in later launches (0 = the 2 s default)."""
    _check(lib().moe_set_wait_limit_ns(ns))


def wait_limit_ns() -> int:
    return lib().moe_get_wait_limit_ns()


ROUTES = {"auto": 0, "cluster": 1, "grid": 2, "tensor_core": 3}
EXPERT_KERNELS = {"auto": 0, "weights_m": 1, "tokens_m": 2, "cuda_cores": 3}


def set_plan(tile_rows: int = 0, route: str = "auto", expert: str = "auto"):
    """Force the token rows per expert tile (0 = default), the routing path ("auto",
    "cluster", "grid", "tensor_core") and the expert kernel ("auto", "weights_m",
    "tokens_m") of later forwards (measurement hook)."""
    _check(lib().moe_set_plan(tile_rows, ROUTES[route], EXPERT_KERNELS[expert]))


HOLD_DOWN_UNITS = 1
HOLD_ROUTING_BARRIER = 2


def debug_hold_waits(which: int):
    """Failure-detection test hook: make the masked waits of later forwards unreachable
    (HOLD_DOWN_UNITS, HOLD_ROUTING_BARRIER); 0 restores normal forwards."""
    _check(lib().moe_debug_hold_waits(which))


def view(workspace: torch.Tensor, offset: int, shape, dtype) -> torch.Tensor:
    """A typed view of a workspace section (for tests and debugging)."""
    n = 1
    for s in shape:
        n *= s
    nbytes = n * torch.empty(0, dtype=dtype).element_size()
    return workspace[offset:offset + nbytes].view(dtype).view(*shape)


# ----------------------------------------------------------------------- dense MXFP4 linears
def dense_quantize_weights(w: torch.Tensor, stream=None):
    """bf16 [N, K] -> (MXFP4 blocks uint8 [N, K/32, 16], E8M0 scales uint8 [N, K/32])."""
    N, K = w.shape
    blocks = torch.empty((N, K // 32, 16), dtype=torch.uint8, device=w.device)
    scales = torch.empty((N, K // 32), dtype=torch.uint8, device=w.device)
    _check(lib().moe_dense_quantize_weights(N, K, _dev_ptr(w, "w", torch.bfloat16), _dev_ptr(blocks, "blocks"),
                                            _dev_ptr(scales, "scales"), _stream(stream)))
    return blocks, scales


def dense_pack(blocks: torch.Tensor, scales: torch.Tensor, bias: torch.Tensor | None = None, stream=None):
    """MXFP4 checkpoint-layout W [N, K/32, 16] + [N, K/32] (+ bf16 bias [N]) -> packed buffer."""
    N, nb = scales.shape
    K = nb * 32
    n = lib().moe_dense_packed_size(N, K)
    if n == 0:
        _check(lib().moe_dense_pack(N, K, None, None, None, None, 0, None))
    packed = _alloc_aligned(n, blocks.device)
    _check(lib().moe_dense_pack(N, K, _dev_ptr(blocks, "blocks", torch.uint8), _dev_ptr(scales, "scales", torch.uint8),
                                None if bias is None else _dev_ptr(bias, "bias", torch.bfloat16),
                                _dev_ptr(packed, "packed"), n, _stream(stream)))
    return packed


def dense_forward(N: int, K: int, x: torch.Tensor, packed: torch.Tensor, out: torch.Tensor | None = None,
                  workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """bf16 x [T, K] -> bf16 out [T, N] = MXFP8(x) . W^T + b."""
    T = x.shape[0]
    if out is None:
        out = torch.empty((T, N), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = _alloc_aligned(max(lib().moe_dense_workspace_size(N, K, T), 256), x.device)
    _check(lib().moe_dense_forward(N, K, _dev_ptr(x, "x", torch.bfloat16), T, _dev_ptr(packed, "packed"),
                                   _dev_ptr(out, "out", torch.bfloat16), _dev_ptr(workspace, "workspace"),
                                   workspace.numel() * workspace.element_size(), _stream(stream)))
    return out
