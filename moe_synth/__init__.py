"""Seeded synthetic inputs for the MXFP4 mixture-of-experts layer.

This module only draws numbers.  It holds none of the layer's arithmetic: no
E2M1/E8M0 decoding, no quantisation, no routing.  Both the CUDA library's
tests/benchmark and the CPU oracle take their inputs from here, so the two
sides always see the same bytes.

Generator (counter-based, so any slice can be regenerated on its own):

* ``key(seed, stream)`` = splitmix64 finaliser of ``seed * 0x100000001B3 + stream``.
* element ``i`` of a stream uses ``h(i) = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)``,
  i.e. the (i+1)-th output of a splitmix64 sequence (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014) started at
  ``key``.
* bytes: byte ``b`` of a byte stream is byte ``b % 8`` (little-endian) of
  ``h(b // 8)``; each 4-bit nibble is therefore uniform over its 16 codes.
* block scales: ``118 + ((h(i) >> 1) mod 7)``, uniform over the E8M0 codes
  118..124.
* Gaussians: Box-Muller on two 24-bit uniforms of one hash,
  ``u1 = (h>>40)+1)/2^24``, ``u2 = ((h>>8) & 0xFFFFFF)/2^24``,
  ``z = sqrt(-2 ln u1) cos(2 pi u2)``, in float64, times the standard
  deviation (plus an optional mean shift), rounded to bfloat16 (RNE).

The arithmetic is done with torch int64 tensors (wrapping multiply, masked
logical shifts), so the same call gives the same bits on CPU and on CUDA.

Tensor shapes follow the checkpoint layout of the MXFP4 gpt-oss release as
described in "GPT-OSS-120B on DGX Spark: From MXFP4 to NVFP4" (section
"MXFP4 Tensor Structure"): ``*_blocks`` uint8 ``[E, out, in/32, 16]``,
``*_scales`` uint8 ``[E, out, in/32]``, ``*_bias`` bf16 ``[E, out]``.
"""
from __future__ import annotations

import dataclasses
import math

import torch

_GOLDEN = -7046029254386353131  # 0x9E3779B97F4A7C15 as int64
_M1 = -4658895280553007687      # 0xBF58476D1CE4E5B9
_M2 = -7723592293110705685      # 0x94D049BB133111EB
_FNV = 0x100000001B3

# stream ids of the tensors of one layer (stream = layer * 16 + tensor)
S_X, S_ROUTER_W, S_ROUTER_B = 1, 2, 3
S_GU_BLOCKS, S_GU_SCALES, S_GU_BIAS = 4, 5, 6
S_D_BLOCKS, S_D_SCALES, S_D_BIAS = 7, 8, 9


def _srl(z: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 lanes."""
    return (z >> k) & ((1 << (64 - k)) - 1)


def _mix64(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _srl(z, 30)) * _M1
    z = (z ^ _srl(z, 27)) * _M2
    return z ^ _srl(z, 31)


def _wrap64(v: int) -> int:
    v &= (1 << 64) - 1
    return v - (1 << 64) if v >= (1 << 63) else v


def stream_key(seed: int, stream: int) -> int:
    z = torch.tensor([_wrap64(seed * _FNV + stream)], dtype=torch.int64)
    return int(_mix64(z + _GOLDEN)[0])


def hashes(seed: int, stream: int, start: int, count: int, device="cpu") -> torch.Tensor:
    """h(i) for i in [start, start + count), int64."""
    key = stream_key(seed, stream)
    i = torch.arange(start + 1, start + count + 1, dtype=torch.int64, device=device)
    return _mix64(i * _GOLDEN + key)


def rand_bytes(seed: int, stream: int, start: int, count: int, device="cpu") -> torch.Tensor:
    """Bytes [start, start+count) of a byte stream, uint8."""
    if count == 0:
        return torch.empty(0, dtype=torch.uint8, device=device)
    h0, h1 = start // 8, (start + count + 7) // 8
    h = hashes(seed, stream, h0, h1 - h0, device)
    parts = [(_srl(h, 8 * b) & 0xFF) for b in range(8)]
    b = torch.stack(parts, dim=1).reshape(-1).to(torch.uint8)
    off = start - 8 * h0
    return b[off:off + count]


def rand_scales(seed: int, stream: int, start: int, count: int, lo=118, hi=124,
                device="cpu") -> torch.Tensor:
    h = hashes(seed, stream, start, count, device)
    return (lo + torch.remainder(_srl(h, 1), hi - lo + 1)).to(torch.uint8)


def rand_normal_bf16(seed: int, stream: int, start: int, count: int, std: float,
                     mean: float = 0.0, device="cpu") -> torch.Tensor:
    h = hashes(seed, stream, start, count, device)
    u1 = (_srl(h, 40) + 1).to(torch.float64) / float(1 << 24)
    u2 = (_srl(h, 8) & 0xFFFFFF).to(torch.float64) / float(1 << 24)
    z = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos(2.0 * math.pi * u2)
    return (z * std + mean).to(torch.bfloat16)


@dataclasses.dataclass(frozen=True)
class LayerShape:
    T: int      # tokens
    H: int      # hidden size
    I: int      # expert intermediate size
    E: int      # experts
    k: int      # experts per token


@dataclasses.dataclass
class LayerInputs:
    """One MoE layer's inputs in the checkpoint layout (all on one device)."""
    shape: LayerShape
    x: torch.Tensor              # bf16 [T, H]
    router_w: torch.Tensor       # bf16 [E, H]
    router_b: torch.Tensor       # bf16 [E]
    gate_up_blocks: torch.Tensor  # uint8 [E, 2I, H/32, 16]; rows [0,I)=gate, [I,2I)=up
    gate_up_scales: torch.Tensor  # uint8 [E, 2I, H/32]
    gate_up_bias: torch.Tensor    # bf16 [E, 2I]
    down_blocks: torch.Tensor     # uint8 [E, H, I/32, 16]
    down_scales: torch.Tensor     # uint8 [E, H, I/32]
    down_bias: torch.Tensor       # bf16 [E, H]

    def to(self, device) -> "LayerInputs":
        kw = {f.name: (getattr(self, f.name).to(device) if f.name != "shape" else self.shape)
              for f in dataclasses.fields(self)}
        return LayerInputs(**kw)


def make_tokens(seed: int, T: int, H: int, layer: int = 0, device="cpu") -> torch.Tensor:
    """Hidden states x ~ N(0, 1), bf16 [T, H]."""
    return rand_normal_bf16(seed, layer * 16 + S_X, 0, T * H, 1.0, device=device).view(T, H)


def make_router(seed: int, H: int, E: int, layer: int = 0, hot_experts: int = 0,
                hot_bias: float = 0.0, device="cpu"):
    """Router weight N(0, 1/sqrt(H)) bf16 [E, H] and bias N(0, 0.01) bf16 [E].

    ``hot_experts`` > 0 adds ``hot_bias`` to the bias of experts
    0..hot_experts-1 before the bf16 rounding (skewed expert load).
    """
    w = rand_normal_bf16(seed, layer * 16 + S_ROUTER_W, 0, E * H, 1.0 / math.sqrt(H),
                         device=device).view(E, H)
    h = hashes(seed, layer * 16 + S_ROUTER_B, 0, E, device)
    u1 = (_srl(h, 40) + 1).to(torch.float64) / float(1 << 24)
    u2 = (_srl(h, 8) & 0xFFFFFF).to(torch.float64) / float(1 << 24)
    z = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos(2.0 * math.pi * u2) * 0.01
    if hot_experts:
        z[:hot_experts] += hot_bias
    return w, z.to(torch.bfloat16)


def make_expert_weights(seed: int, H: int, I: int, E: int, layer: int = 0,
                        experts=None, device="cpu"):
    """MXFP4 expert weights for the listed experts (default: all), checkpoint layout.

    Element indices are global over all E experts, so generating a subset gives
    the same bytes as slicing the full tensors.
    Returns (gu_blocks, gu_scales, gu_bias, d_blocks, d_scales, d_bias).
    """
    if experts is None:
        experts = range(E)
    experts = list(experts)
    nb_h, nb_i = H // 32, I // 32
    base = layer * 16
    gub, gus, gubias, db, ds, dbias = [], [], [], [], [], []
    for e in experts:
        n = 2 * I * nb_h * 16
        gub.append(rand_bytes(seed, base + S_GU_BLOCKS, e * n, n, device).view(2 * I, nb_h, 16))
        n = 2 * I * nb_h
        gus.append(rand_scales(seed, base + S_GU_SCALES, e * n, n, device=device).view(2 * I, nb_h))
        gubias.append(rand_normal_bf16(seed, base + S_GU_BIAS, e * 2 * I, 2 * I, 0.02, device=device))
        n = H * nb_i * 16
        db.append(rand_bytes(seed, base + S_D_BLOCKS, e * n, n, device).view(H, nb_i, 16))
        n = H * nb_i
        ds.append(rand_scales(seed, base + S_D_SCALES, e * n, n, device=device).view(H, nb_i))
        dbias.append(rand_normal_bf16(seed, base + S_D_BIAS, e * H, H, 0.02, device=device))
    st = lambda xs: torch.stack(xs) if xs else None
    return st(gub), st(gus), st(gubias), st(db), st(ds), st(dbias)


def make_layer(shape: LayerShape, seed: int = 0, layer: int = 0, hot_experts: int = 0,
               hot_bias: float = 0.0, device="cpu") -> LayerInputs:
    T, H, I, E, _ = dataclasses.astuple(shape)
    x = make_tokens(seed, T, H, layer, device)
    rw, rb = make_router(seed, H, E, layer, hot_experts, hot_bias, device)
    gub, gus, gubias, db, ds, dbias = make_expert_weights(seed, H, I, E, layer, device=device)
    return LayerInputs(shape, x, rw, rb, gub, gus, gubias, db, ds, dbias)


# The workloads: tiny smoke case, gpt-oss-shaped decode, skewed batched decode,
# prefill, and the 36-layer residual stack.
WORKLOADS = {
    "tiny": dict(shape=LayerShape(T=8, H=256, I=256, E=8, k=2), hot_experts=0),
    "decode_t4": dict(shape=LayerShape(T=4, H=2880, I=2880, E=128, k=4), hot_experts=0),
    "decode_t32_skewed": dict(shape=LayerShape(T=32, H=2880, I=2880, E=128, k=4),
                              hot_experts=16, hot_bias=1.0),
    "prefill_t2048": dict(shape=LayerShape(T=2048, H=2880, I=2880, E=128, k=4), hot_experts=0),
}
STACK_LAYERS = 36
STACK_TOKENS = (8192, 4)
