"""Seeded synthetic inputs for the routed-expert MoE layer forward.

This module is shared by the CPU oracle (``oracle/``) and the CUDA path's
tests and benchmark. It holds input recipes only and none of the layer's own
arithmetic: no quantiser, no GEMM, no activation, no combine. Where a recipe
needs quantised weights it either returns float weights (to be quantised by
whoever consumes them) or draws the code bytes and scale bytes directly.

Shapes follow the five workloads the MoE layer is measured on:

=====================  =====  ====  ====  ===  ==  ======================
name                   T      H     I     E    k   extra
=====================  =====  ====  ====  ===  ==  ======================
bf16_toy               64     256   256   8    2
mxfp8_small            512    2048  768   64   8
nvfp4_decode           128    7168  2048  256  8
mxfp8_prefill_zipf     8192   7168  2048  256  8   Zipf(1.1) expert bias
nvfp4_shared_norm      4096   4096  1536  128  8   MXFP8 shared I_s=4096,
                                                   RMSNorm eps=1e-6
=====================  =====  ====  ====  ===  ==  ======================

Router: logits ~ N(0, 1) fp32 (plus a per-expert bias for the skewed
workload), softmax in fp64, top-k by descending probability with ties going
to the lower expert id, renormalised to sum 1, stored as fp32. This is the
router that sits upstream of the layer (``fused_topk`` with renormalisation
in vllm.models.qwen4_exp.nvidia.mega_moe, ``Qwen4ExpMegaMoeBlock.forward``);
the layer itself takes ``topk_ids`` / ``topk_weights`` as inputs.

Every tensor draws from its own ``SeedSequence([seed, stream, ...])`` so a
subset (one expert's weights) can be regenerated without the rest.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np

FMT_BF16 = "bf16"
FMT_MXFP8 = "mxfp8"
FMT_NVFP4 = "nvfp4"
FMT_MXFP4 = "mxfp4"

# stream ids (fixed draw order: one independent stream per tensor)
_S_X, _S_LOGITS, _S_W13, _S_W2, _S_WS13, _S_WS2, _S_GAMMA, _S_A2, _S_SF13, _S_SF2, \
    _S_GS, _S_SSF13, _S_SSF2 = range(1, 14)


@dataclass(frozen=True)
class MoeShape:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    fmt: str
    zipf_s: float = 0.0          # >0: add bias_e = -s*log(e+1) to the router logits
    shared_I: int = 0            # 0 = no shared expert
    shared_fmt: str = FMT_MXFP8
    post_norm: bool = False
    norm_eps: float = 1e-6

    @property
    def R(self) -> int:
        return self.T * self.k


WORKLOADS = {
    "bf16_toy": MoeShape("bf16_toy", 64, 256, 256, 8, 2, FMT_BF16),
    "mxfp8_small": MoeShape("mxfp8_small", 512, 2048, 768, 64, 8, FMT_MXFP8),
    "nvfp4_decode": MoeShape("nvfp4_decode", 128, 7168, 2048, 256, 8, FMT_NVFP4),
    "mxfp8_prefill_zipf": MoeShape("mxfp8_prefill_zipf", 8192, 7168, 2048, 256, 8,
                                   FMT_MXFP8, zipf_s=1.1),
    "nvfp4_shared_norm": MoeShape("nvfp4_shared_norm", 4096, 4096, 1536, 128, 8,
                                  FMT_NVFP4, shared_I=4096, shared_fmt=FMT_MXFP8,
                                  post_norm=True),
    # the MXFP8 layer's shape in MXFP4 (the format the pages also list for routed experts)
    "mxfp4_small": MoeShape("mxfp4_small", 512, 2048, 768, 64, 8, FMT_MXFP4),
}
WORKLOAD_ORDER = list(WORKLOADS)


def shrink(shape: MoeShape, **kw) -> MoeShape:
    """The same workload recipe at other sizes (for small parity cases)."""
    return replace(shape, **kw)


def _rng(seed: int, *stream: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([seed, *stream]))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------- activations / router

def hidden_states(shape: MoeShape, seed: int = 0, T: int | None = None) -> np.ndarray:
    """x ~ N(0,1), rounded to bf16; returns uint16 bits [T, H]."""
    T = shape.T if T is None else T
    x = _rng(seed, _S_X).standard_normal((T, shape.H), dtype=np.float32)
    return f32_to_bf16_bits(x)


def router(shape: MoeShape, seed: int = 0, T: int | None = None):
    """Softmax top-k routing with renormalisation.

    Returns ``(topk_ids int32 [T,k], topk_weights fp32 [T,k])``.
    """
    T = shape.T if T is None else T
    logits = _rng(seed, _S_LOGITS).standard_normal((T, shape.E), dtype=np.float32)
    z = logits.astype(np.float64)
    if shape.zipf_s > 0:
        rank = np.arange(1, shape.E + 1, dtype=np.float64)
        z = z + (-shape.zipf_s * np.log(rank))[None, :]
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")[:, : shape.k]
    sel = np.take_along_axis(p, order, axis=1)
    w = sel / sel.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w.astype(np.float32)


def norm_gamma(shape: MoeShape, seed: int = 0) -> np.ndarray:
    """gamma = 1 + N(0, 0.1), fp32 [H]."""
    g = _rng(seed, _S_GAMMA).standard_normal(shape.H, dtype=np.float32)
    return (np.float32(1.0) + np.float32(0.1) * g).astype(np.float32)


# ----------------------------------------------------------------------------- float weights (recipe A)

def float_weight(rows: int, K: int, seed: int, stream: int, index: int = 0) -> np.ndarray:
    """One weight matrix ~ N(0, sigma = 1/sqrt(K)) in fp32, [rows, K]."""
    w = _rng(seed, stream, index).standard_normal((rows, K), dtype=np.float32)
    return (w * np.float32(1.0 / math.sqrt(K))).astype(np.float32)


def routed_float_weights(shape: MoeShape, seed: int = 0):
    """Routed expert weights in fp32: w13 [E, 2I, H] (gate rows, then up rows), w2 [E, H, I]."""
    w13 = np.stack([float_weight(2 * shape.I, shape.H, seed, _S_W13, e) for e in range(shape.E)])
    w2 = np.stack([float_weight(shape.H, shape.I, seed, _S_W2, e) for e in range(shape.E)])
    return w13, w2


def shared_float_weights(shape: MoeShape, seed: int = 0):
    """Shared expert weights in fp32: w13 [2*I_s, H], w2 [H, I_s]."""
    return (float_weight(2 * shape.shared_I, shape.H, seed, _S_WS13),
            float_weight(shape.H, shape.shared_I, seed, _S_WS2))


# ----------------------------------------------------------------------------- direct code draws (recipe B)
#
# For the full-size workloads the checkpoint (codes + block scales) is drawn
# directly: quantising 11e9 fp32 weights on the host is far too slow for a
# test or a benchmark. The byte distributions are chosen so that the decoded
# weights have roughly the 1/sqrt(K) magnitude of recipe A.

def mxfp8_codes(rows: int, K: int, seed: int, stream: int, index: int = 0):
    """E4M3 codes (any finite byte, both signs) [rows, K] and UE8M0 bytes [rows, K/32]."""
    g = _rng(seed, stream, index)
    # one draw per code: 79 magnitudes 0x30..0x7E (1.0 .. 448) times 2 signs
    v = g.integers(0, 158, size=(rows, K), dtype=np.uint16)
    codes = ((0x30 + v % 79) | ((v >= 79).astype(np.uint16) << 7)).astype(np.uint8)
    centre = 127 + int(round(-math.log2(96.0) - 0.5 * math.log2(K)))
    sf = g.integers(centre - 1, centre + 2, size=(rows, K // 32), dtype=np.int64).astype(np.uint8)
    return codes, sf


def mxfp4_codes(rows: int, K: int, seed: int, stream: int, index: int = 0):
    """Packed E2M1 bytes [rows, K/2] (every nibble equally likely, rms value 2.93) and
    UE8M0 bytes [rows, K/32] around 1 / (2.93 sqrt(K)): weights of rms about 1/sqrt(K)."""
    g = _rng(seed, stream, index)
    codes = np.frombuffer(g.bytes(rows * (K // 2)), np.uint8).reshape(rows, K // 2).copy()
    centre = 127 + int(round(-math.log2(2.93) - 0.5 * math.log2(K)))
    sf = g.integers(centre - 1, centre + 2, size=(rows, K // 32), dtype=np.int64).astype(np.uint8)
    return codes, sf


def nvfp4_codes(rows: int, K: int, seed: int, stream: int, index: int = 0):
    """Packed E2M1 bytes [rows, K/2], E4M3 block-scale bytes [rows, K/16], fp32 global scale."""
    g = _rng(seed, stream, index)
    codes = np.frombuffer(g.bytes(rows * (K // 2)), np.uint8).reshape(rows, K // 2).copy()
    sf = g.integers(0x38, 0x59, size=(rows, K // 16), dtype=np.uint16).astype(np.uint8)  # 1.0 .. 16
    gs = np.float32(1.0 / (12.0 * math.sqrt(K)) * g.uniform(0.8, 1.25))
    return codes, sf, gs


@dataclass
class Checkpoint:
    """Routed-expert weights in the checkpoint layout.

    ``w13 [E, 2I, H/vpe]`` (gate rows first, then up rows), ``w2 [E, H, I/vpe]``,
    row-major block scales ``[..., K/g]`` (u8), NVFP4 per-expert fp32 global
    scales ``w13_gs [E]``, ``w2_gs [E]`` and per-expert L2 input scales
    ``w2_input_scale [E]``. BF16 weights are uint16 bit patterns.
    """
    fmt: str
    w13: np.ndarray
    w2: np.ndarray
    w13_sf: np.ndarray | None = None
    w2_sf: np.ndarray | None = None
    w13_gs: np.ndarray | None = None
    w2_gs: np.ndarray | None = None
    w2_input_scale: np.ndarray | None = None


# nominal L2-input amax / 2688 for recipe-B NVFP4 checkpoints (set from the
# oracle's h on sampled rows of these distributions; any positive value is a
# valid input, it only moves how many L2 input codes saturate)
NVFP4_A2_NOMINAL = 2.0e-2


def routed_code_checkpoint(shape: MoeShape, seed: int = 0, experts=None) -> Checkpoint:
    """Recipe-B checkpoint for the routed experts (all experts, or the listed ones
    with zeros elsewhere so indices stay valid)."""
    E, H, I = shape.E, shape.H, shape.I
    sel = range(E) if experts is None else sorted(set(int(e) for e in experts))
    if shape.fmt == FMT_BF16:
        w13 = np.zeros((E, 2 * I, H), np.uint16)
        w2 = np.zeros((E, H, I), np.uint16)
        for e in sel:
            w13[e] = f32_to_bf16_bits(float_weight(2 * I, H, seed, _S_W13, e))
            w2[e] = f32_to_bf16_bits(float_weight(H, I, seed, _S_W2, e))
        return Checkpoint(FMT_BF16, w13, w2)
    if shape.fmt == FMT_MXFP8:
        w13 = np.zeros((E, 2 * I, H), np.uint8)
        w13_sf = np.full((E, 2 * I, H // 32), 127, np.uint8)
        w2 = np.zeros((E, H, I), np.uint8)
        w2_sf = np.full((E, H, I // 32), 127, np.uint8)
        for e in sel:
            w13[e], w13_sf[e] = mxfp8_codes(2 * I, H, seed, _S_W13, e)
            w2[e], w2_sf[e] = mxfp8_codes(H, I, seed, _S_W2, e)
        return Checkpoint(FMT_MXFP8, w13, w2, w13_sf, w2_sf)
    if shape.fmt == FMT_MXFP4:
        w13 = np.zeros((E, 2 * I, H // 2), np.uint8)
        w13_sf = np.full((E, 2 * I, H // 32), 127, np.uint8)
        w2 = np.zeros((E, H, I // 2), np.uint8)
        w2_sf = np.full((E, H, I // 32), 127, np.uint8)
        for e in sel:
            w13[e], w13_sf[e] = mxfp4_codes(2 * I, H, seed, _S_W13, e)
            w2[e], w2_sf[e] = mxfp4_codes(H, I, seed, _S_W2, e)
        return Checkpoint(FMT_MXFP4, w13, w2, w13_sf, w2_sf)
    assert shape.fmt == FMT_NVFP4
    w13 = np.zeros((E, 2 * I, H // 2), np.uint8)
    w13_sf = np.zeros((E, 2 * I, H // 16), np.uint8)
    w2 = np.zeros((E, H, I // 2), np.uint8)
    w2_sf = np.zeros((E, H, I // 16), np.uint8)
    w13_gs = np.ones(E, np.float32)
    w2_gs = np.ones(E, np.float32)
    for e in sel:
        w13[e], w13_sf[e], w13_gs[e] = nvfp4_codes(2 * I, H, seed, _S_W13, e)
        w2[e], w2_sf[e], w2_gs[e] = nvfp4_codes(H, I, seed, _S_W2, e)
    a2 = _rng(seed, _S_A2).uniform(0.8, 1.0, size=E) * NVFP4_A2_NOMINAL
    return Checkpoint(FMT_NVFP4, w13, w2, w13_sf, w2_sf, w13_gs, w2_gs,
                      a2.astype(np.float32))


def shared_code_checkpoint(shape: MoeShape, seed: int = 0) -> Checkpoint:
    """Recipe-B checkpoint for the shared expert (MXFP8 or BF16), E=1."""
    H, S = shape.H, shape.shared_I
    if shape.shared_fmt == FMT_BF16:
        return Checkpoint(FMT_BF16,
                          f32_to_bf16_bits(float_weight(2 * S, H, seed, _S_WS13))[None],
                          f32_to_bf16_bits(float_weight(H, S, seed, _S_WS2))[None])
    w13, w13_sf = mxfp8_codes(2 * S, H, seed, _S_WS13)
    w2, w2_sf = mxfp8_codes(H, S, seed, _S_WS2)
    return Checkpoint(FMT_MXFP8, w13[None], w2[None], w13_sf[None], w2_sf[None])


# ----------------------------------------------------------------------------- recipe B drawn on a device
#
# The same byte ranges as ``mxfp8_codes`` / ``nvfp4_codes``, drawn with a seeded
# torch generator on the device (the benchmark's full-size weights: 11 GB of
# codes are drawn in milliseconds there). Values differ from the host draw;
# the distribution is the same.

def torch_code_checkpoint(shape: MoeShape, seed: int, device, shared: bool = False) -> dict:
    """Checkpoint-layout tensors (routed, or the shared expert with E = 1) on `device`."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + (7 if shared else 3))
    E = 1 if shared else shape.E
    I = shape.shared_I if shared else shape.I
    fmt = shape.shared_fmt if shared else shape.fmt
    H = shape.H

    def ri(lo, hi, size, dtype=torch.uint8):
        return torch.randint(lo, hi, size, generator=g, device=device, dtype=torch.int32).to(dtype)

    out = {}
    for key, rows, K in (("w13", 2 * I, H), ("w2", H, I)):
        if fmt == FMT_BF16:
            w = torch.randn((E, rows, K), generator=g, device=device) * (1.0 / math.sqrt(K))
            out[key] = w.to(torch.bfloat16).view(torch.int16)
        elif fmt == FMT_MXFP8:
            centre = 127 + int(round(-math.log2(96.0) - 0.5 * math.log2(K)))
            out[key] = ri(0x30, 0x7F, (E, rows, K)) | (ri(0, 2, (E, rows, K)) << 7)
            out[key + "_sf"] = ri(centre - 1, centre + 2, (E, rows, K // 32))
        elif fmt == FMT_MXFP4:
            centre = 127 + int(round(-math.log2(2.93) - 0.5 * math.log2(K)))
            out[key] = ri(0, 256, (E, rows, K // 2))
            out[key + "_sf"] = ri(centre - 1, centre + 2, (E, rows, K // 32))
        else:
            out[key] = ri(0, 256, (E, rows, K // 2))
            out[key + "_sf"] = ri(0x38, 0x59, (E, rows, K // 16))
            u = torch.rand((E,), generator=g, device=device) * 0.45 + 0.8
            out[key + "_gs"] = (u * (1.0 / (12.0 * math.sqrt(K)))).to(torch.float32)
    if fmt == FMT_NVFP4 and not shared:
        out["w2_input_scale"] = (torch.rand((E,), generator=g, device=device) * 0.2 + 0.8) * NVFP4_A2_NOMINAL
    return out
