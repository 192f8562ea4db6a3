"""Oracle forward of the routed-expert MoE layer (plus optional shared expert and post-norm).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The unfused pipeline of vllm.model_executor.layers.fused_moe,
``DeepGemmExperts.apply``: permute -> grouped L1 GEMM -> gated activation ->
requantise the L2 input -> grouped L2 GEMM -> unpermute with a top-k-weighted
reduce. Formats and scales follow vllm.model_executor.layers.fused_moe.
deep_gemm_mega_moe (module docstring; ``DeepGemmMegaMoEExperts._create_weights``:
``w13_weight_scale_2`` is the L1 alpha, the w2 global scale times the L2
activation scale is the L2 alpha; ``_record_global_scale``: the L2 input
scale is the max of ``w2_input_scale`` over experts, or 1.0). The activation
is ``MegaMoEActivation``'s swiglu. The shared expert is one more always-on
SwiGLU MLP added to the routed output (``DeepGemmMegaMoEExperts.forward``,
``y += shared_experts(hidden)``), and the post-expert RMSNorm applies gamma
verbatim (vllm.models.muse_spark.nvidia.mega_moe, ``finalize_weights`` /
``forward_prepared``).

All GEMMs and the combine accumulate in fp64 on dequantised operands.
Readings where the pages are silent:
  * a clamp (if any) applies to gate and up before alpha and beta;
  * the L2 input is quantised from the fp32 value of h (the precision the
    kernel holds it in), so a quantised code is decided in fp32;
  * the combine sums slots in ascending j; masked slots (id -1) add nothing;
  * the final value is rounded once to bf16.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import formats as F
from .routing import permute

BF16, MXFP8, NVFP4, MXFP4 = "bf16", "mxfp8", "nvfp4", "mxfp4"


@dataclass
class Activation:
    """gate * sigmoid(alpha * gate) * (up + beta), after clamping gate from above and
    up symmetrically to ``clamp`` (MegaMoEActivation, name "swiglu")."""
    alpha: float = 1.0
    beta: float = 0.0
    clamp: float | None = None


def swiglu(g, u, act: Activation = Activation()) -> np.ndarray:
    g = np.asarray(g, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    if act.clamp is not None:
        g = np.minimum(g, act.clamp)
        u = np.clip(u, -act.clamp, act.clamp)
    with np.errstate(over="ignore"):
        sig = 1.0 / (1.0 + np.exp(-act.alpha * g))
    return g * sig * (u + act.beta)


@dataclass
class ExpertWeights:
    """One format's checkpoint tensors (see ``synthetic.Checkpoint``) for E experts."""
    fmt: str
    w13: np.ndarray
    w2: np.ndarray
    w13_sf: np.ndarray | None = None
    w2_sf: np.ndarray | None = None
    w13_gs: np.ndarray | None = None
    w2_gs: np.ndarray | None = None
    _cache: dict = field(default_factory=dict, repr=False)

    def _deq(self, codes, sf, gs):
        if self.fmt == BF16:
            return F.bf16_bits_to_f64(codes)
        if self.fmt == MXFP8:
            return F.mxfp8_dequantize(codes, sf)
        if self.fmt == MXFP4:
            return F.mxfp4_dequantize(codes, sf)
        return F.nvfp4_dequantize(codes, sf, gs)

    def w13_of(self, e: int) -> np.ndarray:
        """Dequantised [2I, H] (gate rows, then up rows)."""
        gs = None if self.w13_gs is None else self.w13_gs[e]
        return self._deq(self.w13[e], None if self.w13_sf is None else self.w13_sf[e], gs)

    def w2_of(self, e: int) -> np.ndarray:
        """Dequantised [H, I]."""
        gs = None if self.w2_gs is None else self.w2_gs[e]
        return self._deq(self.w2[e], None if self.w2_sf is None else self.w2_sf[e], gs)


def quantize_weights(fmt: str, w13_f, w2_f) -> ExpertWeights:
    """Checkpoint tensors from fp32 weights: w13 [E, 2I, H], w2 [E, H, I].

    NVFP4: one global scale per expert per tensor, amax over all of w13[e]
    (gate and up share it: one L1 scale per expert) and over w2[e].
    """
    w13_f = np.asarray(w13_f, dtype=np.float32)
    w2_f = np.asarray(w2_f, dtype=np.float32)
    if fmt == BF16:
        return ExpertWeights(BF16, F.bf16_bits(w13_f), F.bf16_bits(w2_f))
    if fmt == MXFP8:
        c13, s13 = F.mxfp8_quantize(w13_f)
        c2, s2 = F.mxfp8_quantize(w2_f)
        return ExpertWeights(MXFP8, c13, c2, s13, s2)
    if fmt == MXFP4:
        c13, s13 = F.mxfp4_quantize(w13_f)
        c2, s2 = F.mxfp4_quantize(w2_f)
        return ExpertWeights(MXFP4, c13, c2, s13, s2)
    E = w13_f.shape[0]
    gs13 = F.nvfp4_global_scale(np.abs(w13_f).reshape(E, -1).max(axis=1))
    gs2 = F.nvfp4_global_scale(np.abs(w2_f).reshape(E, -1).max(axis=1))
    c13, s13 = F.nvfp4_quantize(w13_f, gs13[:, None])
    c2, s2 = F.nvfp4_quantize(w2_f, gs2[:, None])
    return ExpertWeights(NVFP4, c13, c2, s13, s2, gs13, gs2)


# ----------------------------------------------------------------------------- dispatch (activation) quantisation

@dataclass
class Dispatched:
    fmt: str
    x: np.ndarray                  # dequantised [T, H] fp64
    codes: np.ndarray | None = None
    sf: np.ndarray | None = None
    x_scale: np.ndarray | None = None   # NVFP4 per-token fp32 scale [T]


def dispatch_quantize(x_bits, fmt: str) -> Dispatched:
    """Quantise each token once (bf16: no change; MXFP8 / MXFP4: 1x32 UE8M0; NVFP4:
    per-token fp32 scale amax/2688, then 1x16 E4M3 block scales)."""
    x = F.bf16_bits_to_f64(x_bits)
    if fmt == BF16:
        return Dispatched(BF16, x)
    if fmt == MXFP8:
        codes, sf = F.mxfp8_quantize(x)
        return Dispatched(MXFP8, F.mxfp8_dequantize(codes, sf), codes, sf)
    if fmt == MXFP4:
        codes, sf = F.mxfp4_quantize(x)
        return Dispatched(MXFP4, F.mxfp4_dequantize(codes, sf), codes, sf)
    gs = F.nvfp4_global_scale(np.abs(x).max(axis=1).astype(np.float32))
    codes, sf = F.nvfp4_quantize(x, gs)
    return Dispatched(NVFP4, F.nvfp4_dequantize(codes, sf, gs), codes, sf, gs)


def l2_input_quantize(h, fmt: str, a2: float | None = None) -> np.ndarray:
    """Requantise the L2 input (held in fp32) and return its dequantised value (fp64)."""
    h32 = np.asarray(h, dtype=np.float64).astype(np.float32).astype(np.float64)
    if fmt == BF16:
        return F.bf16_round(h32)
    if fmt == MXFP8:
        return F.mxfp8_dequantize(*F.mxfp8_quantize(h32))
    if fmt == MXFP4:
        return F.mxfp4_dequantize(*F.mxfp4_quantize(h32))
    gs = np.float32(a2)
    codes, sf = F.nvfp4_quantize(h32, gs)
    return F.nvfp4_dequantize(codes, sf, gs)


def l2_input_codes(h32, fmt: str, a2: float | None = None):
    """The L2 input codes and scale bytes of fp32 h (for bit-exact checks)."""
    h32 = np.asarray(h32, dtype=np.float32).astype(np.float64)
    if fmt == BF16:
        return F.bf16_bits(h32), None
    if fmt == MXFP8:
        return F.mxfp8_quantize(h32)
    if fmt == MXFP4:
        return F.mxfp4_quantize(h32)
    return F.nvfp4_quantize(h32, np.float32(a2))


def l2_activation_scale(w2_input_scale) -> float:
    """One L2 input scale for all experts: max over experts, or 1.0 if that is 0."""
    m = float(np.max(np.asarray(w2_input_scale, dtype=np.float32)))
    return np.float32(m if m != 0.0 else 1.0)


# ----------------------------------------------------------------------------- expert MLP

def expert_mlp(x_rows, w13, w2, fmt: str, act: Activation, a2=None, return_h=False):
    """One expert on its rows: g|u = x W13^T, h = swiglu(g, u), y = requant(h) W2^T (fp64)."""
    I = w13.shape[0] // 2
    gu = np.asarray(x_rows, dtype=np.float64) @ w13.T
    h = swiglu(gu[:, :I], gu[:, I:], act)
    y = l2_input_quantize(h, fmt, a2) @ w2.T
    return (y, h) if return_h else y


# ----------------------------------------------------------------------------- layer

@dataclass
class Layer:
    """Everything ``moe_forward`` takes besides the activations and the routing."""
    num_experts: int
    top_k: int
    routed: ExpertWeights
    act: Activation = field(default_factory=Activation)
    a2: float | None = None                  # NVFP4: the L2 input scale (fp32)
    shared: ExpertWeights | None = None      # E = 1
    norm_gamma: np.ndarray | None = None     # [H] fp32, applied verbatim
    norm_eps: float = 1e-6


def forward(layer: Layer, x_bits, topk_ids, topk_weights, tokens=None, block_m: int = 128,
            return_parts: bool = False):
    """Output bf16 bits [len(tokens), H] of the layer for the listed tokens (default: all).

    Every token is independent, so a subset is computed exactly as it would be
    in the full batch.
    """
    x_bits = np.asarray(x_bits)
    ids = np.asarray(topk_ids)
    w = np.asarray(topk_weights, dtype=np.float32).astype(np.float64)
    T, k = ids.shape
    toks = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    sub_ids = ids[toks]
    disp = dispatch_quantize(x_bits[toks], layer.routed.fmt)

    # permutation over the selected tokens (rows grouped by expert, stable)
    _, off, src, inv = permute(sub_ids, layer.num_experts, block_m)
    H = layer.routed.w2.shape[1]
    y_rows = np.zeros((len(src), H), dtype=np.float64)
    h_rows = {}
    for e in range(layer.num_experts):
        rows = [r for r in range(off[e], off[e + 1]) if src[r] >= 0]
        if not rows:
            continue
        slots = src[rows]
        xr = disp.x[slots // k]
        y, h = expert_mlp(xr, layer.routed.w13_of(e), layer.routed.w2_of(e),
                          layer.routed.fmt, layer.act, layer.a2, return_h=True)
        y_rows[rows] = y
        if return_parts:
            for r, hh in zip(rows, h):
                h_rows[r] = hh

    z = _combine_shared_norm(layer, x_bits[toks], w[toks], inv, y_rows)
    out = F.bf16_bits(z)
    if return_parts:
        return out, dict(z=z, dispatched=disp, off=off, src=src, inv=inv, h=h_rows, y=y_rows)
    return out


def _combine_shared_norm(layer: Layer, x_bits_sub, w_sub, inv, y_rows) -> np.ndarray:
    """z[i] = sum over j (ascending) of w[i, j] * y[inv[i, j]] (masked slots add nothing), plus the
    shared expert, then the post-norm: the layer's value before its final bf16 rounding (fp64)."""
    H = y_rows.shape[1]
    n, k = inv.shape
    z = np.zeros((n, H), dtype=np.float64)
    for i in range(n):
        for j in range(k):
            r = inv[i, j]
            if r >= 0:
                z[i] += w_sub[i, j] * y_rows[r]
    if layer.shared is not None:
        sd = dispatch_quantize(x_bits_sub, layer.shared.fmt)
        z += expert_mlp(sd.x, layer.shared.w13_of(0), layer.shared.w2_of(0),
                        layer.shared.fmt, Activation())
    if layer.norm_gamma is not None:
        gamma = np.asarray(layer.norm_gamma, dtype=np.float32).astype(np.float64)
        rms = np.sqrt(np.mean(z * z, axis=1, keepdims=True) + layer.norm_eps)
        z = z / rms * gamma[None, :]
    return z


def forward_from_l2_inputs(layer: Layer, x_bits, topk_ids, topk_weights, token: int, l2_inputs) -> np.ndarray:
    """The layer's value before its final bf16 rounding (fp64) for one token, continuing from given
    dequantised L2 inputs: ``l2_inputs[j]`` is slot j's requantised h (fp64 [I]; ignored for masked
    slots). The same L2 GEMM, combine, shared expert and norm as ``forward``; used where a rounding
    decision of the L2-input quantiser is a tie within fp32 accumulation noise, so that either
    neighbouring code is a correct result."""
    ids = np.asarray(topk_ids)
    w = np.asarray(topk_weights, dtype=np.float32).astype(np.float64)
    k = ids.shape[1]
    H = layer.routed.w2.shape[1]
    y_rows = np.zeros((k, H), dtype=np.float64)
    inv = np.full((1, k), -1, dtype=np.int64)
    for j in range(k):
        e = int(ids[token, j])
        if e < 0:
            continue
        y_rows[j] = np.asarray(l2_inputs[j], dtype=np.float64) @ layer.routed.w2_of(e).T
        inv[0, j] = j
    x_bits = np.asarray(x_bits)
    return _combine_shared_norm(layer, x_bits[[token]], w[[token]], inv, y_rows)[0]


def forward_batched(layer: Layer, x_bits, expert_num_tokens, exact: bool = False) -> np.ndarray:
    """The routed experts on the batched (masked) layout (vllm.model_executor.layers.fused_moe,
    ``BatchedDeepGemmExperts.apply``): ``x_bits`` bf16 bits [E, M, H] holds each expert's rows
    in its own slab, of which the first ``expert_num_tokens[e]`` are used. Each used row is
    quantised on its own (the dispatch quantiser), then L1 -> activation -> L2 requant -> L2
    of its expert. Returns bf16 bits [E, M, H] with the unused rows zero (``exact``: the fp64
    values before that rounding). No routing weights, no combine, no shared expert, no norm.
    """
    x_bits = np.asarray(x_bits)
    E, M, H = x_bits.shape
    counts = np.asarray(expert_num_tokens, dtype=np.int64)
    out = np.zeros((E, M, H), dtype=np.float64 if exact else np.uint16)
    for e in range(E):
        n = int(counts[e])
        if n <= 0:
            continue
        d = dispatch_quantize(x_bits[e, :n], layer.routed.fmt)
        y = expert_mlp(d.x, layer.routed.w13_of(e), layer.routed.w2_of(e), layer.routed.fmt, layer.act, layer.a2)
        out[e, :n] = y if exact else F.bf16_bits(y)
    return out


def calibrate_a2(layer: Layer, x_bits, topk_ids, block_m: int = 128) -> np.float32:
    """NVFP4 L2 input scale from per-expert w2_input_scale = amax(h over the expert's rows)/2688,
    then the max over experts (the scale the layer takes for all experts)."""
    x_bits = np.asarray(x_bits)
    ids = np.asarray(topk_ids)
    k = ids.shape[1]
    disp = dispatch_quantize(x_bits, layer.routed.fmt)
    _, off, src, _ = permute(ids, layer.num_experts, block_m)
    I = layer.routed.w13.shape[1] // 2
    per_expert = np.zeros(layer.num_experts, dtype=np.float32)
    for e in range(layer.num_experts):
        rows = [r for r in range(off[e], off[e + 1]) if src[r] >= 0]
        if not rows:
            continue
        gu = disp.x[src[rows] // k] @ layer.routed.w13_of(e).T
        h = swiglu(gu[:, :I], gu[:, I:], layer.act).astype(np.float32)
        per_expert[e] = F.nvfp4_global_scale(np.abs(h).max())
    return l2_activation_scale(per_expert)
