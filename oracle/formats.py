"""Oracle number formats: E2M1, E4M3, UE8M0, BF16 and the MXFP8 / MXFP4 / NVFP4 quantisers.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this module;
only tests, the smoke check and the benchmark's CPU-baseline leg do.

Formats (vllm.model_executor.layers.fused_moe.deep_gemm_mega_moe, module
docstring): MX weights and activations carry one UE8M0 scale per 1x32 block;
NVFP4 weights carry one E4M3 scale per 1x16 block plus a per-expert FP32
global scale, and NVFP4 dispatch scales each token by its own FP32 scale.

Decoding goes through explicit tables built from each format's closed form
(sign, biased exponent, mantissa). Encoding rounds to the nearest
representable value, ties to the even code, and saturates to the largest
finite magnitude. Pages are silent on:
  * the nibble order of packed E2M1: element 2i is the low nibble,
    element 2i+1 the high nibble;
  * the NVFP4 scale arithmetic: the plain two-level recipe in fp32 (see
    ``nvfp4_quantize``), whose global scale is amax / (448 * 6);
  * the UE8M0 byte of an all-zero block: 127 (scale 1.0);
  * the MX block exponent: the smallest e with amax <= (largest element value) * 2^e,
    i.e. 2^ceil(log2(amax / 448)) for MXFP8 (as the MXFP8 workloads state) and,
    by the same rule, 2^ceil(log2(amax / 6)) for MXFP4, so no element saturates.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32

# ----------------------------------------------------------------------------- decode tables


def _e2m1_value(code: int) -> float:
    """E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit, no inf/NaN."""
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1.0 + m / 2.0)
    return -mag if s else mag


def _e4m3_value(code: int) -> float:
    """E4M3 (fn): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; S.1111.111 is NaN, no inf."""
    s, e, m = (code >> 7) & 1, (code >> 3) & 0xF, code & 7
    if e == 0xF and m == 7:
        return float("nan")
    mag = m * 2.0 ** -9 if e == 0 else 2.0 ** (e - 7) * (1.0 + m / 8.0)
    return -mag if s else mag


def _ue8m0_value(code: int) -> float:
    """UE8M0: an unsigned biased exponent, value 2^(b-127); 0xFF is NaN."""
    return float("nan") if code == 0xFF else 2.0 ** (code - 127)


E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)
E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)
UE8M0_TABLE = np.array([_ue8m0_value(c) for c in range(256)], dtype=np.float64)

E4M3_MAX = 448.0
E2M1_MAX = 6.0
E4M3_MAX_CODE = 0x7E     # largest finite magnitude code
E2M1_MAX_CODE = 0x7


# ----------------------------------------------------------------------------- encoders (RNE, saturating)

def _encode_magnitude(a: np.ndarray, pos_table: np.ndarray) -> np.ndarray:
    """Nearest magnitude code for |v| (ties to the even code), saturating at the top code.

    ``pos_table[c]`` is the (strictly increasing) value of magnitude code c.
    """
    top = len(pos_table) - 1
    a = np.minimum(a, pos_table[top])
    hi = np.searchsorted(pos_table, a, side="left")          # first code with value >= a
    hi = np.clip(hi, 0, top)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - pos_table[lo]
    d_hi = pos_table[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    return np.where(take_hi, hi, lo).astype(np.uint8)


def e4m3_encode(v) -> np.ndarray:
    """Round each value to E4M3 (nearest, ties to even, saturate to +-448). NaN is rejected."""
    v = np.asarray(v, dtype=np.float64)
    if np.isnan(v).any():
        raise ValueError("e4m3_encode: NaN input")
    mag = _encode_magnitude(np.abs(v), E4M3_TABLE[: E4M3_MAX_CODE + 1])
    return (mag | (np.signbit(v).astype(np.uint8) << 7)).astype(np.uint8)


def e2m1_encode(v) -> np.ndarray:
    """Round each value to E2M1 (nearest, ties to even, saturate to +-6); one code per byte."""
    v = np.asarray(v, dtype=np.float64)
    if np.isnan(v).any():
        raise ValueError("e2m1_encode: NaN input")
    mag = _encode_magnitude(np.abs(v), E2M1_TABLE[: E2M1_MAX_CODE + 1])
    return (mag | (np.signbit(v).astype(np.uint8) << 3)).astype(np.uint8)


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """Two E2M1 codes per byte along the last axis: element 2i low nibble, 2i+1 high nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


# ----------------------------------------------------------------------------- BF16

def bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_round(v) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (8 significant bits, ties to even)."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)                                   # v = m * 2^e, 0.5 <= |m| < 1
    normal = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    sub = np.ldexp(np.rint(np.ldexp(v, 133)), -133)      # bf16 subnormal quantum 2^-133
    return np.where(np.abs(v) < 2.0 ** -126, sub, normal)


def bf16_bits(v) -> np.ndarray:
    """bf16 bit patterns of the rounded values."""
    r = bf16_round(v).astype(np.float32)                 # exact: a bf16 value is an fp32 value
    return (r.view(np.uint32) >> 16).astype(np.uint16)


# ----------------------------------------------------------------------------- MXFP8 (E4M3 + UE8M0 per 1x32)

MX_BLOCK = 32


def mx_exponent(amax, vmax: float) -> np.ndarray:
    """The smallest integer e with amax <= vmax * 2^e (i.e. ceil(log2(amax / vmax))),
    decided exactly against that inequality; 0 for amax == 0; clamped to [-127, 127]."""
    amax = np.asarray(amax, dtype=np.float64)
    pos = amax > 0
    safe = np.where(pos, amax, vmax)
    e = np.ceil(np.log2(safe / vmax)).astype(np.int64)
    for _ in range(3):                                   # exact fix-up of the float log2
        e = np.where(safe > np.ldexp(vmax, e), e + 1, e)
        e = np.where(safe <= np.ldexp(vmax, e - 1), e - 1, e)
    e = np.where(pos, e, 0)
    return np.clip(e, -127, 127)


def ue8m0_exponent(amax) -> np.ndarray:
    """MXFP8 block exponent: the smallest integer e with amax <= 448 * 2^e."""
    return mx_exponent(amax, E4M3_MAX)


def mxfp8_quantize(x) -> tuple[np.ndarray, np.ndarray]:
    """Quantise rows of x (last axis K, a multiple of 32) to MXFP8.

    Per 1x32 block: e = ue8m0_exponent(amax), code = E4M3(x * 2^-e), scale byte = e + 127.
    Returns (codes u8 [..., K], scale bytes u8 [..., K/32]).
    """
    x = np.asarray(x, dtype=np.float64)
    K = x.shape[-1]
    if K % MX_BLOCK:
        raise ValueError("mxfp8_quantize: K must be a multiple of 32")
    xb = x.reshape(x.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    e = ue8m0_exponent(np.abs(xb).max(axis=-1))
    codes = e4m3_encode(xb * np.ldexp(1.0, -e)[..., None])
    return codes.reshape(x.shape), (e + 127).astype(np.uint8)


def mxfp8_dequantize(codes, sf) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    K = codes.shape[-1]
    v = E4M3_TABLE[codes].reshape(codes.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    return (v * UE8M0_TABLE[np.asarray(sf, dtype=np.uint8)][..., None]).reshape(codes.shape)


# ----------------------------------------------------------------------------- MXFP4 (E2M1 + UE8M0 per 1x32)

E2M1_MAX = 6.0


def mxfp4_quantize(x) -> tuple[np.ndarray, np.ndarray]:
    """Quantise rows of x (last axis K, a multiple of 32) to MXFP4.

    Per 1x32 block: e = the smallest integer with amax <= 6 * 2^e, code = E2M1(x * 2^-e)
    (nearest, ties to even), scale byte = e + 127. Returns (codes packed two per byte,
    element 2i in the low nibble, u8 [..., K/2]; scale bytes u8 [..., K/32]).
    """
    x = np.asarray(x, dtype=np.float64)
    K = x.shape[-1]
    if K % MX_BLOCK:
        raise ValueError("mxfp4_quantize: K must be a multiple of 32")
    xb = x.reshape(x.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    e = mx_exponent(np.abs(xb).max(axis=-1), E2M1_MAX)
    codes = e2m1_encode(xb * np.ldexp(1.0, -e)[..., None])
    return pack_e2m1(codes.reshape(x.shape)), (e + 127).astype(np.uint8)


def mxfp4_dequantize(packed, sf) -> np.ndarray:
    codes = unpack_e2m1(packed)
    K = codes.shape[-1]
    v = E2M1_TABLE[codes].reshape(codes.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    return (v * UE8M0_TABLE[np.asarray(sf, dtype=np.uint8)][..., None]).reshape(codes.shape)


# ----------------------------------------------------------------------------- NVFP4 (E2M1 + E4M3 per 1x16 + FP32 global)

NV_BLOCK = 16
NV_GLOBAL_DIV = F32(448.0 * 6.0)      # 2688: the largest E4M3 scale times the largest E2M1 value


def nvfp4_global_scale(amax) -> np.ndarray:
    """FP32 global (per-token or per-expert) scale amax / 2688; 1.0 when amax == 0."""
    a = np.asarray(amax, dtype=F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        gs = (a / NV_GLOBAL_DIV).astype(F32)
    return np.where(a > 0, gs, F32(1.0)).astype(F32)


def nvfp4_quantize(x, gs) -> tuple[np.ndarray, np.ndarray]:
    """Quantise rows of x (last axis K, a multiple of 16) to NVFP4 under global scale gs.

    ``x`` must hold fp32-representable values; ``gs`` broadcasts against
    ``x.shape[:-1]``. All scale arithmetic is fp32 with round-to-nearest:
      sb   = E4M3(amax_b / (gs * 6))        one block scale per 1x16 block
      eff  = value(sb) * gs
      code = E2M1(x / eff), or 0 when eff == 0
    Returns (packed codes u8 [..., K/2], block-scale bytes u8 [..., K/16]).
    """
    x32 = np.asarray(x, dtype=np.float64).astype(F32)
    if not np.array_equal(x32.astype(np.float64), np.asarray(x, dtype=np.float64)):
        raise ValueError("nvfp4_quantize: inputs must be fp32-representable")
    K = x32.shape[-1]
    if K % NV_BLOCK:
        raise ValueError("nvfp4_quantize: K must be a multiple of 16")
    gs = np.broadcast_to(np.asarray(gs, dtype=F32), x32.shape[:-1])
    xb = x32.reshape(x32.shape[:-1] + (K // NV_BLOCK, NV_BLOCK))
    amax_b = np.abs(xb).max(axis=-1)
    denom = (gs * F32(6.0)).astype(F32)
    ratio = (amax_b / denom[..., None]).astype(F32)
    sb = e4m3_encode(ratio)
    eff = (E4M3_TABLE[sb].astype(F32) * gs[..., None]).astype(F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (xb / eff[..., None]).astype(F32)
    q = np.where(eff[..., None] > 0, q, F32(0.0))
    codes = np.where(eff[..., None] > 0, e2m1_encode(q), np.uint8(0)).astype(np.uint8)
    return pack_e2m1(codes.reshape(x32.shape)), sb


def nvfp4_dequantize(packed, sb, gs) -> np.ndarray:
    """code * value(sb) * gs, in fp64 (exact)."""
    codes = unpack_e2m1(packed)
    K = codes.shape[-1]
    v = E2M1_TABLE[codes].reshape(codes.shape[:-1] + (K // NV_BLOCK, NV_BLOCK))
    s = E4M3_TABLE[np.asarray(sb, dtype=np.uint8)] * np.asarray(gs, dtype=np.float64)[..., None]
    return (v * s[..., None]).reshape(codes.shape)
