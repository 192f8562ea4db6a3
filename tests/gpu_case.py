"""Shared helpers of the GPU parity tests: build a seeded case, run it through the
C ABI (serving_topk_permute_gb300), run the oracle on the same inputs, compare.

Two weight recipes:
  float  fp32 weights ~ N(0, 1/sqrt(K)) quantised by the oracle's quantiser
         (reduced sizes; the exact recipe of the workloads)
  codes  checkpoint bytes drawn directly (synthetic.routed_code_checkpoint) for
         the experts the sampled tokens touch; every other expert gets random
         device bytes, which only feed outputs that are not compared
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import synthetic as S
from oracle import formats as OF
from oracle import moe as OM
import serving_topk_permute_gb300 as pkg

# max |gpu - oracle| <= REL * rms(oracle) + ABS
REL = {"bf16": 2e-2, "mxfp8": 2e-2, "nvfp4": 5e-2, "mxfp4": 5e-2}   # MXFP4: 4-bit elements like NVFP4
ABS = 1e-3


def dev():
    return torch.device("cuda", torch.cuda.current_device())


def to_dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev())
    return torch.from_numpy(a).to(dev())


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    return to_dev(bits.astype(np.uint16)).view(torch.bfloat16)


@dataclass
class Case:
    shape: S.MoeShape
    x: np.ndarray                    # bf16 bits [T, H]
    ids: np.ndarray                  # int32 [T, k]
    w: np.ndarray                    # fp32 [T, k]
    layer: OM.Layer                  # oracle side (routed / shared checkpoints, a2, gamma)
    touched: list | None = None      # codes recipe: experts with real weights
    extra: dict = field(default_factory=dict)


def float_case(shape: S.MoeShape, seed: int = 0, ids=None, w=None) -> Case:
    x = S.hidden_states(shape, seed)
    if ids is None:
        ids, w = S.router(shape, seed)
    w13f, w2f = S.routed_float_weights(shape, seed)
    routed = OM.quantize_weights(shape.fmt, w13f, w2f)
    layer = OM.Layer(shape.E, shape.k, routed)
    if shape.fmt == "nvfp4":
        layer.a2 = OM.calibrate_a2(layer, x, ids)
    if shape.shared_I:
        s13, s2 = S.shared_float_weights(shape, seed)
        layer.shared = OM.quantize_weights(shape.shared_fmt, s13[None], s2[None])
    if shape.post_norm:
        layer.norm_gamma = S.norm_gamma(shape, seed)
        layer.norm_eps = shape.norm_eps
    return Case(shape, x, np.asarray(ids, np.int32), np.asarray(w, np.float32), layer)


def code_case(shape: S.MoeShape, sample_tokens, seed: int = 0) -> Case:
    x = S.hidden_states(shape, seed)
    ids, w = S.router(shape, seed)
    touched = sorted(set(int(e) for e in ids[sample_tokens].reshape(-1) if e >= 0))
    ck = S.routed_code_checkpoint(shape, seed, experts=touched)
    routed = OM.ExpertWeights(ck.fmt, ck.w13, ck.w2, ck.w13_sf, ck.w2_sf, ck.w13_gs, ck.w2_gs)
    layer = OM.Layer(shape.E, shape.k, routed)
    if shape.fmt == "nvfp4":
        layer.a2 = OM.l2_activation_scale(ck.w2_input_scale)
    if shape.shared_I:
        sc = S.shared_code_checkpoint(shape, seed)
        layer.shared = OM.ExpertWeights(sc.fmt, sc.w13, sc.w2, sc.w13_sf, sc.w2_sf)
    if shape.post_norm:
        layer.norm_gamma = S.norm_gamma(shape, seed)
        layer.norm_eps = shape.norm_eps
    return Case(shape, x, ids, w, layer, touched=touched)


def _ckpt_dev(ew: OM.ExpertWeights, touched=None) -> dict:
    out = {}
    for key in ("w13", "w13_sf", "w2", "w2_sf", "w13_gs", "w2_gs"):
        a = getattr(ew, key)
        if a is None:
            continue
        if touched is None or key.endswith("_gs"):
            out[key] = to_dev(a)
            continue
        if a.dtype == np.uint16:
            t = torch.randint(-2 ** 15, 2 ** 15, a.shape, dtype=torch.int16, device=dev())
        else:
            t = torch.randint(0, 256, a.shape, dtype=torch.uint8, device=dev())
        for e in touched:
            t[e] = to_dev(a[e])
        out[key] = t
    return out


def layer_config(case: Case, debug_h=False, max_tokens=None, tile=0, cta="auto", split=False) -> pkg.LayerConfig:
    s = case.shape
    act = case.layer.act
    return pkg.LayerConfig(s.E, s.H, s.I, s.k, max_tokens or max(case.x.shape[0], 1), s.fmt,
                           act_alpha=act.alpha, act_beta=act.beta, act_clamp=act.clamp,
                           shared_inter=s.shared_I, shared_fmt=s.shared_fmt, post_norm=s.post_norm,
                           norm_eps=s.norm_eps, debug_h=debug_h, tile=tile, cta=cta, split_gemm=split)


@dataclass
class GpuRun:
    plan: pkg.Plan
    out: torch.Tensor
    workspace: torch.Tensor
    kweights: dict
    kshared: dict | None
    inputs: dict


# GEMM variants: L1 and L2 in one kernel (256-wide single-CTA tiles, the default); two
# single-CTA kernels with 128- or 256-wide tiles; CTA pairs (256 x 256 tiles, two kernels)
MODES = {"fused": dict(tile=256, cta="single"), "single128": dict(tile=128, cta="single"),
         "split256": dict(tile=256, cta="single", split=True), "pair": dict(cta="pair")}


def run_gpu(case: Case, debug_h=False, max_tokens=None, tile=0, cta="auto", split=False) -> GpuRun:
    plan = pkg.Plan(layer_config(case, debug_h, max_tokens, tile, cta, split))
    ck = _ckpt_dev(case.layer.routed, case.touched)
    kw = plan.transform_weights(ck)
    ks = None
    if case.layer.shared is not None:
        ks = plan.transform_shared_weights(_ckpt_dev(case.layer.shared))
    T = case.x.shape[0]
    inputs = dict(hidden=bf16_dev(case.x), topk_ids=to_dev(case.ids.astype(np.int32)),
                  topk_weights=to_dev(case.w.astype(np.float32)))
    a2 = None
    if case.shape.fmt == "nvfp4":
        a2 = torch.tensor([np.float32(case.layer.a2)], dtype=torch.float32, device=dev())
    gamma = None if case.layer.norm_gamma is None else to_dev(np.asarray(case.layer.norm_gamma, np.float32))
    ws = plan.alloc_workspace(T)
    out = plan.forward(inputs["hidden"], inputs["topk_ids"], inputs["topk_weights"], kw, l2_act_scale=a2,
                       shared=ks, norm_gamma=gamma, workspace=ws)
    torch.cuda.synchronize()
    inputs.update(a2=a2, gamma=gamma)
    return GpuRun(plan, out, ws, kw, ks, inputs)


def out_f64(run: GpuRun) -> np.ndarray:
    return run.out.float().cpu().numpy().astype(np.float64)


def oracle_out(case: Case, tokens=None) -> np.ndarray:
    """The oracle's output before its final bf16 rounding (fp64).

    The GPU's bf16 output is compared with this exact value: two correct
    results that differ by 1e-4 relative before the final rounding can land on
    neighbouring bf16 values, and one bf16 step at |z| > 2.56 rms is already
    more than 2e-2 rms."""
    return OM.forward(case.layer, case.x, case.ids, case.w, tokens=tokens, return_parts=True)[1]["z"]


def half_ulp_bf16(z: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 values around |z| (8 significant bits)."""
    e = np.floor(np.log2(np.maximum(np.abs(z), 2.0 ** -126)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def assert_close(got: np.ndarray, want: np.ndarray, fmt: str, what=""):
    """max |gpu - oracle| <= REL * rms(oracle) + ABS, for the value before the final bf16 rounding.

    `want` is the oracle's exact (fp64) output; the GPU's output is bf16, whose own
    rounding (at most half a bf16 step of the output, which the oracle's bf16 result
    carries too) is allowed on top: at |z| > 5 rms half a step alone exceeds 2e-2 rms."""
    rms = float(np.sqrt(np.mean(want ** 2))) if want.size else 0.0
    tol = REL[fmt] * rms + ABS
    assert np.isfinite(got).all(), f"{what}: non-finite GPU output"
    if not want.size:
        return 0.0, tol
    excess = np.abs(got - want) - half_ulp_bf16(want)
    err = float(excess.max())
    assert err <= tol, f"{what}: max |gpu - oracle| - half bf16 step = {err:.4g} > {tol:.4g} (rms {rms:.4g})"
    return err, tol


def region_i32(run: GpuRun, T: int, name: str) -> np.ndarray:
    return run.plan.region(run.workspace, T, name).cpu().numpy().view(np.int32)


def region_u8(run: GpuRun, T: int, name: str) -> np.ndarray:
    return run.plan.region(run.workspace, T, name).cpu().numpy()


def unpack_act_sf(atoms: np.ndarray, rows: np.ndarray, n_blocks: int, S: int) -> np.ndarray:
    """Scale bytes [len(rows), n_blocks] from activation scale atoms laid out
    [row tile][K stage][S][512] with row 32j+i / scale b at byte 16i + 4j + b."""
    nks = n_blocks // (4 * S)
    r = rows[:, None].astype(np.int64)
    kb = np.arange(n_blocks)[None, :]
    mt, m = r // 128, r % 128
    ks, s, b = kb // (4 * S), (kb // 4) % S, kb % 4
    off = ((mt * nks + ks) * S + s) * 512 + (m % 32) * 16 + (m // 32) * 4 + b
    return atoms[off]


# ----------------------------------------------------------------------------- L2-input ties

ROW_BYTES = {"mxfp8": 1.0, "nvfp4": 0.5, "mxfp4": 0.5}
SF_ATOMS = {"mxfp8": 1, "nvfp4": 4, "mxfp4": 2}
SF_BLOCK = {"mxfp8": 32, "nvfp4": 16, "mxfp4": 32}


def near_midpoint(v, a, b, tau):
    """v lies within tau of the midpoint of the two neighbouring grid values a, b."""
    return np.abs(v - (a + b) / 2) <= tau


def certify_l2_codes(h_or, got_codes, got_sf, fmt, a2, tau):
    """Check the GPU's L2-input codes (and block scales) of rows whose oracle value is h_or (fp64
    [n, I]) against the oracle's codes of its own fp32 h: equal, except where the oracle's value lies
    within tau of a rounding midpoint (or a block's amax within tau of a scale boundary), where the
    other neighbour is correct too. Returns (the GPU inputs dequantised by the oracle's tables [n, I],
    number of differing values)."""
    codes, sf = OM.l2_input_codes(h_or.astype(np.float32), fmt, a2)
    if fmt == "bf16":
        diff = got_codes != codes
        a, b = OF.bf16_bits_to_f64(got_codes[diff]), OF.bf16_bits_to_f64(codes[diff])
        assert np.all(near_midpoint(h_or[diff], a, b, tau))
        return OF.bf16_bits_to_f64(got_codes), int(diff.sum())
    g = SF_BLOCK[fmt]
    amax = np.abs(h_or.astype(np.float32).astype(np.float64)).reshape(len(h_or), -1, g).max(-1)
    sf_diff = got_sf != sf
    if fmt in ("mxfp8", "mxfp4"):
        top = 448.0 if fmt == "mxfp8" else 6.0
        e = sf[sf_diff].astype(np.int64) - 127
        bound = np.ldexp(top, np.minimum(e, got_sf[sf_diff].astype(np.int64) - 127))
        assert np.all(np.abs(amax[sf_diff] - bound) <= tau)
        deq = OF.mxfp8_dequantize if fmt == "mxfp8" else OF.mxfp4_dequantize
        deq_or, deq_gpu = deq(codes, sf), deq(got_codes, got_sf)
        scale = OF.UE8M0_TABLE[sf].repeat(g, axis=1)
        if fmt == "mxfp8":
            step = scale * 2.0 ** (np.floor(np.log2(np.maximum(np.abs(h_or) / scale, 2.0 ** -6))) - 3)
        else:
            q = np.abs(h_or) / scale
            step = scale * np.where(q < 2, 0.5, np.where(q < 4, 1.0, 2.0))
    else:
        a2 = np.float32(a2)
        ratio = amax / (float(a2) * 6.0)
        assert np.all(near_midpoint(ratio[sf_diff], OF.E4M3_TABLE[sf[sf_diff]], OF.E4M3_TABLE[got_sf[sf_diff]],
                                    tau / (float(a2) * 6.0)))
        deq_or = OF.nvfp4_dequantize(codes, sf, a2)
        deq_gpu = OF.nvfp4_dequantize(got_codes, got_sf, a2)
        eff = (OF.E4M3_TABLE[sf] * float(a2)).repeat(g, axis=1)
        q = np.abs(h_or) / np.maximum(eff, 1e-30)
        step = eff * np.where(q < 2, 0.5, np.where(q < 4, 1.0, 2.0))
    same_block = ~np.repeat(sf_diff, g, axis=1)
    bad = (deq_gpu != deq_or) & same_block
    # a differing value in a block with the same scale is the other neighbour of a midpoint
    assert np.all(np.abs(deq_gpu[bad] - deq_or[bad]) <= step[bad] * (1 + 1e-9))
    assert np.all(near_midpoint(h_or[bad], deq_gpu[bad], deq_or[bad], tau))
    return deq_gpu, int(bad.sum() + sf_diff.sum())


def gpu_l2_inputs(run: GpuRun, case: Case, T: int, rows) -> tuple:
    """The GPU's L2-input codes and block-scale bytes of the given permuted rows."""
    fmt, I = case.shape.fmt, case.shape.I
    hq = region_u8(run, T, "hq")
    if fmt == "bf16":
        return hq.reshape(-1, I * 2)[rows].view(np.uint16), None
    rb = int(I * ROW_BYTES[fmt])
    g = SF_BLOCK[fmt]
    return hq.reshape(-1, rb)[rows], unpack_act_sf(region_u8(run, T, "hsf"), np.asarray(rows), I // g, SF_ATOMS[fmt])


# fp32 accumulation noise of h at the full K loop (H = 7168): the GPU's h lies within ~5e-6 of the
# row's max |h| of the oracle's fp64 value; a tie is certified within 4x that
TIE_TAU_REL = 2e-5


def assert_close_allowing_ties(run: GpuRun, case: Case, sample, got, want, what=""):
    """assert_close for the sampled tokens; a token over the tolerance is accepted only if its L2-input
    codes differ from the oracle's at certified ties (certify_l2_codes, within TIE_TAU_REL of each slot's
    max |h|) and its output is within the tolerance of the oracle's value continued from those codes
    (oracle.moe.forward_from_l2_inputs). Returns the number of tokens that needed this."""
    fmt = case.shape.fmt
    rms = float(np.sqrt(np.mean(want ** 2)))
    tol = REL[fmt] * rms + ABS
    exc = (np.abs(got - want) - half_ulp_bf16(want)).max(axis=1)
    over = np.nonzero(exc > tol)[0]
    T, k = case.x.shape[0], case.shape.k
    inv = region_i32(run, T, "inv_perm")[:T * k].reshape(T, k)
    for i in over:
        t = int(sample[i])
        _, parts = OM.forward(case.layer, case.x, case.ids, case.w, tokens=[t], return_parts=True)
        l2 = []
        flips = 0
        for j in range(k):
            r_or = int(parts["inv"][0, j])
            if r_or < 0:
                l2.append(None)
                continue
            h_or = np.asarray(parts["h"][r_or], np.float64)[None]
            codes, sf = gpu_l2_inputs(run, case, T, [int(inv[t, j])])
            deq, n = certify_l2_codes(h_or, codes, sf, fmt, case.layer.a2, TIE_TAU_REL * np.abs(h_or).max())
            flips += n
            l2.append(deq[0])
        assert flips > 0, f"{what}: token {t} over the tolerance without any L2-input tie"
        z = OM.forward_from_l2_inputs(case.layer, case.x, case.ids, case.w, t, l2)
        excess = float((np.abs(got[i] - z) - half_ulp_bf16(z)).max())
        assert excess <= tol, f"{what}: token {t}: {excess:.4g} > {tol:.4g} even from the GPU's tie decisions"
    keep = np.setdiff1d(np.arange(len(sample)), over)
    assert_close(got[keep], want[keep], fmt, what)
    return len(over)
