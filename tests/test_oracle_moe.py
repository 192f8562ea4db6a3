"""Pins for the oracle's layer forward (CPU only).

Checks against: a hand-worked BF16 layer whose every step is exact
(tests/golden/mlp_exact_bf16.json), SwiGLU identities that hold for any
alpha/beta (sigmoid(z) + sigmoid(-z) = 1) and its clamp rule, the
invariants named for the layer (routing weights sum to 1; top_k = 1 with
weight 1 equals one dense MLP; a permutation and its inverse), token
independence, masking, and the placement of the NVFP4 alphas.
"""
import json
import math
import os

import numpy as np
import pytest

import synthetic as S
from oracle import formats as F
from oracle import moe as M


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------- SwiGLU

def test_swiglu_known_values():
    e = math.e
    assert M.swiglu(1.0, 1.0) == pytest.approx(e / (e + 1), rel=1e-15)         # silu(1) = e/(e+1)
    assert M.swiglu(0.0, 123.0) == 0.0
    assert M.swiglu(-1.0, 1.0) == pytest.approx(-1.0 / (e + 1), rel=1e-15)
    # alpha scales only the sigmoid's argument; beta shifts up
    assert M.swiglu(2.0, 0.0, M.Activation(alpha=0.5, beta=1.0)) == pytest.approx(2 * e / (e + 1), rel=1e-15)


@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (1.702, 1.0), (0.3, -2.0)])
def test_swiglu_odd_part_identity(alpha, beta):
    # swiglu(g,u) - swiglu(-g,u) = g*(u+beta) for any alpha, since sigmoid(z)+sigmoid(-z)=1
    rng = np.random.default_rng(0)
    g, u = rng.standard_normal(1000) * 3, rng.standard_normal(1000) * 3
    act = M.Activation(alpha=alpha, beta=beta)
    lhs = M.swiglu(g, u, act) - M.swiglu(-g, u, act)
    assert np.allclose(lhs, g * (u + beta), rtol=1e-12, atol=1e-12)


def test_swiglu_large_gate_and_clamp():
    assert M.swiglu(100.0, 7.5) == 750.0                                          # sigmoid(100) == 1 in fp64
    act = M.Activation(clamp=1.0)
    # gate clamped from above only, up symmetrically
    assert M.swiglu(50.0, 3.0, act) == M.swiglu(1.0, 1.0)
    assert M.swiglu(-3.0, -9.0, act) == M.swiglu(-3.0, -1.0)
    assert M.swiglu(-3.0, 0.5, act) == M.swiglu(-3.0, 0.5)


# ----------------------------------------------------------------------------- hand-worked layer

def _golden_layer(g):
    w13 = np.array(g["w13"], dtype=np.float32)
    w2 = np.array(g["w2"], dtype=np.float32)
    x = F.bf16_bits(np.array(g["x"]))
    ew = M.quantize_weights("bf16", w13, w2)
    layer = M.Layer(num_experts=w13.shape[0], top_k=2, routed=ew)
    return layer, x, np.array(g["topk_ids"]), np.array(g["topk_weights"], dtype=np.float32)


def test_golden_bf16_layer(golden_dir):
    g = _golden(golden_dir, "mlp_exact_bf16.json")
    layer, x, ids, w = _golden_layer(g)
    out, parts = M.forward(layer, x, ids, w, block_m=1, return_parts=True)
    assert F.bf16_bits_to_f64(out).tolist() == g["out"]
    assert [parts["h"][r][0] for r in sorted(parts["h"])] == g["h"]


def test_golden_bf16_layer_norm(golden_dir):
    g = _golden(golden_dir, "mlp_exact_bf16.json")
    layer, x, ids, w = _golden_layer(g)
    layer.norm_gamma = np.array(g["norm"]["gamma"], dtype=np.float32)
    layer.norm_eps = g["norm"]["eps"]
    out = F.bf16_bits_to_f64(M.forward(layer, x, ids, w, block_m=1))[0]
    z = np.array(g["out"][0])
    want = F.bf16_round(z / math.sqrt(g["norm"]["mean_z2"]) * np.array(g["norm"]["gamma"]))
    assert out.tolist() == want.tolist()


# ----------------------------------------------------------------------------- invariants

def _small(fmt, **kw):
    base = {"bf16": "bf16_toy", "mxfp8": "mxfp8_small", "nvfp4": "nvfp4_decode", "mxfp4": "mxfp8_small"}[fmt]
    shape = S.shrink(S.WORKLOADS[base], **{"T": 16, "H": 256, "I": 256, "E": 4, "k": 2, "fmt": fmt, **kw})
    x = S.hidden_states(shape)
    ids, w = S.router(shape)
    w13, w2 = S.routed_float_weights(shape)
    layer = M.Layer(shape.E, shape.k, M.quantize_weights(fmt, w13, w2))
    if fmt == "nvfp4":
        layer.a2 = M.calibrate_a2(layer, x, ids)
    return shape, layer, x, ids, w


def test_router_weights_sum_to_one():
    for name in S.WORKLOAD_ORDER:
        shape = S.shrink(S.WORKLOADS[name], T=min(S.WORKLOADS[name].T, 256))
        ids, w = S.router(shape)
        assert np.allclose(w.astype(np.float64).sum(1), 1.0, atol=1e-6)
        assert np.all((ids >= 0) & (ids < shape.E))
        assert all(len(set(r)) == shape.k for r in ids.tolist())


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "nvfp4", "mxfp4"])
def test_top1_weight1_equals_dense_mlp(fmt):
    shape, layer, x, _, _ = _small(fmt, k=1)
    ids = np.full((shape.T, 1), 2)
    w = np.ones((shape.T, 1), np.float32)
    out = M.forward(layer, x, ids, w)
    d = M.dispatch_quantize(x, fmt)
    dense = M.expert_mlp(d.x, layer.routed.w13_of(2), layer.routed.w2_of(2), fmt, layer.act, layer.a2)
    assert np.array_equal(out, F.bf16_bits(dense))


def test_identical_experts_combine_to_one_expert():
    # with every expert equal, sum_j w_j y = y because the weights sum to 1
    shape, layer, x, ids, w = _small("bf16", E=3, k=3)
    for arr in (layer.routed.w13, layer.routed.w2):
        arr[:] = arr[0]
    z = F.bf16_bits_to_f64(M.forward(layer, x, ids, w))
    d = M.dispatch_quantize(x, "bf16")
    y = M.expert_mlp(d.x, layer.routed.w13_of(0), layer.routed.w2_of(0), "bf16", layer.act)
    assert np.allclose(z, y, rtol=2 ** -7, atol=1e-6)


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "nvfp4", "mxfp4"])
def test_token_subset_is_exact(fmt):
    shape, layer, x, ids, w = _small(fmt)
    full = M.forward(layer, x, ids, w)
    pick = [0, 5, 11, 15]
    assert np.array_equal(M.forward(layer, x, ids, w, tokens=pick), full[pick])


def test_masked_slot_adds_nothing():
    shape, layer, x, ids, w = _small("mxfp8")
    ids2 = ids.copy()
    ids2[:, 1] = -1
    z_masked = M.forward(layer, x, ids2, w, return_parts=True)[1]["z"]
    z_only0 = M.forward(layer, x, ids[:, :1], w[:, :1], return_parts=True)[1]["z"]
    assert np.array_equal(z_masked, z_only0)


def test_nvfp4_l2_alpha_placement():
    # doubling every w2 global scale doubles y exactly (the L2 alpha multiplies the output)
    shape, layer, x, ids, w = _small("nvfp4")
    z1 = M.forward(layer, x, ids, w, return_parts=True)[1]["z"]
    layer.routed.w2_gs = layer.routed.w2_gs * np.float32(2)
    z2 = M.forward(layer, x, ids, w, return_parts=True)[1]["z"]
    assert np.array_equal(z2, 2 * z1)


def test_nvfp4_dispatch_token_scale():
    shape, layer, x, ids, w = _small("nvfp4")
    d = M.dispatch_quantize(x, "nvfp4")
    amax = np.abs(F.bf16_bits_to_f64(x)).max(1).astype(np.float32)
    assert np.array_equal(d.x_scale, (amax / np.float32(2688)).astype(np.float32))


@pytest.mark.parametrize("fmt,tol", [("mxfp8", 0.08), ("nvfp4", 0.35), ("mxfp4", 0.45)])
def test_quantised_layer_tracks_bf16_layer(fmt, tol):
    # a dropped or doubled scale anywhere would push this far past the format's noise
    shape, layer, x, ids, w = _small(fmt, T=32)
    w13, w2 = S.routed_float_weights(shape)
    # near-exact reference: the same layer in BF16 (relative rounding 2^-9 instead of 2^-4 / 2^-2)
    ref_layer = M.Layer(shape.E, shape.k, M.quantize_weights("bf16", w13, w2))
    q = F.bf16_bits_to_f64(M.forward(layer, x, ids, w))
    r = F.bf16_bits_to_f64(M.forward(ref_layer, x, ids, w))
    rel = np.sqrt(np.mean((q - r) ** 2)) / np.sqrt(np.mean(r ** 2))
    assert rel < tol


def test_shared_expert_and_norm_compose():
    shape, layer, x, ids, w = _small("nvfp4", H=256)
    s13, s2 = S.shared_float_weights(S.shrink(shape, shared_I=256))
    layer.shared = M.quantize_weights("mxfp8", s13[None], s2[None])
    out_s, parts = M.forward(layer, x, ids, w, return_parts=True)
    d = M.dispatch_quantize(x, "mxfp8")
    ys = M.expert_mlp(d.x, layer.shared.w13_of(0), layer.shared.w2_of(0), "mxfp8", M.Activation())
    layer.shared = None
    z0 = M.forward(layer, x, ids, w, return_parts=True)[1]["z"]
    assert np.allclose(parts["z"], z0 + ys, rtol=0, atol=1e-12)
    layer.norm_gamma = np.ones(shape.H, np.float32)
    zn = F.bf16_bits_to_f64(M.forward(layer, x, ids, w))
    # rms of a normalised row is 1 (up to bf16 rounding)
    assert np.allclose(np.sqrt(np.mean(zn ** 2, axis=1)), 1.0, atol=4e-3)


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "nvfp4", "mxfp4"])
def test_batched_layout_equals_routed_top1(fmt):
    """The batched (masked) layout is the routed layer with top_k = 1 and weight 1: every
    token goes to one expert, and its slot's row of the routed output is its batched row."""
    shape, layer, _, _, _ = _small(fmt, T=24, E=4, k=1)
    cap = 8
    counts = np.array([3, 0, 8, 5])
    xb = S.hidden_states(S.shrink(shape, T=4 * cap)).reshape(4, cap, shape.H)
    out_b = M.forward_batched(layer, xb, counts)
    # the same rows as a routed batch: token i of expert e -> expert e, weight 1
    rows = [(e, m) for e in range(4) for m in range(counts[e])]
    x_r = np.stack([xb[e, m] for e, m in rows])
    ids = np.array([[e] for e, _ in rows])
    w = np.ones((len(rows), 1), np.float32)
    out_r = M.forward(layer, x_r, ids, w)
    for i, (e, m) in enumerate(rows):
        assert np.array_equal(out_b[e, m], out_r[i]), (e, m)
    for e in range(4):
        assert not out_b[e, counts[e]:].any()


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "bf16"])
def test_forward_from_l2_inputs_reproduces_forward(fmt):
    """Continuing from the oracle's own requantised L2 inputs gives the forward's value (shared
    expert and norm included) up to fp64 summation order (one row at a time instead of a
    matrix product), so the continuation adds nothing of its own."""
    shape = S.shrink(S.WORKLOADS["nvfp4_shared_norm"], T=6, H=256, I=256, E=4, k=3, fmt=fmt, shared_I=256)
    x = S.hidden_states(shape)
    ids, w = S.router(shape)
    ids = ids.copy()
    ids[2, 1] = -1                                   # a masked slot
    w13f, w2f = S.routed_float_weights(shape)
    layer = M.Layer(shape.E, shape.k, M.quantize_weights(fmt, w13f, w2f))
    if fmt == "nvfp4":
        layer.a2 = M.calibrate_a2(layer, x, ids)
    s13, s2 = S.shared_float_weights(shape)
    layer.shared = M.quantize_weights("mxfp8", s13[None], s2[None])
    layer.norm_gamma = S.norm_gamma(shape)
    _, parts = M.forward(layer, x, ids, w, return_parts=True)
    for t in range(shape.T):
        l2 = []
        for j in range(shape.k):
            r = parts["inv"][t, j]
            l2.append(None if r < 0 else M.l2_input_quantize(parts["h"][r][None], fmt, layer.a2)[0])
        z = M.forward_from_l2_inputs(layer, x, ids, w, t, l2)
        assert np.allclose(z, parts["z"][t], rtol=1e-12, atol=1e-12 * np.abs(parts["z"][t]).max())
