"""GPU parity of the C-ABI path against the CPU oracle (needs a GB300).

Bit-exact: routing (counts, padded offsets, permutation, inverse), dispatch
codes and scales, per-token NVFP4 scales, the weight layouts. The L2-input
codes equal the oracle's codes of the oracle's h except where the oracle's
value is within accumulation noise of a rounding midpoint. Within the layer's
tolerance (max |gpu - oracle| <= rel * rms + 1e-3, rel 2e-2 BF16/MXFP8, 5e-2
NVFP4, for the value before the output's final bf16 rounding, i.e. against the
oracle's exact value with half a bf16 step of the output on top): every output
at reduced sizes spanning several tiles with ragged tails, and sampled tokens
at the full workload sizes. Every expected value comes from the oracle.
"""
import numpy as np
import pytest
import torch

import synthetic as S
from oracle import formats as OF
from oracle import moe as OM
from oracle import routing as OR
import gpu_case as G

pytestmark = pytest.mark.gpu

W = S.WORKLOADS

REDUCED = {
    "bf16_toy": W["bf16_toy"],
    "mxfp8_small": S.shrink(W["mxfp8_small"], T=200, H=512, I=384, E=16, k=4),
    "mxfp8_h384": S.shrink(W["mxfp8_small"], T=77, H=384, I=256, E=8, k=3),
    "nvfp4_decode": S.shrink(W["nvfp4_decode"], T=40, H=1024, I=512, E=32, k=8),
    "mxfp8_prefill_zipf": S.shrink(W["mxfp8_prefill_zipf"], T=512, H=768, I=256, E=32, k=8),
    "nvfp4_shared_norm": S.shrink(W["nvfp4_shared_norm"], T=130, H=512, I=256, E=16, k=4, shared_I=512),
    "mxfp4_small": S.shrink(W["mxfp4_small"], T=200, H=512, I=512, E=16, k=4),
    # NVFP4 routed experts beside a BF16 shared expert (the other shared precision the pages list)
    "nvfp4_bf16_shared": S.shrink(W["nvfp4_shared_norm"], name="nvfp4_bf16_shared", T=130, H=512, I=256, E=16, k=4,
                                  shared_I=512, shared_fmt="bf16"),
}
# bytes per element, scale atoms per 128-byte K stage, elements per scale block
ROW_BYTES = {"mxfp8": 1.0, "nvfp4": 0.5, "mxfp4": 0.5}
SF_ATOMS = {"mxfp8": 1, "nvfp4": 4, "mxfp4": 2}
SF_BLOCK = {"mxfp8": 32, "nvfp4": 16, "mxfp4": 32}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    import serving_topk_permute_gb300 as pkg
    pkg.lib()


# ----------------------------------------------------------------------------- routing + dispatch, full size

def _ids_only_case(shape):
    """Full-size inputs; weights are random device bytes (routing / dispatch do not read them)."""
    return G.code_case(shape, sample_tokens=[], seed=0)


@pytest.mark.parametrize("name", S.WORKLOAD_ORDER)
def test_routing_and_dispatch_bit_exact_full_size(name):
    _check_routing_and_dispatch(W[name])


def _check_routing_and_dispatch(shape):
    case = _ids_only_case(shape)
    run = G.run_gpu(case)
    T, k, E = shape.T, shape.k, shape.E
    cnt, off, src, inv = OR.permute(case.ids, E, run.plan.block_m(T))
    assert np.array_equal(G.region_i32(run, T, "counts")[:E], cnt)
    assert np.array_equal(G.region_i32(run, T, "offsets")[:E + 1], off)
    M_pad = int(off[-1])
    assert np.array_equal(G.region_i32(run, T, "src")[:M_pad], src)
    assert np.array_equal(G.region_i32(run, T, "inv_perm")[:T * k].reshape(T, k), inv)
    meta = G.region_i32(run, T, "meta")
    assert meta[0] == M_pad and meta[1] == M_pad // run.plan.block_m(T)

    # dispatch codes: every routed row holds its token's codes
    d = OM.dispatch_quantize(case.x, shape.fmt)
    rows = inv.reshape(-1)
    toks = np.repeat(np.arange(T), k)
    xq = G.region_u8(run, T, "xq")
    if shape.fmt == "bf16":
        got = xq.reshape(-1, shape.H * 2)[rows].view(np.uint16)
        assert np.array_equal(got, case.x[toks])
        return
    row_bytes = int(shape.H * ROW_BYTES[shape.fmt])
    got_codes = xq.reshape(-1, row_bytes)[rows]
    assert np.array_equal(got_codes, d.codes[toks])
    S_atoms = SF_ATOMS[shape.fmt]
    nblk = shape.H // SF_BLOCK[shape.fmt]
    got_sf = G.unpack_act_sf(G.region_u8(run, T, "xsf"), rows, nblk, S_atoms)
    assert np.array_equal(got_sf, d.sf[toks])
    if shape.fmt == "nvfp4":
        xs = G.region_u8(run, T, "x_scale").view(np.float32)[:T]
        assert np.array_equal(xs, d.x_scale)
    assert run.plan.last_status(run.workspace) == 0


# ----------------------------------------------------------------------------- outputs, reduced sizes, every element

@pytest.mark.parametrize("mode", list(G.MODES))
@pytest.mark.parametrize("name", list(REDUCED))
def test_forward_matches_oracle_reduced(name, mode):
    """Every GEMM variant: L1 and L2 in one kernel (the default); two single-CTA kernels with
    128-wide tiles (double-buffered accumulators) or 256-wide tiles; CTA pairs (256 x 256 tiles
    over 256-row segments)."""
    shape = REDUCED[name]
    case = G.float_case(shape)
    run = G.run_gpu(case, **G.MODES[mode])
    G.assert_close(G.out_f64(run), G.oracle_out(case), shape.fmt, name)
    assert run.plan.last_status(run.workspace) == 0


@pytest.mark.parametrize("name", ["mxfp8_small", "nvfp4_decode", "nvfp4_shared_norm", "bf16_toy", "mxfp4_small"])
def test_l2_input_matches_oracle(name):
    """The GPU's fp32 h against the oracle's h, and the GPU's L2-input codes against the
    oracle's codes of its own h: equal except where the oracle's value sits within
    fp32 accumulation noise of a rounding midpoint (then either neighbour is correct)."""
    shape = REDUCED[name]
    case = G.float_case(shape)
    run = G.run_gpu(case, debug_h=True)
    T, I = shape.T, shape.I
    src = G.region_i32(run, T, "src")
    M_pad = int(G.region_i32(run, T, "meta")[0])
    rows = np.nonzero(src[:M_pad] >= 0)[0]
    parts = OM.forward(case.layer, case.x, case.ids, case.w, return_parts=True)[1]
    h_or = np.stack([parts["h"][r] for r in rows])                      # rows are the oracle's rows too
    h_gpu = G.region_u8(run, T, "h_debug").view(np.float32).reshape(-1, I)[rows].astype(np.float64)
    hmax = np.abs(h_or).max()
    rel_err = np.abs(h_gpu - h_or).max() / hmax
    assert rel_err < 1e-5, rel_err
    # fp32 accumulation noise of h (the GPU is ~1.5e-7 of max|h| off the fp64 oracle);
    # a code may differ only where the oracle's value is this close to a rounding midpoint
    TAU = 1e-6 * hmax
    codes, sf = G.gpu_l2_inputs(run, case, T, rows)
    _, n_diff = G.certify_l2_codes(h_or, codes, sf, shape.fmt, case.layer.a2, TAU)
    assert n_diff < 1e-3 * h_or.size, n_diff


# ----------------------------------------------------------------------------- outputs, full size, sampled tokens

def _tile_covering_sample(shape, block_m: int, n_min: int = 256):
    """Tokens whose rows cover every row tile of the five largest experts and the last row
    tile of every touched expert (from the oracle's own permutation at the library's
    BLOCK_M), plus evenly spaced tokens up to n_min (all tokens when T <= n_min)."""
    T, k = shape.T, shape.k
    if T <= n_min:
        return list(range(T))
    ids, _ = S.router(shape, 0)
    cnt, off, src, inv = OR.permute(ids, shape.E, block_m)
    chosen = {0, 1, T // 3, T // 2, T - 2, T - 1}
    for e in np.argsort(-cnt, kind="stable")[:5]:
        for r0 in range(int(off[e]), int(off[e] + cnt[e]), block_m):
            chosen.add(int(src[r0]) // k)          # the tile's first row is a routed one
    for e in np.nonzero(cnt)[0]:
        chosen.add(int(src[off[e] + cnt[e] - 1]) // k)   # the last routed row: in the last row tile
    for t in np.linspace(0, T - 1, n_min).astype(int):
        if len(chosen) >= n_min:
            break
        chosen.add(int(t))
    return sorted(chosen)


@pytest.mark.parametrize("name", ["mxfp8_small", "nvfp4_decode", "mxfp8_prefill_zipf", "nvfp4_shared_norm",
                                  "mxfp4_small"])
def test_forward_matches_oracle_full_size_sampled(name):
    """Full workload sizes and launch configuration; at least 256 tokens compared (all of them when T is
    smaller), chosen so that every row tile of the five largest experts and the last row tile of every
    touched expert holds a compared row."""
    import serving_topk_permute_gb300 as pkg
    shape = W[name]
    probe = pkg.Plan(pkg.LayerConfig(shape.E, shape.H, shape.I, shape.k, shape.T, shape.fmt))
    sample = _tile_covering_sample(shape, probe.block_m(shape.T))
    del probe
    case = G.code_case(shape, sample)
    ids = case.ids
    cnt, off, src, inv = OR.permute(ids, shape.E, 128)
    rows = {int(inv[t, j]) // 128 for t in sample for j in range(shape.k) if inv[t, j] >= 0}
    for e in np.argsort(-cnt, kind="stable")[:5]:
        assert set(range(int(off[e]) // 128, int(off[e] + cnt[e] + 127) // 128)) <= rows
    run = G.run_gpu(case)
    got = G.out_f64(run)[sample]
    # a token whose L2-input code is a tie within fp32 accumulation noise may take the other (equally
    # correct) neighbour; at the full K loop one such value near the top of its block can move the
    # token's output by more than the tolerance, so those tokens are compared with the oracle's value
    # continued from the GPU's (certified) decisions
    G.assert_close_allowing_ties(run, case, sample, got, G.oracle_out(case, tokens=sample), name)


_FULL_PREFILL = {}


@pytest.mark.parametrize("mode", ["split256", "pair"])
def test_prefill_full_size_other_gemm_modes(mode):
    """The two-kernel GEMM and the CTA-pair GEMM (256-row segments) on the full Zipf-routed prefill
    workload, on the same tile-covering token sample as the default mode (the oracle's values are
    computed once for both)."""
    import serving_topk_permute_gb300 as pkg
    shape = W["mxfp8_prefill_zipf"]
    if "case" not in _FULL_PREFILL:
        probe = pkg.Plan(pkg.LayerConfig(shape.E, shape.H, shape.I, shape.k, shape.T, shape.fmt))
        sample = _tile_covering_sample(shape, probe.block_m(shape.T))
        del probe
        case = G.code_case(shape, sample)
        _FULL_PREFILL.update(case=case, sample=sample, want=G.oracle_out(case, tokens=sample))
    case, sample, want = _FULL_PREFILL["case"], _FULL_PREFILL["sample"], _FULL_PREFILL["want"]
    run = G.run_gpu(case, **G.MODES[mode])
    if mode == "pair":
        assert run.plan.block_m(shape.T) == 256
    G.assert_close_allowing_ties(run, case, sample, G.out_f64(run)[sample], want, f"prefill {mode}")
    assert run.plan.last_status(run.workspace) == 0


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_full_hidden_float_weights(fmt):
    """The full hidden and intermediate sizes (H = 7168, I = 2048: the whole 56-stage L1 and 16-stage L2 K
    loops of the prefill and decode shapes) with float weights quantised by the oracle (the workloads'
    exact recipe, so E4M3 subnormal codes occur, and NVFP4 block scales of 40 to 448, outside the 1 to 16
    of the drawn-code checkpoints), on few experts so the host quantiser stays fast; every token
    compared, full and partial row tiles both present."""
    base = "mxfp8_prefill_zipf" if fmt == "mxfp8" else "nvfp4_decode"
    shape = S.shrink(W[base], T=300, E=4, k=2)
    case = G.float_case(shape)
    codes = case.layer.routed.w13
    if fmt == "mxfp8":
        assert ((codes & 0x78) == 0).any()     # E4M3 subnormal (or zero) codes occur
    else:
        sf = case.layer.routed.w13_sf
        assert (sf > 0x58).any()               # E4M3 block scales above 16 occur
    run = G.run_gpu(case)
    tokens = list(range(shape.T))
    G.assert_close_allowing_ties(run, case, tokens, G.out_f64(run), G.oracle_out(case), f"{fmt} H=7168")


# ----------------------------------------------------------------------------- edge cases

def _small_case(fmt="mxfp8", **kw):
    base = {"bf16": "bf16_toy", "mxfp8": "mxfp8_small", "nvfp4": "nvfp4_decode", "mxfp4": "mxfp4_small"}[fmt]
    shape = S.shrink(W[base], **{"T": 64, "H": 256, "I": 256, "E": 8, "k": 2, **kw})
    return shape


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "nvfp4", "mxfp4"])
def test_single_token(fmt):
    shape = _small_case(fmt, T=1)
    case = G.float_case(shape)
    G.assert_close(G.out_f64(G.run_gpu(case)), G.oracle_out(case), fmt, "T=1")


@pytest.mark.parametrize("H", [10240, 16384])
@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "nvfp4", "mxfp4"])
def test_wide_hidden(fmt, H):
    """H above 8192 (up to the 16384 limit) takes the dispatch variant holding 8 chunks per thread."""
    shape = _small_case(fmt, T=24, H=H, I=256, E=4, k=2)
    _check_routing_and_dispatch(shape)
    case = G.float_case(shape)
    G.assert_close(G.out_f64(G.run_gpu(case)), G.oracle_out(case), fmt, f"H={H}")


@pytest.mark.parametrize("name", ["mxfp8_small", "nvfp4_shared_norm"])
def test_pinned_host_io_matches_device_io(name):
    """hidden, ids, weights, gamma and out in pinned host memory (read and written by the kernels over the
    host link) give the same bits as device buffers."""
    shape = REDUCED[name]
    run = G.run_gpu(G.float_case(shape))
    pin = lambda t: None if t is None else t.cpu().pin_memory()
    h = {k: pin(run.inputs[k]) for k in ("hidden", "topk_ids", "topk_weights", "gamma")}
    out = torch.zeros(run.out.shape, dtype=run.out.dtype).pin_memory()
    run.plan.forward(h["hidden"], h["topk_ids"], h["topk_weights"], run.kweights, l2_act_scale=run.inputs["a2"],
                     shared=run.kshared, norm_gamma=h["gamma"], out=out, workspace=run.workspace)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), run.out.view(torch.int16).cpu())
    assert run.plan.last_status(run.workspace) == 0


def test_masked_slots_and_duplicates():
    shape = _small_case("mxfp8", T=96, k=3)
    ids, w = S.router(shape)
    ids = ids.copy()
    ids[::3, 1] = -1                 # masked slots
    ids[1::5, 2] = ids[1::5, 0]      # the same expert twice in one token
    case = G.float_case(shape, ids=ids, w=w)
    G.assert_close(G.out_f64(G.run_gpu(case)), G.oracle_out(case), "mxfp8", "masked/dup")


@pytest.mark.parametrize("mode", ["fused", "split256", "pair"])
@pytest.mark.parametrize("fmt", ["bf16", "nvfp4"])
def test_all_tokens_one_expert(fmt, mode):
    shape = _small_case(fmt, T=300, k=1)
    ids = np.full((300, 1), 5, np.int32)
    w = np.ones((300, 1), np.float32)
    case = G.float_case(shape, ids=ids, w=w)
    run = G.run_gpu(case, **G.MODES[mode])
    G.assert_close(G.out_f64(run), G.oracle_out(case), fmt, "one expert")
    off = G.region_i32(run, 300, "offsets")[:9]
    pad = 384 if run.plan.block_m(300) == 128 else 512
    assert off.tolist() == [0, 0, 0, 0, 0, 0, pad, pad, pad]


@pytest.mark.parametrize("E,k,T", [(512, 8, 300), (64, 32, 70), (40, 6, 333), (7, 5, 97)])
def test_routing_limits_and_ragged_chunks(E, k, T):
    """The largest expert count and top-k, and k that does not divide the routing chunk (a
    token's slots straddle two chunks): routing bit-exact, outputs within tolerance."""
    shape = _small_case("mxfp8", T=T, E=E, k=k, I=128)
    case = G.float_case(shape)
    run = G.run_gpu(case)
    cnt, off, src, inv = OR.permute(case.ids, E, run.plan.block_m(T))
    assert np.array_equal(G.region_i32(run, T, "counts")[:E], cnt)
    assert np.array_equal(G.region_i32(run, T, "offsets")[:E + 1], off)
    assert np.array_equal(G.region_i32(run, T, "src")[:int(off[-1])], src)
    assert np.array_equal(G.region_i32(run, T, "inv_perm")[:T * k].reshape(T, k), inv)
    G.assert_close(G.out_f64(run), G.oracle_out(case), "mxfp8", f"E={E} k={k}")


def test_bad_expert_id_reports_status_and_is_masked():
    shape = _small_case("bf16", T=32)
    ids, w = S.router(shape)
    bad = ids.copy()
    bad[3, 0] = shape.E + 5
    case = G.float_case(shape, ids=bad, w=w)
    run = G.run_gpu(case)
    assert run.plan.last_status(run.workspace) == 6
    masked = bad.copy()
    masked[3, 0] = -1
    ref = G.Case(case.shape, case.x, masked, case.w, case.layer)
    G.assert_close(G.out_f64(run), G.oracle_out(ref), "bf16", "bad id")


def test_capacity_and_empty_batch():
    import serving_topk_permute_gb300 as pkg
    shape = _small_case("bf16", T=16)
    case = G.float_case(shape)
    run = G.run_gpu(case)
    with pytest.raises(pkg.MoeError) as e:
        big = torch.zeros((17, shape.H), dtype=torch.bfloat16, device="cuda")
        run.plan.forward(big, torch.zeros((17, 2), dtype=torch.int32, device="cuda"),
                         torch.zeros((17, 2), dtype=torch.float32, device="cuda"), run.kweights,
                         workspace=run.workspace)
    assert e.value.status == 3
    empty = torch.zeros((0, shape.H), dtype=torch.bfloat16, device="cuda")
    out = run.plan.forward(empty, torch.zeros((0, 2), dtype=torch.int32, device="cuda"),
                           torch.zeros((0, 2), dtype=torch.float32, device="cuda"), run.kweights,
                           workspace=run.workspace)
    assert out.shape == (0, shape.H)


def test_misaligned_pointers_refused():
    """Every device pointer must be 256-byte aligned (the kernels read and write with 16-byte
    and bulk copies): a misaligned hidden, output, norm gamma, scale-atom tensor or L2 input
    scale is refused on the host (MOE_ERR_INVALID_ARG) before anything is launched, and the
    plan then still computes the same answer."""
    import serving_topk_permute_gb300 as pkg
    case = G.float_case(REDUCED["nvfp4_shared_norm"])
    run = G.run_gpu(case)
    i = run.inputs
    T, H = case.x.shape
    big_h = torch.empty(T * H + 8, dtype=torch.bfloat16, device=G.dev())
    big_o = torch.empty(T * H + 8, dtype=torch.bfloat16, device=G.dev())
    big_g = torch.empty(H + 4, dtype=torch.float32, device=G.dev())
    big_g[1:H + 1].copy_(i["gamma"])
    sf = run.kweights["w13_sf"]
    big_sf = torch.empty(sf.numel() + 16, dtype=torch.uint8, device=G.dev())
    big_a2 = torch.empty(8, dtype=torch.float32, device=G.dev())
    big_a2[1:2].copy_(i["a2"])
    bad = {"hidden": dict(hidden=big_h[8:].view(T, H).copy_(i["hidden"])),
           "out": dict(out=big_o[8:].view(T, H)),
           "gamma": dict(norm_gamma=big_g[1:H + 1]),
           "scale atoms": dict(weights={**run.kweights, "w13_sf": big_sf[16:].copy_(sf)}),
           "L2 input scale": dict(a2=big_a2[1:2])}
    for what, kw in bad.items():
        args = dict(hidden=i["hidden"], norm_gamma=i["gamma"], out=None, weights=run.kweights, a2=i["a2"])
        args.update(kw)
        with pytest.raises(pkg.MoeError) as e:
            run.plan.forward(args["hidden"], i["topk_ids"], i["topk_weights"], args["weights"], l2_act_scale=args["a2"],
                             shared=run.kshared, norm_gamma=args["norm_gamma"], out=args["out"],
                             workspace=run.workspace)
        assert e.value.status == 1, what
    out = run.plan.forward(i["hidden"], i["topk_ids"], i["topk_weights"], run.kweights, l2_act_scale=i["a2"],
                           shared=run.kshared, norm_gamma=i["gamma"], workspace=run.workspace)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), run.out.view(torch.int16))


def test_workspace_too_small():
    import serving_topk_permute_gb300 as pkg
    shape = _small_case("bf16", T=16)
    case = G.float_case(shape)
    run = G.run_gpu(case)
    with pytest.raises(pkg.MoeError) as e:
        run.plan.forward(run.inputs["hidden"], run.inputs["topk_ids"], run.inputs["topk_weights"], run.kweights,
                         workspace=run.workspace[:1024])
    assert e.value.status == 4


@pytest.mark.parametrize("mode", ["fused", "split256", "pair"])
@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_deterministic(fmt, mode):
    shape = _small_case(fmt, T=150, k=4, E=8)
    case = G.float_case(shape)
    a = G.run_gpu(case, **G.MODES[mode]).out.clone()
    b = G.run_gpu(case, **G.MODES[mode]).out.clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "nvfp4_shared_norm"])
def test_back_to_back_forwards_overlapped_launch(fmt):
    """Forwards queued back to back on one workspace and stream, each kernel's set-up overlapping the
    previous kernel (the default launch), equal forwards run one at a time with serialised launches.
    Forward n+1's routing rewrites inv_perm while forward n's combine may still be queued. With a
    shared expert, its GEMM launch takes SMs while the routed GEMMs are still finishing (it waits
    for them only before it exits), and the combine must still see both."""
    import serving_topk_permute_gb300 as pkg
    if fmt == "nvfp4_shared_norm":
        shape = S.shrink(W["nvfp4_shared_norm"], T=150, H=512, I=256, E=8, k=4, shared_I=512)
    else:
        shape = _small_case(fmt, T=150, k=4, E=8)
    case = G.float_case(shape)
    x2 = S.hidden_states(shape, 1)
    ids2, w2 = S.router(shape, 1)
    inputs = [(G.bf16_dev(case.x), G.to_dev(case.ids.astype(np.int32)), G.to_dev(case.w.astype(np.float32))),
              (G.bf16_dev(x2), G.to_dev(np.asarray(ids2, np.int32)), G.to_dev(np.asarray(w2, np.float32)))]
    a2 = torch.tensor([np.float32(case.layer.a2)], device=G.dev()) if shape.fmt == "nvfp4" else None
    gamma = None if case.layer.norm_gamma is None else G.to_dev(np.asarray(case.layer.norm_gamma, np.float32))
    outs = {}
    for serial in (True, False):
        cfg = G.layer_config(case)
        cfg.serial = serial
        plan = pkg.Plan(cfg)
        kw = plan.transform_weights(G._ckpt_dev(case.layer.routed))
        ks = plan.transform_shared_weights(G._ckpt_dev(case.layer.shared)) if case.layer.shared else None
        ws = plan.alloc_workspace(shape.T)
        res = []
        for i in (0, 1, 0, 1):
            if serial:
                torch.cuda.synchronize()
            h, ids, w = inputs[i]
            res.append(plan.forward(h, ids, w, kw, l2_act_scale=a2, shared=ks, norm_gamma=gamma, workspace=ws))
        torch.cuda.synchronize()
        assert plan.last_status(ws) == 0
        outs[serial] = [r.view(torch.int16) for r in res]
    for j in range(4):
        assert torch.equal(outs[True][j], outs[False][j]), f"forward {j}"
    assert torch.equal(outs[False][0], outs[False][2]) and torch.equal(outs[False][1], outs[False][3])
    if case.layer.shared is not None:
        G.assert_close(outs[False][0].view(torch.bfloat16).float().cpu().numpy().astype(np.float64),
                       G.oracle_out(case), shape.fmt, "shared expert, overlapped launch")


@pytest.mark.parametrize("alpha,beta,clamp", [(1.702, 1.0, 7.0), (1.0, 0.0, 0.5), (0.5, -0.25, None)])
def test_activation_variants(alpha, beta, clamp):
    shape = _small_case("mxfp8", T=80)
    case = G.float_case(shape)
    case.layer.act = OM.Activation(alpha=alpha, beta=beta, clamp=clamp)
    G.assert_close(G.out_f64(G.run_gpu(case)), G.oracle_out(case), "mxfp8", "activation")


# ----------------------------------------------------------------------------- batched (masked) layout

def _batched_case(fmt, E=6, M=256):
    H, I = (512, 256) if fmt in ("nvfp4", "mxfp4", "bf16") else (384, 256)
    shape = _small_case(fmt, E=E, H=H, I=I, k=1, T=8)
    case = G.float_case(shape)
    xb = S.hidden_states(S.shrink(shape, T=E * M)).reshape(E, M, H)
    import serving_topk_permute_gb300 as pkg
    plan = pkg.Plan(G.layer_config(case))
    kw = plan.transform_weights(G._ckpt_dev(case.layer.routed))
    a2 = torch.tensor([np.float32(case.layer.a2)], device=G.dev()) if fmt == "nvfp4" else None
    return case, xb, plan, kw, a2


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "nvfp4", "mxfp4"])
def test_batched_layout_matches_oracle(fmt):
    """moe_forward_batched on [E, M, H] slabs: used rows (counts 0, 1, a whole tile, a tile
    plus one, the whole slab, a ragged one) within tolerance of the oracle; other rows untouched."""
    E, M = 6, 256
    case, xb, plan, kw, a2 = _batched_case(fmt, E, M)
    counts = np.array([0, 1, 128, 129, 256, 37], np.int32)
    out = torch.full((E, M, xb.shape[2]), 7.0, dtype=torch.bfloat16, device=G.dev())
    ws = torch.zeros(plan.batched_workspace_size(M), dtype=torch.uint8, device=G.dev())
    plan.forward_batched(G.bf16_dev(xb.reshape(E * M, -1)).view(E, M, -1), G.to_dev(counts), kw, l2_act_scale=a2,
                         out=out, workspace=ws)
    torch.cuda.synchronize()
    assert plan.last_status(ws) == 0
    want = OM.forward_batched(case.layer, xb, counts, exact=True)
    got = out.float().cpu().numpy().astype(np.float64)
    used = np.arange(M)[None, :] < counts[:, None]
    G.assert_close(got[used], want[used], fmt, "batched")
    assert np.all(got[~used] == 7.0)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_sparse_row_tile_box_boundaries(fmt):
    """The one-kernel GEMM loads a row tile with at most 96 used rows in 32-row boxes and a fuller
    one whole: used-row counts on each side of every box boundary (batched layout, one tile each)."""
    E, M = 9, 128
    case, xb, plan, kw, a2 = _batched_case(fmt, E, M)
    counts = np.array([31, 32, 33, 64, 65, 96, 97, 127, 128], np.int32)
    out = torch.full((E, M, xb.shape[2]), 7.0, dtype=torch.bfloat16, device=G.dev())
    ws = torch.zeros(plan.batched_workspace_size(M), dtype=torch.uint8, device=G.dev())
    plan.forward_batched(G.bf16_dev(xb.reshape(E * M, -1)).view(E, M, -1), G.to_dev(counts), kw, l2_act_scale=a2,
                         out=out, workspace=ws)
    torch.cuda.synchronize()
    assert plan.last_status(ws) == 0
    want = OM.forward_batched(case.layer, xb, counts, exact=True)
    got = out.float().cpu().numpy().astype(np.float64)
    used = np.arange(M)[None, :] < counts[:, None]
    G.assert_close(got[used], want[used], fmt, "box boundaries")
    assert np.all(got[~used] == 7.0)


def test_batched_layout_errors():
    """max_tokens not a multiple of 128 is refused; a count above max_tokens is clamped and
    reported as MOE_ERR_CAPACITY; a plan on CTA pairs cannot run the batched layout."""
    import serving_topk_permute_gb300 as pkg
    E, M = 6, 256
    case, xb, plan, kw, a2 = _batched_case("mxfp8", E, M)
    with pytest.raises(pkg.MoeError):
        plan.batched_workspace_size(200)
    counts = np.array([3, 300, 0, 5, 256, 1], np.int32)
    ws = torch.zeros(plan.batched_workspace_size(M), dtype=torch.uint8, device=G.dev())
    out = plan.forward_batched(G.bf16_dev(xb.reshape(E * M, -1)).view(E, M, -1), G.to_dev(counts), kw, workspace=ws)
    torch.cuda.synchronize()
    assert plan.last_status(ws) == 3  # MOE_ERR_CAPACITY
    clamped = np.minimum(counts, M)
    want = OM.forward_batched(case.layer, xb, clamped, exact=True)
    used = np.arange(M)[None, :] < clamped[:, None]
    G.assert_close(out.float().cpu().numpy().astype(np.float64)[used], want[used], "mxfp8", "clamped")
    pair = pkg.Plan(G.layer_config(case, cta="pair"))
    with pytest.raises(pkg.MoeError):
        pair.batched_workspace_size(M)


# ----------------------------------------------------------------------------- weight layout

def _expected_interleave(w13: np.ndarray, I: int) -> np.ndarray:
    """Kernel row 128b + 64h + r holds checkpoint row h*I + 64b + r (h 0 gate, 1 up, r < 64)."""
    out = np.empty_like(w13)
    for n in range(2 * I):
        b, h, r = n // 128, (n % 128) // 64, n % 64
        out[:, n] = w13[:, h * I + 64 * b + r]
    return out


def _expected_sf_atoms(sf: np.ndarray, N: int, K: int, g: int, interleave: bool, I: int, S_atoms: int) -> np.ndarray:
    """Row 32j+i / scale b of 4 at byte 16i + 4j + b of a 512-byte atom (the UTCCP row
    permutation 128c + 32j + i -> 128c + 4i + j in 32-bit words), atoms
    [E][K stage][128-row block][S], blocks = round_up(N, 256) / 128."""
    E = sf.shape[0]
    nkb = K // g
    nks = nkb // (4 * S_atoms)
    nblk = -(-N // 256) * 2
    out = np.zeros((E, nks, nblk, S_atoms, 512), np.uint8)
    for n in range(N):
        row = n
        if interleave:
            b, h, r = n // 128, (n % 128) // 64, n % 64
            row = h * I + 64 * b + r
        nb, m = n // 128, n % 128
        for kb in range(nkb):
            ks, s, bb = kb // (4 * S_atoms), (kb // 4) % S_atoms, kb % 4
            out[:, ks, nb, s, (m % 32) * 16 + (m // 32) * 4 + bb] = sf[:, row, kb]
    return out.reshape(-1)


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "nvfp4", "mxfp4"])
def test_weight_transform_layout(fmt):
    shape = _small_case(fmt, H=512 if fmt != "mxfp8" else 384, I=256, E=3)
    case = G.float_case(shape)
    run = G.run_gpu(case)
    ew = case.layer.routed
    kw = {k: v.cpu().numpy() for k, v in run.kweights.items()}
    w13 = ew.w13.view(np.uint8).reshape(shape.E, 2 * shape.I, -1)
    assert np.array_equal(kw["w13"], _expected_interleave(w13, shape.I).reshape(-1))
    assert np.array_equal(kw["w2"], ew.w2.view(np.uint8).reshape(-1))
    if fmt == "bf16":
        return
    g = SF_BLOCK[fmt]
    assert np.array_equal(kw["w13_sf"], _expected_sf_atoms(ew.w13_sf, 2 * shape.I, shape.H, g, True, shape.I, SF_ATOMS[fmt]))
    assert np.array_equal(kw["w2_sf"], _expected_sf_atoms(ew.w2_sf, shape.H, shape.I, g, False, shape.I, SF_ATOMS[fmt]))
    if fmt == "nvfp4":
        assert np.array_equal(kw["w13_gs"], ew.w13_gs) and np.array_equal(kw["w2_gs"], ew.w2_gs)


# ----------------------------------------------------------------------------- failure detection

@pytest.mark.parametrize("fmt,mode", [("mxfp8", "fused"), ("mxfp8", "split256"), ("mxfp8", "pair"),
                                      ("nvfp4", "fused")])
def test_bounded_wait_timeout_reports_and_context_survives(fmt, mode):
    """A 1 ns limit makes the GEMM's pipeline waits run out: the kernel records
    MOE_ERR_TIMEOUT, waits for its own copies and MMAs, and returns. The status reads
    back, and the same plan with the default limit then computes the same answer.
    (The NVFP4 one-kernel GEMM also has the scale-factor warps' waits.)"""
    shape = _small_case(fmt, T=256, H=2048, I=512, E=4, k=2)
    case = G.float_case(shape)
    run = G.run_gpu(case, **G.MODES[mode])
    good = G.out_f64(run)
    a2 = run.inputs.get("a2")
    run.plan.set_wait_timeout(1)
    run.plan.forward(run.inputs["hidden"], run.inputs["topk_ids"], run.inputs["topk_weights"], run.kweights,
                     l2_act_scale=a2, workspace=run.workspace)
    assert run.plan.last_status(run.workspace) == 7
    run.plan.set_wait_timeout(0)
    out = run.plan.forward(run.inputs["hidden"], run.inputs["topk_ids"], run.inputs["topk_weights"], run.kweights,
                           l2_act_scale=a2, workspace=run.workspace)
    torch.cuda.synchronize()
    assert run.plan.last_status(run.workspace) == 0
    assert np.array_equal(out.float().cpu().numpy(), good)


# ----------------------------------------------------------------------------- seeded random shapes

def _random_shape(i: int):
    """Shape i of a seeded sweep over formats, sizes, expert counts, top-k, token counts (1 to 600),
    routing skew, shared expert and norm: the tile, box and segment boundaries fall in many places."""
    g = np.random.default_rng(9000 + i)
    fmt = ["bf16", "mxfp8", "nvfp4", "mxfp4"][i % 4]
    four_bit = fmt in ("nvfp4", "mxfp4")
    H = int(g.choice([256, 512, 768] if four_bit else [256, 384, 512, 768]))
    I = int(g.choice([256, 512] if four_bit else [128, 256, 384, 512]))
    E = int(g.integers(1, 25))
    k = int(g.integers(1, min(8, E) + 1))
    T = int(g.choice([1, 2, 7, 31, 64, 129, 200, 333, 511, 600]))
    shared = fmt == "nvfp4" and bool(g.integers(0, 2))
    base = W["nvfp4_shared_norm"] if shared else W["mxfp8_prefill_zipf"]
    return S.shrink(base, name=f"random{i}", T=T, H=H, I=I, E=E, k=k, fmt=fmt,
                    zipf_s=float(g.choice([0.0, 1.1])), shared_I=256 if shared else 0, post_norm=shared)


@pytest.mark.parametrize("i", range(36))
def test_random_shapes_match_oracle(i):
    """Every output element of each shape against the oracle, the GEMM mode rotating over the
    one-kernel, two-kernel and CTA-pair variants."""
    shape = _random_shape(i)
    case = G.float_case(shape)
    run = G.run_gpu(case, **G.MODES[["fused", "split256", "pair"][(i // 4) % 3]])
    tokens = list(range(shape.T))
    G.assert_close_allowing_ties(run, case, tokens, G.out_f64(run), G.oracle_out(case), shape.name)
    assert run.plan.last_status(run.workspace) == 0
