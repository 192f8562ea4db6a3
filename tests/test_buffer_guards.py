"""Guard bytes around every caller-owned buffer (needs a GB300).

Each buffer the library writes (the kernel-layout weights, the workspace, the
output) sits inside a larger allocation whose bytes before and after it hold a
fixed pattern; after the call every guard byte must still hold it, so no kernel
writes outside the sizes that moe_weight_layout_size / moe_workspace_size and
the output shape give. The workspace itself starts filled with the same
pattern instead of zeros: moe_forward must not depend on what a workspace held
before (the output equals the one from a zeroed workspace bit for bit). The
inputs (hidden states, routing, checkpoint and kernel-layout weights, scales,
gamma) must be left unchanged.
"""
import ctypes

import numpy as np
import pytest
import torch

import synthetic as S
import gpu_case as G
import serving_topk_permute_gb300 as pkg
from serving_topk_permute_gb300 import moe as M

pytestmark = pytest.mark.gpu

W = S.WORKLOADS
GUARD = 4096          # bytes on each side; a multiple of 256 keeps the inner buffer 256-byte aligned
PATTERN = 0xA5

SHAPES = {
    "bf16": S.shrink(W["bf16_toy"], T=77),
    "mxfp8": S.shrink(W["mxfp8_small"], T=200, H=512, I=384, E=16, k=4),
    "nvfp4": S.shrink(W["nvfp4_shared_norm"], T=130, H=512, I=256, E=16, k=4, shared_I=512),
    "mxfp4": S.shrink(W["mxfp4_small"], T=150, H=512, I=512, E=16, k=4),
}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    pkg.lib()


class Guarded:
    """nbytes of device memory between two GUARD-byte runs of PATTERN."""

    def __init__(self, nbytes: int, fill=PATTERN):
        self.n = nbytes
        self.buf = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8, device=G.dev())
        if fill != PATTERN:
            self.buf[GUARD:GUARD + nbytes].fill_(fill)

    def inner(self, dtype=torch.uint8) -> torch.Tensor:
        return self.buf[GUARD:GUARD + self.n].view(dtype)

    def check(self, what: str):
        head = self.buf[:GUARD].cpu().numpy()
        tail = self.buf[GUARD + self.n:].cpu().numpy()
        bad_head = np.flatnonzero(head != PATTERN)
        bad_tail = np.flatnonzero(tail != PATTERN)
        assert bad_head.size == 0, f"{what}: {bad_head.size} bytes written before the buffer (first at -{GUARD - bad_head[0]})"
        assert bad_tail.size == 0, f"{what}: {bad_tail.size} bytes written past the end (first at +{bad_tail[0]})"


def _guarded_layout(plan: pkg.Plan, ids: dict) -> tuple[dict, dict]:
    tensors, guards = {}, {}
    for key, which in ids.items():
        n = plan.weight_layout_size(which)
        if not n:
            continue
        g = Guarded(n)
        guards[key] = g
        tensors[key] = g.inner(torch.float32 if key.endswith("_gs") else torch.uint8)
    return tensors, guards


def _transform(plan: pkg.Plan, ckpt: dict, shared: bool):
    if shared:
        ids = {"w13": M.SHARED_W13, "w13_sf": M.SHARED_W13_SF, "w2": M.SHARED_W2, "w2_sf": M.SHARED_W2_SF}
        fn = M.lib().moe_transform_shared_weights
        name = "moe_transform_shared_weights"
    else:
        ids = {"w13": M.W13, "w13_sf": M.W13_SF, "w2": M.W2, "w2_sf": M.W2_SF, "w13_gs": M.W13_GS,
               "w2_gs": M.W2_GS}
        fn = M.lib().moe_transform_weights
        name = "moe_transform_weights"
    dst, guards = _guarded_layout(plan, ids)
    s, d = M._weights_struct(ckpt), M._weights_struct(dst)
    M._check(name, fn(plan._h, ctypes.byref(s), ctypes.byref(d), M._stream(None)))
    return dst, guards


def _snapshot(d: dict) -> dict:
    return {k: v.clone() for k, v in d.items() if v is not None}


def _assert_unchanged(before: dict, after: dict, what: str):
    for k, v in before.items():
        assert torch.equal(v.view(torch.uint8) if v.dtype != torch.uint8 else v,
                           after[k].view(torch.uint8) if after[k].dtype != torch.uint8 else after[k]), \
            f"{what}: input {k} was written"


@pytest.mark.parametrize("fmt,mode", [("bf16", "fused"), ("mxfp8", "fused"), ("mxfp8", "split256"),
                                      ("mxfp8", "pair"), ("mxfp8", "single128"), ("nvfp4", "fused"),
                                      ("nvfp4", "pair"), ("mxfp4", "fused")])
def test_forward_writes_only_its_buffers(fmt, mode):
    case = G.float_case(SHAPES[fmt])
    ref = G.run_gpu(case, **G.MODES[mode])           # zeroed workspace, library-sized buffers
    plan = ref.plan
    T, H = case.x.shape

    ck = G._ckpt_dev(case.layer.routed)
    ck_before = _snapshot(ck)
    kw, kw_guards = _transform(plan, ck, shared=False)
    ks, ks_guards = None, {}
    if case.layer.shared is not None:
        sck = G._ckpt_dev(case.layer.shared)
        sck_before = _snapshot(sck)
        ks, ks_guards = _transform(plan, sck, shared=True)
    torch.cuda.synchronize()
    for key, g in {**kw_guards, **{"shared " + k: v for k, v in ks_guards.items()}}.items():
        g.check(f"{fmt} {mode} layout {key}")
    _assert_unchanged(ck_before, ck, "routed transform")
    if ks is not None:
        _assert_unchanged(sck_before, sck, "shared transform")
        for k in ks:
            assert torch.equal(ks[k], ref.kshared[k]), f"shared layout {k} differs from the binding's"
    for k in kw:
        assert torch.equal(kw[k].view(torch.uint8), ref.kweights[k].view(torch.uint8)), \
            f"layout {k} differs from the binding's"

    ws = Guarded(plan.workspace_size(T))             # workspace starts as the guard pattern, not zeros
    out = Guarded(T * H * 2)
    inputs = {k: v for k, v in ref.inputs.items() if v is not None}
    in_before = _snapshot(inputs)
    kw_before = _snapshot(kw)
    for rep in range(2):                              # the second forward reuses the first's workspace
        plan.forward(inputs["hidden"], inputs["topk_ids"], inputs["topk_weights"], kw,
                     l2_act_scale=inputs.get("a2"), shared=ks, norm_gamma=inputs.get("gamma"),
                     out=out.inner(torch.bfloat16).view(T, H), workspace=ws.inner())
        torch.cuda.synchronize()
        assert plan.last_status(ws.inner()) == 0
        ws.check(f"{fmt} {mode} workspace, forward {rep}")
        out.check(f"{fmt} {mode} output, forward {rep}")
        got = out.inner(torch.int16).view(T, H)
        assert torch.equal(got, ref.out.view(torch.int16)), f"forward {rep} on a patterned workspace differs"
    _assert_unchanged(in_before, inputs, "forward")
    _assert_unchanged(kw_before, kw, "forward (kernel-layout weights)")


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_batched_forward_writes_only_its_buffers(fmt):
    """moe_forward_batched: guards around its workspace and output; rows past each expert's
    count keep the pattern; a patterned workspace gives the zeroed one's output."""
    E, Mt = 5, 256
    shape = S.shrink(W["mxfp8_small"] if fmt == "mxfp8" else W["nvfp4_decode"], T=E * Mt, H=512, I=256, E=E, k=1)
    case = G.float_case(shape)
    plan = pkg.Plan(G.layer_config(case))
    kw = plan.transform_weights(G._ckpt_dev(case.layer.routed))
    a2 = torch.tensor([np.float32(case.layer.a2)], device=G.dev()) if fmt == "nvfp4" else None
    counts = G.to_dev(np.array([0, 1, 129, 256, 77], np.int32))
    hidden = G.bf16_dev(case.x).view(E, Mt, -1)
    H = shape.H

    ref = torch.zeros((E, Mt, H), dtype=torch.bfloat16, device=G.dev())
    plan.forward_batched(hidden, counts, kw, l2_act_scale=a2, out=ref,
                         workspace=torch.zeros(plan.batched_workspace_size(Mt), dtype=torch.uint8, device=G.dev()))
    ws = Guarded(plan.batched_workspace_size(Mt))
    out = Guarded(E * Mt * H * 2)
    before = hidden.clone()
    plan.forward_batched(hidden, counts, kw, l2_act_scale=a2, out=out.inner(torch.bfloat16).view(E, Mt, H),
                         workspace=ws.inner())
    torch.cuda.synchronize()
    assert plan.last_status(ws.inner()) == 0
    ws.check(f"batched {fmt} workspace")
    out.check(f"batched {fmt} output")
    got = out.inner(torch.int16).view(E, Mt, H)
    used = (torch.arange(Mt, device=G.dev())[None, :] < counts[:, None].long())
    assert torch.equal(got[used], ref.view(torch.int16)[used])
    untouched = got[~used].view(torch.uint8) if got[~used].numel() else torch.empty(0, dtype=torch.uint8)
    assert bool((untouched == PATTERN).all()), "rows past expert_num_tokens were written"
    assert torch.equal(before, hidden)
