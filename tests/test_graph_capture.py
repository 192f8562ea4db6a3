"""moe_forward and moe_forward_batched inside a CUDA graph: captured once on a side stream (no
host synchronisation, no allocation inside the forward), then replayed with new inputs copied
into the captured buffers. Every replay equals an eager forward on the same inputs, bit for bit."""
import numpy as np
import pytest
import torch

import synthetic as S
import gpu_case as G

pytestmark = pytest.mark.gpu


def _inputs(shape, seed):
    x = S.hidden_states(shape, seed)
    ids, w = S.router(shape, seed)
    return G.bf16_dev(x), G.to_dev(ids.astype(np.int32)), G.to_dev(w.astype(np.float32))


@pytest.mark.parametrize("name", ["mxfp8_small", "nvfp4_shared_norm"])
def test_forward_replays_in_a_graph(name):
    from test_gpu_parity import REDUCED
    shape = REDUCED[name]
    case = G.float_case(shape)
    run = G.run_gpu(case)
    plan, kw, ks = run.plan, run.kweights, run.kshared
    a2, gamma = run.inputs["a2"], run.inputs["gamma"]
    h, ids, w = (t.clone() for t in _inputs(shape, 0))
    out = torch.empty_like(h)
    ws = plan.alloc_workspace(shape.T)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        plan.forward(h, ids, w, kw, l2_act_scale=a2, shared=ks, norm_gamma=gamma, out=out, workspace=ws)  # warm-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        plan.forward(h, ids, w, kw, l2_act_scale=a2, shared=ks, norm_gamma=gamma, out=out, workspace=ws,
                     stream=side)
    for seed in (1, 2, 3):
        nh, nids, nw = _inputs(shape, seed)
        h.copy_(nh), ids.copy_(nids), w.copy_(nw)
        g.replay()
        want = plan.forward(nh, nids, nw, kw, l2_act_scale=a2, shared=ks, norm_gamma=gamma)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), want.view(torch.int16)), seed
    assert plan.last_status(ws) == 0


def test_batched_forward_replays_in_a_graph():
    shape = S.shrink(S.WORKLOADS["nvfp4_decode"], T=64, H=512, I=256, E=6, k=1)
    case = G.float_case(shape)
    run = G.run_gpu(case)
    plan, kw, a2 = run.plan, run.kweights, run.inputs["a2"]
    M = 256
    rng = np.random.default_rng(5)
    xb = torch.from_numpy(S.hidden_states(S.shrink(shape, T=shape.E * M), 0).view(np.int16)).cuda().view(torch.bfloat16)
    hb = xb.view(shape.E, M, shape.H).clone()
    counts = torch.zeros(shape.E, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(hb)
    ws = torch.zeros(plan.batched_workspace_size(M), dtype=torch.uint8, device="cuda")
    plan.forward_batched(hb, counts, kw, l2_act_scale=a2, out=out, workspace=ws)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        plan.forward_batched(hb, counts, kw, l2_act_scale=a2, out=out, workspace=ws, stream=side)
    for _ in range(3):
        c = torch.from_numpy(rng.integers(0, M + 1, size=shape.E).astype(np.int32)).cuda()
        counts.copy_(c)
        out.zero_()
        g.replay()
        want = plan.forward_batched(hb.clone(), c, kw, l2_act_scale=a2)
        torch.cuda.synchronize()
        for e in range(shape.E):
            n = int(c[e])
            assert torch.equal(out[e, :n].view(torch.int16), want[e, :n].view(torch.int16))
    assert plan.last_status(ws) == 0
