"""moe_permute_noalloc, the routing permutation for callers that must not allocate
device memory (its scratch is a fixed array inside libmoe.so), against the
permutation moe_forward computes in its workspace: same inverse permutation and
segment offsets, bit for bit, on two calls in a row, and again after a call of
another shape reused the shared array. Collected last on purpose."""
import numpy as np
import pytest
import torch

import synthetic as S
import gpu_case as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)


def _forward_routing(shape):
    case = G.float_case(shape)
    run = G.run_gpu(case)
    T, k, E = shape.T, shape.k, shape.E
    inv = G.region_i32(run, T, "inv_perm")[:T * k].reshape(T, k)
    off = G.region_i32(run, T, "offsets")[:E + 1]
    return run.inputs["topk_ids"], inv, off


def test_noalloc_permutation_matches_forward():
    import serving_topk_permute_gb300 as pkg
    a = S.shrink(S.WORKLOADS["mxfp8_prefill_zipf"], T=300, H=256, I=256, E=32, k=8)
    b = S.shrink(S.WORKLOADS["mxfp8_small"], T=77, H=256, I=256, E=64, k=4)
    ids_a, inv_a, off_a = _forward_routing(a)
    ids_b, inv_b, off_b = _forward_routing(b)
    for ids, inv, off, E in ((ids_a, inv_a, off_a, a.E), (ids_a, inv_a, off_a, a.E), (ids_b, inv_b, off_b, b.E),
                             (ids_a, inv_a, off_a, a.E)):
        got_inv = torch.full(ids.shape, -7, dtype=torch.int32, device=ids.device)
        got_off = torch.full((E + 1,), -7, dtype=torch.int32, device=ids.device)
        pkg.permute_noalloc(ids, E, got_inv, got_off)
        torch.cuda.synchronize()
        assert np.array_equal(got_inv.cpu().numpy(), inv)
        assert np.array_equal(got_off.cpu().numpy(), off)


def test_noalloc_rejects_sizes_beyond_its_array():
    import serving_topk_permute_gb300 as pkg
    ids = torch.zeros((40000, 8), dtype=torch.int32, device="cuda")
    with pytest.raises(pkg.MoeError) as e:
        pkg.permute_noalloc(ids, 16)
    assert e.value.status == 3
