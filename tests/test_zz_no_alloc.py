"""moe_permute_noalloc, the routing permutation for callers that must not allocate
device memory (a runtime that owns all of HBM through its own pools, or a path
where cudaMalloc is not allowed): its scratch is a fixed array inside libmoe.so.

Checked three ways, through the C ABI:
  * against the permutation moe_forward computes in its workspace: the same
    inverse permutation and segment offsets, bit for bit, on two calls in a row
    and again after a call of another shape reused the shared array;
  * against the oracle's stable scatter (oracle/routing.py) at the entry point's
    limits: E = 512, k = 32 and exactly T*k + E*127 = 262144 padded rows, with
    masked (-1) and out-of-range ids (which it treats as masked);
  * its errors: one row over the limit is rejected before anything is written,
    T = 0 takes null id and inverse pointers, and the binding refuses tensors of
    the wrong type or shape.
Collected last on purpose."""
import numpy as np
import pytest
import torch

import synthetic as S
import gpu_case as G
from oracle import routing as OR

pytestmark = pytest.mark.gpu

MAX_ROWS = 262144
MOE_ERR_CAPACITY = 3


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


def _noalloc(ids: torch.Tensor, E: int):
    import serving_topk_permute_gb300 as pkg
    got_inv = torch.full(tuple(ids.shape), -7, dtype=torch.int32, device=ids.device)
    got_off = torch.full((E + 1,), -7, dtype=torch.int32, device=ids.device)
    pkg.permute_noalloc(ids, E, got_inv, got_off)
    torch.cuda.synchronize()
    return got_inv.cpu().numpy(), got_off.cpu().numpy()


def _oracle(ids: np.ndarray, E: int):
    """The oracle's permutation with BLOCK_M = 128; ids outside [-1, E) count as masked."""
    masked = np.where((ids >= 0) & (ids < E), ids, -1)
    cnt, off, src, inv = OR.permute(masked, E, 128)
    return inv.astype(np.int32), off.astype(np.int32)


def test_noalloc_permutation_matches_forward():
    a = S.shrink(S.WORKLOADS["mxfp8_prefill_zipf"], T=300, H=256, I=256, E=32, k=8)
    b = S.shrink(S.WORKLOADS["mxfp8_small"], T=77, H=256, I=256, E=64, k=4)
    ids_a, inv_a, off_a = _forward_routing(a)
    ids_b, inv_b, off_b = _forward_routing(b)
    for ids, inv, off, E in ((ids_a, inv_a, off_a, a.E), (ids_a, inv_a, off_a, a.E), (ids_b, inv_b, off_b, b.E),
                             (ids_a, inv_a, off_a, a.E)):
        got_inv, got_off = _noalloc(ids, E)
        assert np.array_equal(got_inv, inv)
        assert np.array_equal(got_off, off)


def test_noalloc_matches_oracle_at_its_limits():
    # E = 512 and k = 32 (both maxima) with T * k + E * 127 = 262144 exactly (the array's capacity)
    E, k = 512, 32
    T = (MAX_ROWS - E * 127) // k
    assert T * k + E * 127 == MAX_ROWS
    shape = S.shrink(S.WORKLOADS["mxfp8_small"], T=T, E=E, k=k)
    ids, _ = S.router(shape, 3)
    ids = np.array(ids, np.int32)
    want_inv, want_off = _oracle(ids, E)
    assert want_off[-1] <= MAX_ROWS
    d = torch.from_numpy(ids).cuda()
    for _ in range(2):  # two calls in a row on the shared array
        got_inv, got_off = _noalloc(d, E)
        assert np.array_equal(got_off, want_off)
        assert np.array_equal(got_inv, want_inv)


def test_noalloc_masked_and_out_of_range_ids_match_oracle():
    shape = S.shrink(S.WORKLOADS["mxfp8_prefill_zipf"], T=1000, E=96, k=6)
    ids, _ = S.router(shape, 5)
    ids = np.array(ids, np.int32)
    rng = np.random.default_rng(11)
    flat = ids.reshape(-1)
    pick = rng.choice(flat.size, size=flat.size // 5, replace=False)
    # a mix of masked slots (-1) and ids outside [-1, E), which the entry point treats as masked
    flat[pick] = rng.choice(np.array([-1, -1, -1, -2, shape.E, shape.E + 7, -1000], np.int32), size=pick.size)
    ids[0, :] = -1        # a token with every slot masked
    ids[1, :] = ids[2, 0]  # a token whose slots all pick one expert
    want_inv, want_off = _oracle(ids, shape.E)
    got_inv, got_off = _noalloc(torch.from_numpy(ids).cuda(), shape.E)
    assert np.array_equal(got_off, want_off)
    assert np.array_equal(got_inv, want_inv)
    assert (got_inv[0] == -1).all()


def test_noalloc_zero_tokens_and_capacity():
    import serving_topk_permute_gb300 as pkg
    E = 16
    # T = 0: null ids and inverse; every segment is empty
    got_inv, got_off = _noalloc(torch.zeros((0, 4), dtype=torch.int32, device="cuda"), E)
    assert got_inv.shape == (0, 4)
    assert np.array_equal(got_off, np.zeros(E + 1, np.int32))
    # one padded row over the array: rejected before launch, outputs untouched
    k = 1
    T = MAX_ROWS - E * 127 + 1
    ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    inv = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    with pytest.raises(pkg.MoeError) as e:
        pkg.permute_noalloc(ids, E, inv, off)
    assert e.value.status == MOE_ERR_CAPACITY
    torch.cuda.synchronize()
    assert (off.cpu() == -7).all() and (inv.cpu() == -7).all()
    # exactly at the limit with the same E and k is accepted
    T = MAX_ROWS - E * 127
    ids = torch.arange(T, dtype=torch.int32, device="cuda").remainder(E).reshape(T, k)
    got_inv, got_off = _noalloc(ids, E)
    want_inv, want_off = _oracle(ids.cpu().numpy(), E)
    assert np.array_equal(got_off, want_off) and np.array_equal(got_inv, want_inv)
    # the large rejection of before
    with pytest.raises(pkg.MoeError) as e:
        pkg.permute_noalloc(torch.zeros((40000, 8), dtype=torch.int32, device="cuda"), 16)
    assert e.value.status == MOE_ERR_CAPACITY


def test_noalloc_binding_refuses_wrong_tensors():
    import serving_topk_permute_gb300 as pkg
    ids64 = torch.zeros((8, 2), dtype=torch.int64, device="cuda")   # torch.topk's default index type
    with pytest.raises(ValueError):
        pkg.permute_noalloc(ids64, 4)
    ids = torch.zeros((8, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        pkg.permute_noalloc(ids, 4, expert_offsets=torch.zeros(4, dtype=torch.int32, device="cuda"))
    with pytest.raises(ValueError):
        pkg.permute_noalloc(ids, 4, inv_perm=torch.zeros((8, 3), dtype=torch.int32, device="cuda"))
    with pytest.raises(ValueError):
        pkg.permute_noalloc(ids.reshape(-1), 4)
