"""Pins for the oracle's routing / permutation (CPU only): a hand-worked case,
brute force over every id pattern of tiny shapes against an independent
formulation (a stable library sort), and the permutation invariants."""
import itertools
import json
import os

import numpy as np
import pytest

from oracle.routing import expert_counts, padded_offsets, permute


def test_golden_small(golden_dir):
    with open(os.path.join(golden_dir, "routing_small.json")) as f:
        g = json.load(f)
    cnt, off, src, inv = permute(np.array(g["topk_ids"]), g["num_experts"], g["block_m"])
    assert cnt.tolist() == g["cnt"]
    assert off.tolist() == g["off"]
    assert src.tolist() == g["src"]
    assert inv.tolist() == g["inv_perm"]


def _by_stable_sort(ids, E, bm):
    """Independent route: a stable argsort of the flat ids gives each expert's slots in
    ascending order; rows are the padded segment start plus the rank inside the expert."""
    flat = ids.reshape(-1)
    cnt = np.bincount(flat[flat >= 0], minlength=E)
    seg = -(-cnt // bm) * bm
    start = np.concatenate([[0], np.cumsum(seg)])
    order = np.argsort(np.where(flat >= 0, flat, E), kind="stable")
    first = np.concatenate([[0], np.cumsum(cnt)])     # expert e's slots are order[first[e]:first[e+1]]
    inv = np.full(flat.shape, -1)
    for e in range(E):
        slots = order[first[e]:first[e + 1]]
        inv[slots] = start[e] + np.arange(len(slots))
    return cnt, start, inv.reshape(ids.shape)


def _check_invariants(ids, E, bm, cnt, off, src, inv):
    T, k = ids.shape
    routed = (ids >= 0)
    assert cnt.sum() == routed.sum()
    assert np.all(off % bm == 0) and off[0] == 0 and len(src) == off[-1]
    # inverse is a bijection onto the non-padding rows, and src undoes it
    rows = inv[routed]
    assert len(set(rows.tolist())) == len(rows)
    assert set(rows.tolist()) == set(np.nonzero(src >= 0)[0].tolist())
    for t, j in zip(*np.nonzero(routed)):
        r = inv[t, j]
        assert src[r] == t * k + j
        assert off[ids[t, j]] <= r < off[ids[t, j]] + cnt[ids[t, j]]
    # permute then inverse is the identity on data
    data = np.arange(T * k).reshape(T, k) * 7 + 3
    buf = np.full(max(len(src), 1), -99)
    buf[inv[routed]] = data[routed]
    back = np.where(routed, buf[np.where(routed, inv, 0)], data)
    assert np.array_equal(back, data)


@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (2, 1, 2), (2, 2, 2), (3, 2, 2), (4, 1, 2)])
@pytest.mark.parametrize("bm", [1, 2, 4])
def test_brute_force_all_patterns(T, k, E, bm):
    for pat in itertools.product(range(-1, E), repeat=T * k):
        ids = np.array(pat).reshape(T, k)
        cnt, off, src, inv = permute(ids, E, bm)
        c2, off2, inv2 = _by_stable_sort(ids, E, bm)
        assert np.array_equal(cnt, c2)
        assert np.array_equal(off, off2)
        assert np.array_equal(inv, inv2)
        _check_invariants(ids, E, bm, cnt, off, src, inv)


def test_random_large_invariants():
    rng = np.random.default_rng(7)
    T, k, E, bm = 2048, 8, 64, 128
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    ids[rng.random((T, k)) < 0.01] = -1
    cnt, off, src, inv = permute(ids, E, bm)
    _check_invariants(ids, E, bm, cnt, off, src, inv)
    c2, off2, inv2 = _by_stable_sort(ids, E, bm)
    assert np.array_equal(inv, inv2) and np.array_equal(off, off2)


def test_empty_and_edge():
    cnt, off, src, inv = permute(np.zeros((0, 4), dtype=np.int64), 3, 128)
    assert cnt.tolist() == [0, 0, 0] and off.tolist() == [0, 0, 0, 0] and len(src) == 0
    cnt, off, src, inv = permute(np.full((2, 2), -1), 2, 4)
    assert off[-1] == 0 and np.all(inv == -1)
    with pytest.raises(ValueError):
        expert_counts(np.array([[0, 5]]), 3)
    assert padded_offsets(np.array([0, 1, 128, 129]), 128).tolist() == [0, 0, 128, 256, 512]
