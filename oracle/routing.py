"""Oracle routing: per-expert histogram, BLOCK_M-padded segment offsets, stable permutation.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Follows vllm.model_executor.layers.fused_moe (DeepGemmExperts.workspace_shapes and
DeepGemmExperts.apply): the permuted buffer holds every routed (token, slot)
row, grouped by expert, each expert's segment padded to a multiple of
BLOCK_M (``compute_aligned_M``, ``assert M_sum % block_m == 0``), and the
permute returns the inverse permutation the combine uses
(``deepgemm_moe_permute`` -> ``inv_perm``).

Readings where the pages are silent:
  * rows inside one expert's segment are ordered by ascending flat slot
    s = t * k + j (a stable scatter);
  * a slot whose id is -1 is masked (not routed here): it gets no row and its
    inverse entry is -1; padding rows have source -1.
"""
from __future__ import annotations

import numpy as np


def expert_counts(topk_ids: np.ndarray, num_experts: int) -> np.ndarray:
    """cnt[e] = number of (t, j) with topk_ids[t, j] == e (masked -1 slots skipped)."""
    ids = np.asarray(topk_ids).reshape(-1)
    if ((ids < -1) | (ids >= num_experts)).any():
        raise ValueError("expert id out of range")
    cnt = np.zeros(num_experts, dtype=np.int64)
    for e in ids:
        if e >= 0:
            cnt[e] += 1
    return cnt


def padded_offsets(cnt: np.ndarray, block_m: int) -> np.ndarray:
    """off[0] = 0, off[e+1] = off[e] + ceil(cnt[e] / BLOCK_M) * BLOCK_M."""
    off = np.zeros(len(cnt) + 1, dtype=np.int64)
    for e, c in enumerate(cnt):
        off[e + 1] = off[e] + ((int(c) + block_m - 1) // block_m) * block_m
    return off


def permute(topk_ids: np.ndarray, num_experts: int, block_m: int):
    """Stable scatter of routed slots into BLOCK_M-padded expert segments.

    Returns ``(cnt [E], off [E+1], src [M_pad], inv_perm [T, k])`` where
    ``src[row]`` is the flat slot routed to ``row`` (or -1 for padding) and
    ``inv_perm[t, j]`` is the row of slot (t, j) (or -1 if masked).
    """
    ids = np.asarray(topk_ids)
    T, k = ids.shape
    cnt = expert_counts(ids, num_experts)
    off = padded_offsets(cnt, block_m)
    fill = np.zeros(num_experts, dtype=np.int64)
    src = np.full(int(off[-1]), -1, dtype=np.int64)
    inv = np.full((T, k), -1, dtype=np.int64)
    for s in range(T * k):
        t, j = divmod(s, k)
        e = int(ids[t, j])
        if e < 0:
            continue
        row = int(off[e] + fill[e])
        fill[e] += 1
        src[row] = s
        inv[t, j] = row
    return cnt, off, src, inv
