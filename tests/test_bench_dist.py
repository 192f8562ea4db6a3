"""The benchmark's multi-rank host logic on CPU (gloo, world size 2): per-rank
seeds differ, and the reported time is the max over ranks."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, _ = bench.dist_env()
    mx = bench.reduce_max(10.0 + rank)
    bench.barrier()
    q.put((r, w, mx, bench.rank_seed(r)))
    dist.destroy_process_group()


def test_two_rank_max_and_seeds():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 for r in res)
    assert all(r[2] == 11.0 for r in res)
    assert res[0][3] != res[1][3]


def test_single_process_identity():
    import bench
    assert bench.reduce_max(3.5) == 3.5


def test_algorithmic_work_counts_touched_experts():
    import numpy as np
    import bench
    import synthetic as S
    shape = S.WORKLOADS["mxfp8_small"]
    ids = np.zeros((shape.T, shape.k), np.int32)
    ids[:, :] = np.arange(shape.k)
    w = bench.algorithmic_work(shape, ids)
    assert w["touched_experts"] == shape.k
    R = shape.T * shape.k
    assert w["flops"] == 2.0 * R * 3 * shape.I * shape.H
    per_expert = 3 * shape.I * shape.H * (1 + 1 / 32)
    assert w["bytes"] == pytest.approx(shape.k * per_expert + 2 * shape.T * shape.H * 2)


def test_roofline_picks_the_binding_resource_and_peak():
    """An HBM-bound kernel is held against copy bandwidth, a tensor-bound one against the format's
    tensor peak (the sustained bf16 figure x the nominal ratio when the power cap acted)."""
    import bench
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1500.0}
    work = {"per_kernel": {"mem": {"fmt": "mxfp8", "bytes": 6e9, "flops": 1e12},
                           "mma": {"fmt": "mxfp8", "bytes": 1e9, "flops": 6e15}}}
    r = bench.roofline("mem", work, 2.0, peaks, "measured", sustained=False)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6000.0
    assert abs(r["achieved"] - 3000.0) < 1e-6 and abs(r["frac"] - 0.5) < 1e-9
    r = bench.roofline("mma", work, 2000.0, peaks, "measured", sustained=True)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["peak"] == 1500.0 * bench.TENSOR_RATIO["mxfp8"]
    assert abs(r["achieved"] - 3000.0) < 1e-6 and abs(r["frac"] - 3000.0 / r["peak"]) < 1e-6
    r = bench.roofline("mma", work, 2000.0, peaks, "measured", sustained=False)
    assert r["peak"] == 2000.0 * bench.TENSOR_RATIO["mxfp8"]


def test_binding_accepts_host_memory_only_where_documented():
    """Device tensors everywhere; a CPU tensor is refused unless pinned and the argument allows it."""
    import torch
    from serving_topk_permute_gb300 import moe as M
    t = torch.zeros(4)
    with pytest.raises(ValueError):
        M._ptr(t)
    with pytest.raises(ValueError):
        M._ptr(t, host_ok=True)   # not pinned
    assert M._ptr(None) is None
