"""C-ABI checks that need no GPU: libmoe.so loads, exports every function
include/moe.h declares, and the host-only calls (validation, workspace sizing,
status strings) behave as documented."""
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def pkg():
    import serving_topk_permute_gb300 as p
    if not os.path.exists(p.library_path()):
        from serving_topk_permute_gb300 import build
        build.build()
    return p


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(moe_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("moe_plan", "moe_transform_weights", "moe_forward", "moe_workspace_size", "moe_last_status"):
        assert must in names


def test_every_declared_symbol_is_exported(pkg):
    lib = pkg.lib()
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing


def _cfg(pkg, **kw):
    base = dict(num_experts=8, hidden=256, inter=256, top_k=2, max_tokens=64, fmt="bf16")
    base.update(kw)
    return pkg.LayerConfig(**base)


@pytest.mark.parametrize("kw,status", [
    ({}, 0),
    ({"fmt": "mxfp8"}, 0),
    ({"fmt": "nvfp4"}, 0),
    ({"hidden": 384, "fmt": "mxfp8"}, 0),
    ({"hidden": 384, "fmt": "nvfp4"}, 1),          # NVFP4 needs multiples of 256
    ({"hidden": 200}, 1),                           # multiples of 128
    ({"inter": 64}, 1),
    ({"top_k": 9}, 1),                              # top_k <= num_experts
    ({"top_k": 0}, 1),
    ({"num_experts": 1024, "top_k": 2}, 1),         # E <= 512
    ({"max_tokens": 0}, 1),
    ({"act_clamp": -1.0}, 1),                       # clamp >= 0
    ({"act_alpha": float("inf")}, 1),               # finite alpha / beta
    ({"act_beta": float("nan")}, 1),
    ({"shared_inter": 100}, 1),
    ({"shared_inter": 384, "shared_fmt": "bf16"}, 1),
    ({"shared_inter": 384, "shared_fmt": "mxfp8"}, 0),
    ({"shared_inter": 256, "shared_fmt": "nvfp4"}, 2),
    ({"norm_eps": -1.0}, 1),
])
def test_validation(pkg, kw, status):
    assert pkg.validate(_cfg(pkg, **kw)) == status


def test_unknown_format_is_unsupported(pkg):
    c = _cfg(pkg).to_c()
    c.format = 7
    import ctypes
    assert pkg.lib().moe_config_validate(ctypes.byref(c)) == 2


def test_workspace_size(pkg):
    cfg = _cfg(pkg, fmt="mxfp8", max_tokens=512)
    sizes = [pkg.config_workspace_size(cfg, t) for t in (0, 1, 64, 512)]
    assert all(s > 0 for s in sizes)
    assert sizes == sorted(sizes)
    with pytest.raises(pkg.MoeError) as e:
        pkg.config_workspace_size(cfg, 513)
    assert e.value.status == 3


def test_error_strings(pkg):
    assert pkg.error_string(0) == "ok"
    for s in range(1, 8):
        assert pkg.error_string(s) and pkg.error_string(s) != "unknown status"
    assert pkg.error_string(99) == "unknown status"


def test_noalloc_binding_refuses_host_tensors(pkg):
    """moe_permute_noalloc reads raw device buffers: the binding refuses host or 1-D ids
    before anything reaches the library."""
    import torch
    with pytest.raises(ValueError):
        pkg.permute_noalloc(torch.zeros((4, 2), dtype=torch.int32), 8)
    with pytest.raises(ValueError):
        pkg.permute_noalloc(torch.zeros(8, dtype=torch.int32), 8)


def _defines(prefix: str) -> dict:
    """The #define constants of include/moe.h whose names start with prefix."""
    out = {}
    for m in re.finditer(r"^#define\s+(" + prefix + r"\w+)\s+(\d+)u?\b", open(HEADER).read(), flags=re.M):
        out[m.group(1)] = int(m.group(2))
    return out


def _struct_fields(name: str) -> list:
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct " + name + r" \{(.*?)\}", text, flags=re.S).group(1)
    return re.findall(r"(\w+)\s*;", body)


def test_binding_constants_match_the_header(pkg):
    """The Python binding restates the header's numbers: formats, flags, weight ids, workspace
    regions, kernel timing slots, status codes, and the field order of the two structs it passes."""
    from serving_topk_permute_gb300 import moe as M
    fmts = _defines("MOE_FMT_")
    assert {k: fmts["MOE_FMT_" + k.upper()] for k in M.FORMATS} == M.FORMATS
    flags = _defines("MOE_FLAG_")
    assert flags["MOE_FLAG_DEBUG_H"] == M.FLAG_DEBUG_H
    assert flags["MOE_FLAG_TILE_128"] == M.FLAG_TILE[128] and flags["MOE_FLAG_TILE_256"] == M.FLAG_TILE[256]
    assert flags["MOE_FLAG_CTA_PAIR"] == M.FLAG_CTA["pair"] and flags["MOE_FLAG_CTA_SINGLE"] == M.FLAG_CTA["single"]
    assert flags["MOE_FLAG_SERIAL"] == M.FLAG_SERIAL and flags["MOE_FLAG_SPLIT_GEMM"] == M.FLAG_SPLIT_GEMM
    w = _defines("MOE_W") | _defines("MOE_SHARED_W")
    assert [w[n] for n in ("MOE_W13", "MOE_W13_SF", "MOE_W2", "MOE_W2_SF", "MOE_SHARED_W13", "MOE_SHARED_W13_SF",
                           "MOE_SHARED_W2", "MOE_SHARED_W2_SF", "MOE_W13_GS", "MOE_W2_GS")] == [
        M.W13, M.W13_SF, M.W2, M.W2_SF, M.SHARED_W13, M.SHARED_W13_SF, M.SHARED_W2, M.SHARED_W2_SF, M.W13_GS, M.W2_GS]
    regions = _defines("MOE_REGION_")
    names = {"counts": "COUNTS", "offsets": "OFFSETS", "src": "SRC", "inv_perm": "INV_PERM", "xq": "XQ", "xsf": "XSF",
             "x_scale": "XSCALE", "hq": "HQ", "hsf": "HSF", "h_debug": "H_DEBUG", "y": "Y", "meta": "META",
             "shared_y": "SHARED_Y"}
    assert {k: regions["MOE_REGION_" + v] for k, v in names.items()} == M.REGIONS
    kernels = _defines("MOE_KERNEL_")
    assert [kernels["MOE_KERNEL_" + k.upper()] for k in M.KERNELS] == list(range(len(M.KERNELS)))
    every = _defines("MOE_")
    assert every["MOE_NUM_KERNELS"] == len(M.KERNELS)
    assert every["MOE_OK"] == M.MOE_OK == 0
    assert [f for f, _ in M.Config._fields_] == _struct_fields("moe_config")
    assert [f for f, _ in M.Weights._fields_] == _struct_fields("moe_weights")
