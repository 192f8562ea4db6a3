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
