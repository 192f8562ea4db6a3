"""The C ABI from plain C: tests/c_abi_forward.c (include/moe.h and the CUDA runtime only, no
Python or torch in the process) is compiled against libmoe.so with the system C compiler and runs
one forward of a seeded case: plan, weight transform, workspace, forward, status. Its output must
equal the Python binding's bit for bit and match the oracle within the layer's tolerance."""
import os
import shutil
import struct
import subprocess

import numpy as np
import pytest
import torch

import synthetic as S
import gpu_case as G
import serving_topk_permute_gb300 as pkg
from conftest import ROOT

pytestmark = pytest.mark.gpu

FMT_CODE = {"bf16": 0, "mxfp8": 1, "nvfp4": 2, "mxfp4": 3}


def _compile(tmp_path) -> str:
    cc = shutil.which("gcc") or shutil.which("cc")
    assert cc, "a C compiler is needed"
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    lib_dir = os.path.dirname(pkg.library_path())
    exe = str(tmp_path / "c_abi_forward")
    cmd = [cc, "-std=c99", "-O2", os.path.join(ROOT, "tests", "c_abi_forward.c"), "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), "-L", lib_dir, "-lmoe", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           f"-Wl,-rpath,{lib_dir}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def _write_input(path, case: G.Case):
    s, L = case.shape, case.layer.routed
    blobs = [case.x.astype(np.uint16), case.ids.astype(np.int32), case.w.astype(np.float32),
             L.w13, L.w13_sf, L.w2, L.w2_sf, L.w13_gs, L.w2_gs,
             None if case.layer.a2 is None else np.array([case.layer.a2], np.float32)]
    with open(path, "wb") as f:
        f.write(b"MOEC" + struct.pack("<6i", s.E, s.H, s.I, s.k, s.T, FMT_CODE[s.fmt]))
        for b in blobs:
            raw = b"" if b is None else np.ascontiguousarray(b).tobytes()
            f.write(struct.pack("<q", len(raw)) + raw)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "bf16"])
def test_c_abi_program(fmt, tmp_path):
    base = {"mxfp8": "mxfp8_small", "nvfp4": "nvfp4_decode", "bf16": "bf16_toy"}[fmt]
    shape = S.shrink(S.WORKLOADS[base], T=150, H=512, I=256, E=12, k=4)
    case = G.float_case(shape)
    inp, outp = str(tmp_path / "in.bin"), str(tmp_path / "out.bin")
    _write_input(inp, case)
    exe = _compile(tmp_path)
    r = subprocess.run([exe, inp, outp], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr + r.stdout
    with open(outp, "rb") as f:
        n = struct.unpack("<q", f.read(8))[0]
        got = np.frombuffer(f.read(n), dtype=np.uint16).reshape(shape.T, shape.H)
    run = G.run_gpu(case)
    torch.cuda.synchronize()
    assert np.array_equal(got, run.out.view(torch.int16).cpu().numpy().view(np.uint16))
    got_f64 = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    G.assert_close(got_f64, G.oracle_out(case), fmt, f"C program {fmt}")
