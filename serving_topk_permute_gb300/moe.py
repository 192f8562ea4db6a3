"""Thin Python binding of libmoe.so (include/moe.h): argument marshalling only.

Every step of the layer runs in the library's CUDA kernels; PyTorch only
provides device memory (tensors) and the current stream. If the library is
missing this module raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libmoe.so")
_lib = None

MOE_OK = 0
FORMATS = {"bf16": 0, "mxfp8": 1, "nvfp4": 2, "mxfp4": 3}

# weight tensor ids (moe_weight_layout_size)
W13, W13_SF, W2, W2_SF, SHARED_W13, SHARED_W13_SF, SHARED_W2, SHARED_W2_SF, W13_GS, W2_GS = range(10)
# workspace regions (moe_workspace_region)
REGIONS = {"counts": 0, "offsets": 1, "src": 2, "inv_perm": 3, "xq": 4, "xsf": 5, "x_scale": 6, "hq": 7,
           "hsf": 8, "h_debug": 9, "y": 10, "meta": 11, "shared_y": 12}
FLAG_DEBUG_H = 1
FLAG_TILE = {0: 0, 128: 2, 256: 4}   # GEMM tile width: 0 = the library's choice
FLAG_CTA = {"auto": 0, "pair": 8, "single": 16}   # GEMMs on CTA pairs: by rows per expert / always / never
FLAG_SERIAL = 32   # no programmatic dependent launch between the forward's kernels
FLAG_SPLIT_GEMM = 64   # L1 and L2 as two kernels instead of one
KERNELS = ["route", "dispatch", "l1", "l2", "shared_l1", "shared_l2", "combine"]


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status} ({error_string(status)})")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("num_experts", ctypes.c_int32), ("hidden", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("max_tokens", ctypes.c_int32), ("format", ctypes.c_int32),
                ("activation", ctypes.c_int32), ("act_alpha", ctypes.c_float), ("act_beta", ctypes.c_float),
                ("act_clamp", ctypes.c_float), ("act_has_clamp", ctypes.c_int32),
                ("shared_inter", ctypes.c_int32), ("shared_format", ctypes.c_int32),
                ("post_norm", ctypes.c_int32), ("norm_eps", ctypes.c_float), ("flags", ctypes.c_uint32)]


class Weights(ctypes.Structure):
    _fields_ = [("w13", ctypes.c_void_p), ("w13_sf", ctypes.c_void_p), ("w13_gs", ctypes.c_void_p),
                ("w2", ctypes.c_void_p), ("w2_sf", ctypes.c_void_p), ("w2_gs", ctypes.c_void_p)]


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libmoe.so is not built ({_LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(_LIB_PATH)
        P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        sigs = {
            "moe_config_validate": [P],
            "moe_plan": [P, P],
            "moe_plan_destroy": [P],
            "moe_plan_block_m": [P, I32, P],
            "moe_workspace_size": [P, I32, P],
            "moe_config_workspace_size": [P, I32, P],
            "moe_weight_layout_size": [P, I32, P],
            "moe_transform_weights": [P, P, P, P],
            "moe_transform_shared_weights": [P, P, P, P],
            "moe_forward": [P, I32, P, P, P, P, P, P, P, P, P, SZ, P],
            "moe_last_status": [P, P, P, P],
            "moe_workspace_region": [P, I32, I32, P, P],
            "moe_plan_enable_timing": [P, I32],
            "moe_plan_kernel_times": [P, P, I32],
            "moe_permute_noalloc": [P, I32, I32, I32, P, P, P],
            "moe_plan_set_wait_timeout": [P, ctypes.c_uint64],
            "moe_batched_workspace_size": [P, I32, P],
            "moe_forward_batched": [P, I32, P, P, P, P, P, P, SZ, P],
        }
        for name, args in sigs.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        L.moe_error_string.argtypes = [I32]
        L.moe_error_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def error_string(status: int) -> str:
    return lib().moe_error_string(status).decode()


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoeError(fn, status)


def _ptr(t, host_ok: bool = False) -> int | None:
    """Device address of t. With host_ok, a pinned CPU tensor is also accepted: under
    unified addressing its pointer is valid on the device (the kernels access it over
    the host link)."""
    if t is None:
        return None
    if not t.is_cuda and not (host_ok and t.is_pinned()):
        raise ValueError("expected a CUDA tensor" + (" or a pinned CPU tensor" if host_ok else ""))
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def permute_noalloc(topk_ids: torch.Tensor, num_experts: int, inv_perm: torch.Tensor | None = None,
                    expert_offsets: torch.Tensor | None = None, stream=None):
    """moe_permute_noalloc: the routing permutation with the library's fixed scratch array
    (for callers that must not allocate device memory; the output tensors are the
    caller's). Returns (inv_perm int32 [T, k], expert_offsets int32 [E + 1]).

    The kernel reads and writes raw int32 buffers, so the tensors are checked here:
    int32, contiguous, on one CUDA device, topk_ids 2-D, inv_perm of shape [T, k] and
    expert_offsets with at least E + 1 elements. The call runs with that device
    current, on its current stream unless `stream` is given."""
    if not isinstance(topk_ids, torch.Tensor) or topk_ids.dim() != 2:
        raise ValueError("topk_ids must be a 2-D tensor [T, k]")
    if not topk_ids.is_cuda:
        raise ValueError("topk_ids must be a CUDA tensor")
    dev = topk_ids.device
    T, k = topk_ids.shape
    if inv_perm is None:
        inv_perm = torch.empty((T, k), dtype=torch.int32, device=dev)
    if expert_offsets is None:
        expert_offsets = torch.empty(max(num_experts, 0) + 1, dtype=torch.int32, device=dev)
    for name, t in (("topk_ids", topk_ids), ("inv_perm", inv_perm), ("expert_offsets", expert_offsets)):
        if t.dtype != torch.int32:
            raise ValueError(f"{name} must be int32, got {t.dtype}")
        if not t.is_cuda or t.device != dev:
            raise ValueError(f"{name} must be on {dev}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if tuple(inv_perm.shape) != (T, k):
        raise ValueError(f"inv_perm must have shape {(T, k)}, got {tuple(inv_perm.shape)}")
    if expert_offsets.numel() < num_experts + 1:
        raise ValueError(f"expert_offsets needs at least {num_experts + 1} elements")
    with torch.cuda.device(dev):
        st = torch.cuda.current_stream(dev) if stream is None else stream
        _check("moe_permute_noalloc", lib().moe_permute_noalloc(
            topk_ids.data_ptr() if T else None, T, k, num_experts, inv_perm.data_ptr() if T else None,
            expert_offsets.data_ptr(), st.cuda_stream))
    return inv_perm, expert_offsets


@dataclass
class LayerConfig:
    num_experts: int
    hidden: int
    inter: int
    top_k: int
    max_tokens: int
    fmt: str = "bf16"
    act_alpha: float = 1.0
    act_beta: float = 0.0
    act_clamp: float | None = None
    shared_inter: int = 0
    shared_fmt: str = "mxfp8"
    post_norm: bool = False
    norm_eps: float = 1e-6
    debug_h: bool = False
    tile: int = 0
    cta: str = "auto"
    serial: bool = False
    split_gemm: bool = False

    def to_c(self) -> Config:
        return Config(self.num_experts, self.hidden, self.inter, self.top_k, self.max_tokens, FORMATS[self.fmt], 0,
                      self.act_alpha, self.act_beta, 0.0 if self.act_clamp is None else self.act_clamp,
                      0 if self.act_clamp is None else 1, self.shared_inter, FORMATS[self.shared_fmt],
                      1 if self.post_norm else 0, self.norm_eps,
                      (FLAG_DEBUG_H if self.debug_h else 0) | FLAG_TILE[self.tile] | FLAG_CTA[self.cta]
                      | (FLAG_SERIAL if self.serial else 0) | (FLAG_SPLIT_GEMM if self.split_gemm else 0))


def validate(cfg: LayerConfig) -> int:
    c = cfg.to_c()
    return lib().moe_config_validate(ctypes.byref(c))


def config_workspace_size(cfg: LayerConfig, num_tokens: int) -> int:
    c = cfg.to_c()
    n = ctypes.c_size_t()
    _check("moe_config_workspace_size", lib().moe_config_workspace_size(ctypes.byref(c), num_tokens, ctypes.byref(n)))
    return n.value


def _weights_struct(d: dict | None) -> Weights | None:
    if d is None:
        return None
    return Weights(*[_ptr(d.get(k)) for k in ("w13", "w13_sf", "w13_gs", "w2", "w2_sf", "w2_gs")])


class Plan:
    """A configured layer on the current CUDA device (moe_plan)."""

    def __init__(self, cfg: LayerConfig):
        self.cfg = cfg
        self._c = cfg.to_c()
        h = ctypes.c_void_p()
        _check("moe_plan", lib().moe_plan(ctypes.byref(self._c), ctypes.byref(h)))
        self._h = h

    def __del__(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.moe_plan_destroy(self._h)
            self._h = None

    def block_m(self, num_tokens: int) -> int:
        v = ctypes.c_int32()
        _check("moe_plan_block_m", lib().moe_plan_block_m(self._h, num_tokens, ctypes.byref(v)))
        return v.value

    def workspace_size(self, num_tokens: int) -> int:
        n = ctypes.c_size_t()
        _check("moe_workspace_size", lib().moe_workspace_size(self._h, num_tokens, ctypes.byref(n)))
        return n.value

    def weight_layout_size(self, which: int) -> int:
        n = ctypes.c_size_t()
        _check("moe_weight_layout_size", lib().moe_weight_layout_size(self._h, which, ctypes.byref(n)))
        return n.value

    def region(self, workspace: torch.Tensor, num_tokens: int, name: str) -> torch.Tensor:
        """A uint8 view of one workspace region (intermediate results of moe_forward)."""
        off, n = ctypes.c_size_t(), ctypes.c_size_t()
        _check("moe_workspace_region",
               lib().moe_workspace_region(self._h, num_tokens, REGIONS[name], ctypes.byref(off), ctypes.byref(n)))
        return workspace[off.value: off.value + n.value]

    def alloc_workspace(self, num_tokens: int, device=None) -> torch.Tensor:
        return torch.zeros(max(self.workspace_size(num_tokens), 1), dtype=torch.uint8,
                           device=device or torch.cuda.current_device())

    def _alloc_layout(self, ids: dict, device) -> dict:
        out = {}
        for key, which in ids.items():
            n = self.weight_layout_size(which)
            if n:
                dt = torch.float32 if key.endswith("_gs") else torch.uint8
                out[key] = torch.empty(n // (4 if dt == torch.float32 else 1), dtype=dt, device=device)
        return out

    def transform_weights(self, ckpt: dict, stream=None) -> dict:
        """Checkpoint-layout routed weights (device tensors) -> kernel-layout tensors."""
        dev = ckpt["w13"].device
        dst = self._alloc_layout({"w13": W13, "w13_sf": W13_SF, "w2": W2, "w2_sf": W2_SF,
                                  "w13_gs": W13_GS, "w2_gs": W2_GS}, dev)
        s, d = _weights_struct(ckpt), _weights_struct(dst)
        _check("moe_transform_weights",
               lib().moe_transform_weights(self._h, ctypes.byref(s), ctypes.byref(d), _stream(stream)))
        return dst

    def transform_shared_weights(self, ckpt: dict, stream=None) -> dict:
        dev = ckpt["w13"].device
        dst = self._alloc_layout({"w13": SHARED_W13, "w13_sf": SHARED_W13_SF, "w2": SHARED_W2,
                                  "w2_sf": SHARED_W2_SF}, dev)
        s, d = _weights_struct(ckpt), _weights_struct(dst)
        _check("moe_transform_shared_weights",
               lib().moe_transform_shared_weights(self._h, ctypes.byref(s), ctypes.byref(d), _stream(stream)))
        return dst

    def forward(self, hidden: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor, weights: dict,
                l2_act_scale: torch.Tensor | None = None, shared: dict | None = None,
                norm_gamma: torch.Tensor | None = None, out: torch.Tensor | None = None,
                workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """moe_forward: hidden bf16 [T, H] -> out bf16 [T, H].

        hidden, topk_ids, topk_weights, norm_gamma and out may be pinned CPU tensors
        (the kernels then read and write them in host memory directly); weights and
        the workspace are device tensors."""
        T = hidden.shape[0]
        dev = hidden.device if hidden.is_cuda else torch.device("cuda", torch.cuda.current_device())
        if out is None:
            out = torch.empty_like(hidden)
        if workspace is None:
            workspace = self.alloc_workspace(T, dev)
        w = _weights_struct(weights)
        sh = _weights_struct(shared)
        _check("moe_forward", lib().moe_forward(
            self._h, T, _ptr(hidden, True), _ptr(topk_ids, True), _ptr(topk_weights, True), ctypes.byref(w),
            _ptr(l2_act_scale), ctypes.byref(sh) if sh is not None else None, _ptr(norm_gamma, True),
            _ptr(out, True), _ptr(workspace), workspace.numel(), _stream(stream)))
        return out

    def batched_workspace_size(self, max_tokens: int) -> int:
        n = ctypes.c_size_t()
        _check("moe_batched_workspace_size", lib().moe_batched_workspace_size(self._h, max_tokens, ctypes.byref(n)))
        return n.value

    def forward_batched(self, hidden: torch.Tensor, expert_num_tokens: torch.Tensor, weights: dict,
                        l2_act_scale: torch.Tensor | None = None, out: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """moe_forward_batched: hidden bf16 [E, M, H] with expert_num_tokens int32 [E] -> out bf16
        [E, M, H] (rows m >= expert_num_tokens[e] are not written)."""
        E, M, _ = hidden.shape
        if out is None:
            out = torch.zeros_like(hidden)
        if workspace is None:
            workspace = torch.zeros(self.batched_workspace_size(M), dtype=torch.uint8, device=hidden.device)
        w = _weights_struct(weights)
        _check("moe_forward_batched", lib().moe_forward_batched(
            self._h, M, _ptr(hidden), _ptr(expert_num_tokens), ctypes.byref(w), _ptr(l2_act_scale), _ptr(out),
            _ptr(workspace), workspace.numel(), _stream(stream)))
        return out

    def set_wait_timeout(self, ns: int):
        """Limit of each bounded wait in the GEMM kernels (0: the default, 2 s)."""
        _check("moe_plan_set_wait_timeout", lib().moe_plan_set_wait_timeout(self._h, ns))

    def enable_timing(self, enable: bool = True):
        _check("moe_plan_enable_timing", lib().moe_plan_enable_timing(self._h, 1 if enable else 0))

    def kernel_times(self) -> dict:
        """Milliseconds of each kernel launch of the last forward (waits for it)."""
        arr = (ctypes.c_float * len(KERNELS))()
        _check("moe_plan_kernel_times", lib().moe_plan_kernel_times(self._h, arr, len(KERNELS)))
        return dict(zip(KERNELS, list(arr)))

    def last_status(self, workspace: torch.Tensor, stream=None) -> int:
        v = ctypes.c_int32()
        _check("moe_last_status", lib().moe_last_status(self._h, _ptr(workspace), _stream(stream), ctypes.byref(v)))
        return v.value
