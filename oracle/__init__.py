"""CPU oracle for the routed-expert MoE layer forward.

TEST INFRASTRUCTURE ONLY. This package is a plain, slow, obviously-correct
NumPy restatement of what the layer computes, written from the vLLM MegaMoE
documentation pages (vllm.model_executor.layers.fused_moe.deep_gemm_mega_moe;
vllm.model_executor.layers.fused_moe, DeepGemmExperts; vllm.models.
qwen4_exp.nvidia.mega_moe; vllm.models.muse_spark.nvidia.mega_moe). It shares
no code with the CUDA path and imports nothing from it; only ``tests/``, the
smoke check and the benchmark's CPU-baseline leg may import it.

Modules:
  formats  decode tables (E2M1, E4M3, UE8M0), RNE-saturating encoders, the
           MXFP8 and NVFP4 quantisers, bf16 rounding
  routing  per-expert histogram, BLOCK_M-padded offsets, stable permutation
  moe      dispatch quantisation, SwiGLU, per-expert MLP, L2-input requant,
           top-k-weighted combine, shared expert, post-norm, bf16 output

Parity status: every function is pinned by tests against closed forms,
brute force or hand-worked values, except the NVFP4 scale arithmetic
(``formats.nvfp4_quantize``): the pages give its structure but not its
steps, so its exact recipe is a reading; it is pinned only by properties
(round trips, error bounds, hand-worked blocks) -- parity unpinned by the
pages for the NVFP4 recipe itself.
"""
from . import formats, routing, moe  # noqa: F401
