"""GB300-native (sm_103a) routed-expert MoE layer forward: a C-ABI library
(libmoe.so, include/moe.h) of hand-written CUDA kernels and this thin binding."""
from .moe import (FORMATS, LayerConfig, MoeError, Plan, config_workspace_size, error_string,  # noqa: F401
                  lib, library_path, permute_noalloc, validate)
