"""B300-native forward pass of a sparse Mixture-of-Experts layer.

The compute path is the C-ABI library ``libmoe_b300.so`` (hand-written CUDA
for sm_103a, declared in include/moe_b300.h); ``api`` is its PyTorch binding.
"""
from .api import (MoeError, MoELayer, capacity, combine, dispatch, expert_ffn, forward, get_device_error,
                  max_rows, new_workspace, route, shape_of, workspace_size)

__all__ = ["MoeError", "MoELayer", "capacity", "combine", "dispatch", "expert_ffn", "forward", "get_device_error",
           "max_rows", "new_workspace", "route", "shape_of", "workspace_size"]
