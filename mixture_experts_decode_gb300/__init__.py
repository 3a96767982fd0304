"""GB300-native small-batch MoE expert-FFN decode layer (MXFP8 weights).

The compute path is the C-ABI library libmoedec.so (hand-written sm_103a
CUDA, see include/moedec.h); the functions below only marshal arguments into
it.  Importing the package is cheap; the first call loads the library and
raises if it has not been built -- there is no CPU fallback.
"""
from ._lib import (MX, MoEError, align_block_size, align_block_size_static, align_sizes, copy, device_error, down, gate_up,
                   layer, layer_grouped, layer_grouped_workspace_bytes, layer_host, layer_host_workspace_bytes,
                   layer_workspace_bytes, load,
                   mx_requant, router_topk, version)

__all__ = ["MX", "MoEError", "align_block_size", "align_block_size_static", "align_sizes", "copy", "device_error", "down",
           "gate_up", "layer", "layer_grouped", "layer_grouped_workspace_bytes", "layer_host", "layer_host_workspace_bytes", "layer_workspace_bytes",
           "load", "mx_requant", "router_topk", "version"]
