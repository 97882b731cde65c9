"""GB300-native dropless token-choice MoE layer (forward and backward).

The compute lives in the CUDA library libmoe_gb300.so (C ABI in include/moe.h);
`binding` exposes its entry points and `layer.MoELayer` manages buffers.
Importing `binding` or `layer` requires the built library; there is no CPU path.
"""
__all__ = ["binding", "layer", "inputs", "build"]
