"""GB300-native token layout, dispatch and combine of one MoE expert-parallel
(EP) layer whose R ranks are partitions of one GPU's HBM.

The product is the C-ABI library libep.so (include/ep.h), built from the
sm_103a CUDA sources in csrc/.  This package holds its build script, a ctypes
binding with the ABI's names (_ep) and a torch-facing wrapper (EpLayer) that
allocates caller-owned outputs and passes device pointers and streams.
Importing it without a built libep.so raises: there is no fallback path.
"""
from . import _ep
from ._ep import EpError
from .layer import CMD_DTYPE, EpLayer, Layout

__all__ = ["EpLayer", "Layout", "EpError", "CMD_DTYPE", "_ep"]
