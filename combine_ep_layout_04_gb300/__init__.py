"""GB300-native token layout, dispatch and combine of one MoE expert-parallel
(EP) layer whose R ranks are partitions of one GPU's HBM.

The product is the C-ABI library libep.so (include/ep.h), built from the
sm_103a CUDA sources in csrc/ by build.py.  This package holds that build
script, a ctypes binding with the ABI's names (_ep) and a torch-facing wrapper
(EpLayer) that allocates caller-owned outputs and passes device pointers and
streams.  Using EpLayer or _ep without a built libep.so raises ImportError:
there is no fallback path.  (The exports load lazily so that build.py can be
imported before the library exists.)
"""

__all__ = ["EpLayer", "Layout", "ExpertLayout", "SmSplit", "EpError", "CMD_DTYPE"]


def __getattr__(name):
    if name in ("EpLayer", "Layout", "ExpertLayout", "SmSplit", "CMD_DTYPE"):
        from . import layer
        return getattr(layer, name)
    if name == "EpError":
        from . import _ep
        return _ep.EpError
    raise AttributeError(name)
