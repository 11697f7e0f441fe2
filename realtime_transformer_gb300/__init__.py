"""GB300 (sm_103a) FP8-quantised pre-norm FFN sublayer behind a C ABI.

The compute path lives in libfrt_ffn.so (hand-written CUDA: norm/quant,
tcgen05 FP8 GEMMs, act/requant, calibration, CUDA-graph plan).  This package
is the thin Python binding: `_native` mirrors the C functions one to one,
`ffn.FFNPlan` adds torch tensors for memory and streams.
"""
from ._native import FrtError, LIB_PATH  # noqa: F401


def __getattr__(name):
    if name == "FFNPlan":
        from .ffn import FFNPlan
        return FFNPlan
    if name == "QKVPlan":
        from .qkv import QKVPlan
        return QKVPlan
    if name == "FP4Plan":
        from .nvfp4 import FP4Plan
        return FP4Plan
    raise AttributeError(name)
