"""GB300-native epilogue fusion: conv2d + BatchNorm + SiLU, bias + GELU and
residual + LayerNorm + affine, each written to HBM once by hand-written
sm_103a CUDA kernels behind a C ABI (include/tf_epilogue.h).

``gemm_conv_epilogues_gb300.binding`` is the Python view of that ABI (loaded
on first use); ``synth`` holds the seeded synthetic inputs; ``build``
compiles the library in-tree.
"""
import importlib

__all__ = ["binding", "build", "synth"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
