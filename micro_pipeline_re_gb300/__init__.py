"""GB300-native synchronous GPipe training step (one GPU, K cells, M micro-batches).

The compute path is libgpipe.so (CUDA kernels for sm_103a behind a C ABI,
include/gpipe.h); ``binding`` is its ctypes marshalling layer.
"""
from ._build import build  # noqa: F401
