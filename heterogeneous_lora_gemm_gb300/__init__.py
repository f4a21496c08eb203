"""GB300-native multi-LoRA linear layer (sm_103a).

The compute lives in ``libmlora.so`` (CUDA kernels behind the C ABI of
``include/mlora.h``); ``mlora`` is its ctypes binding.
"""
from . import mlora  # noqa: F401
from .mlora import Pool, MloraError  # noqa: F401
