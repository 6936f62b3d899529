"""GB300-native (sm_103a) Dory looped normalized-GPT token forward.

The compute lives in libdory.so (hand-written CUDA kernels behind the C ABI of
include/dory.h); this package holds its build script and a ctypes binding.
"""
from .dory import Dory, DoryError, load_library  # noqa: F401
from .build import build  # noqa: F401
