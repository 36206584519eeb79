"""Chunk-bounded, top-k-softmax-routed MoE block on one GB300 (sm_103a).

The compute lives in libmoe.so (hand-written CUDA; C ABI in include/moe.h, include/moe_adamw.h
and include/moe_ce.h); this package is the build script and a thin ctypes binding.
"""
from .api import *  # noqa: F401,F403
from .adamw import *  # noqa: F401,F403
from .ce import *  # noqa: F401,F403
from .autograd import *  # noqa: F401,F403
