"""CompKV decode step on one GB300: a C-ABI CUDA library (libcompkv.so) and its binding.

The decode step of CompKV (onedev.kr/papers/157) -- block summaries, block
scoring, forced + Top-K selection, exact attention on the selected blocks and
joint Mean compensation of the others -- runs entirely in hand-written sm_103a
kernels behind include/compkv.h.  This package only builds and loads that
library and marshals arguments to it.
"""
from ._build import build, LIB as library_file  # noqa: F401
from .compkv import *  # noqa: F401,F403
from .compkv import CompKVError, lib  # noqa: F401


def __getattr__(name):
    if name == "CompKVCache":
        from .cache import CompKVCache
        return CompKVCache
    raise AttributeError(name)
