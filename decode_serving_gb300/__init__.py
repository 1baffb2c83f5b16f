"""GB300-native sparse-KV reuse decode step (C library libavsg + thin binding).

``avsg`` is the ctypes binding of include/avsg.h (same function names);
``session`` holds pinned host memory and one handle; ``build`` compiles the
CUDA sources for sm_103a in-tree.
"""
from . import avsg  # noqa: F401
from .avsg import AvsgError, load_library  # noqa: F401
