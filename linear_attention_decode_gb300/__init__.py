"""ReplaySSM GDN / KDA decode for one GB300 (sm_103a).

The compute path is libgdnreplay.so (hand-written CUDA behind a C ABI declared
in include/gdnreplay.h); ``binding`` is its ctypes binding, ``inputs`` the
seeded synthetic workloads, ``build`` the in-tree nvcc build.
"""
from .constants import *  # noqa: F401,F403
