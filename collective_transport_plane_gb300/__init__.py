"""GB300-native FIFO data plane of a collective transport (SIMPLE, LL, zero
copy, host-placed FIFO, virtual ring allreduce) behind the C ABI in
include/xp.h.  `xp` is the ctypes binding; `build` compiles libxp.so."""
from . import xp  # noqa: F401  (raises ImportError if libxp.so is not built)
from .xp import *  # noqa: F401,F403
