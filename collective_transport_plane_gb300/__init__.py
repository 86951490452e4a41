"""GB300-native FIFO data plane of a collective transport (SIMPLE, LL, zero
copy, receiver-driven credit, host-placed FIFO, virtual ring allreduce)
behind the C ABI in include/xp.h.  `xp` is the ctypes binding; `build`
compiles libxp.so.

The binding is imported on first use, so `build` can run before libxp.so
exists; importing `xp` (or reading any of its names from this package)
raises ImportError while the library is not built."""
import importlib


def __getattr__(name):
    if name in ("xp", "build"):
        return importlib.import_module(f".{name}", __name__)
    xp = importlib.import_module(".xp", __name__)
    try:
        return getattr(xp, name)
    except AttributeError:
        raise AttributeError(f"module {__name__!r} has no attribute {name!r}") from None
