"""Helpers for the GPU tests: move numpy arrays to and from the device and
view raw device words (FIFO control blocks) as tensors."""
import numpy as np


def torch_cuda():
    import pytest
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def to_dev(torch, a: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def from_dev(t) -> np.ndarray:
    return t.cpu().numpy()


class _Iface:
    def __init__(self, ptr, n, typestr):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": None}


def raw_view(torch, ptr: int, n: int, typestr: str = "<u8"):
    """A tensor aliasing n elements at device-accessible address ptr."""
    return torch.as_tensor(_Iface(ptr, n, typestr), device="cuda")


def ctl_words(torch, xp, fifo, channel):
    """(tail, head, ptrExchange, base) of one channel, read from the device."""
    d = xp.xp_fifo_describe(fifo, channel)
    v = raw_view(torch, d.ctl, 128, "<u8").cpu().numpy()
    return int(v[0]), int(v[16]), int(v[32]), int(v[48])
