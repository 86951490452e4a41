"""ctypes binding of libxp.so (include/xp.h): same names, argument marshalling only.

Every call goes straight to the C ABI; nothing here computes any part of the
transport.  Pointers may be given as integers or as objects with a
`data_ptr()` method (torch tensors); streams as integers, objects with a
`cuda_stream` attribute (torch.cuda.Stream) or None (the legacy default
stream).  A non-OK status raises `XpError` (the status queries return it).
If libxp.so is missing the import fails: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libxp.so")

XP_OK, XP_ERR_INVALID, XP_ERR_CUDA, XP_ERR_TIMEOUT, XP_ERR_BOUNDS, XP_ERR_ABORTED, XP_ERR_INTERNAL = range(7)
XP_PROTO_SIMPLE, XP_PROTO_LL, XP_PROTO_LL128 = 0, 1, 2
XP_PLACE_DEVICE, XP_PLACE_HOST_MAPPED = 0, 1
XP_U8, XP_U32, XP_I32, XP_F32, XP_BF16 = range(5)
XP_DISCARD_AUTO_BYTES = 48 << 20   # include/xp.h: FIFOs at least this large drop read slot lines by default
(XP_WAIT_NONE, XP_WAIT_HEAD, XP_WAIT_TAIL, XP_WAIT_PTR_EXCHANGE, XP_WAIT_LL_FLAG, XP_WAIT_SLOT_BARRIER,
 XP_WAIT_SIZE_WORD, XP_WAIT_OCCUPANCY, XP_WAIT_STICKY, XP_WAIT_POST, XP_WAIT_COMPLETION) = range(11)

# every entry point include/xp.h declares
EXPORTS = [
    "xp_fifo_create", "xp_fifo_destroy", "xp_fifo_set_lanes", "xp_fifo_describe", "xp_send_recv",
    "xp_send_recv_zero_copy", "xp_fifo_status", "xp_fifo_reset", "xp_ll_pingpong", "xp_ring_create",
    "xp_ring_destroy", "xp_ring_set_lanes", "xp_ring_allreduce_virtual", "xp_ring_status", "xp_ring_reset",
    "xp_set_spin_timeout_ns", "xp_abort", "xp_status_string", "xp_last_error", "xp_version",
    "xp_send_recv_noalloc", "xp_fifo_set_recv_lanes", "xp_send_recv_posted", "xp_fifo_enable_ce",
    "xp_send_recv_ce", "xp_send_recv_staged", "xp_fifo_stats", "xp_fifo_set_discard",
]


class xp_report(ctypes.Structure):
    _fields_ = [("code", ctypes.c_int32), ("channel", ctypes.c_int32), ("where", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("observed", ctypes.c_uint64), ("expected", ctypes.c_uint64),
                ("max_occupancy", ctypes.c_uint32), ("reserved2", ctypes.c_uint32)]


class xp_channel_desc(ctypes.Structure):
    _fields_ = [("ctl", ctypes.c_void_p), ("slots", ctypes.c_void_p), ("slot_stride", ctypes.c_size_t),
                ("nslots", ctypes.c_int), ("proto", ctypes.c_int), ("placement", ctypes.c_int),
                ("lanes", ctypes.c_int), ("recv_lanes", ctypes.c_int), ("posted", ctypes.c_void_p),
                ("ce", ctypes.c_void_p), ("send_ring", ctypes.c_void_p), ("recv_ring", ctypes.c_void_p),
                ("discard", ctypes.c_int)]


class xp_channel_stats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_uint64), ("t_start_ns", ctypes.c_uint64), ("t_end_ns", ctypes.c_uint64),
                ("send_polls", ctypes.c_uint64), ("recv_polls", ctypes.c_uint64)]


class XpError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: status {status} ({message})")
        self.status = status


def load(path: str = _LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"{path} is not built: run collective_transport_plane_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I, Z, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint64
    sig = {
        "xp_fifo_create": [I, I, Z, I, I, ctypes.POINTER(P)],
        "xp_fifo_destroy": [P],
        "xp_fifo_set_lanes": [P, I],
        "xp_fifo_set_recv_lanes": [P, I],
        "xp_fifo_describe": [P, I, ctypes.POINTER(xp_channel_desc)],
        "xp_send_recv": [P, P, P, Z, P],
        "xp_send_recv_zero_copy": [P, P, P, Z, P],
        "xp_send_recv_posted": [P, P, P, Z, I, P],
        "xp_fifo_enable_ce": [P],
        "xp_send_recv_ce": [P, P, P, Z, P],
        "xp_send_recv_staged": [P, P, P, P, P, Z, Z, P],
        "xp_fifo_stats": [P, I, ctypes.POINTER(xp_channel_stats)],
        "xp_fifo_set_discard": [P, I],
        "xp_fifo_status": [P, I, ctypes.POINTER(xp_report)],
        "xp_fifo_reset": [P],
        "xp_ll_pingpong": [P, P, I, ctypes.POINTER(U64), P],
        "xp_ring_create": [I, I, I, Z, I, ctypes.POINTER(P)],
        "xp_ring_destroy": [P],
        "xp_ring_set_lanes": [P, I],
        "xp_ring_allreduce_virtual": [P, ctypes.POINTER(P), ctypes.POINTER(P), Z, I, P],
        "xp_ring_status": [P, I, ctypes.POINTER(xp_report)],
        "xp_ring_reset": [P],
        "xp_set_spin_timeout_ns": [U64],
        "xp_abort": [I],
        "xp_status_string": [I],
        "xp_last_error": [],
        "xp_version": [],
        "xp_send_recv_noalloc": [P, P, Z, I, I, Z, P, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.xp_status_string.restype = ctypes.c_char_p
    lib.xp_last_error.restype = ctypes.c_char_p
    return lib


_lib = load()


def _ptr(x) -> int | None:
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return int(x)


def _stream(s) -> int | None:
    if s is None:
        return None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    return int(s)


def _check(st: int, where: str):
    if st != XP_OK:
        raise XpError(st, where, _lib.xp_last_error().decode() or xp_status_string(st))


def xp_version() -> int:
    return _lib.xp_version()


def xp_status_string(st: int) -> str:
    return _lib.xp_status_string(st).decode()


def xp_last_error() -> str:
    return _lib.xp_last_error().decode()


def xp_fifo_create(nchannels: int, nslots: int, slot_bytes: int, proto: int = XP_PROTO_SIMPLE,
                   place: int = XP_PLACE_DEVICE) -> int:
    out = ctypes.c_void_p()
    _check(_lib.xp_fifo_create(nchannels, nslots, slot_bytes, proto, place, ctypes.byref(out)), "xp_fifo_create")
    return out.value


def xp_fifo_destroy(fifo: int) -> None:
    _check(_lib.xp_fifo_destroy(fifo), "xp_fifo_destroy")


def xp_fifo_set_lanes(fifo: int, lanes: int) -> None:
    _check(_lib.xp_fifo_set_lanes(fifo, lanes), "xp_fifo_set_lanes")


def xp_fifo_set_recv_lanes(fifo: int, rlanes: int) -> None:
    _check(_lib.xp_fifo_set_recv_lanes(fifo, rlanes), "xp_fifo_set_recv_lanes")


def xp_fifo_describe(fifo: int, channel: int) -> xp_channel_desc:
    d = xp_channel_desc()
    _check(_lib.xp_fifo_describe(fifo, channel, ctypes.byref(d)), "xp_fifo_describe")
    return d


def xp_send_recv(fifo: int, src, dst, nbytes: int, stream=None) -> None:
    _check(_lib.xp_send_recv(fifo, _ptr(src), _ptr(dst), nbytes, _stream(stream)), "xp_send_recv")


def xp_send_recv_zero_copy(fifo: int, src, dst, nbytes: int, stream=None) -> None:
    _check(_lib.xp_send_recv_zero_copy(fifo, _ptr(src), _ptr(dst), nbytes, _stream(stream)),
           "xp_send_recv_zero_copy")


def xp_fifo_stats(fifo: int, channel: int) -> xp_channel_stats:
    out = xp_channel_stats()
    _check(_lib.xp_fifo_stats(fifo, channel, ctypes.byref(out)), "xp_fifo_stats")
    return out


def xp_fifo_set_discard(fifo: int, on: bool | None) -> None:
    """True: drop read slot lines; False: keep them; None: choose by the FIFO's size."""
    _check(_lib.xp_fifo_set_discard(fifo, -1 if on is None else (1 if on else 0)), "xp_fifo_set_discard")


def xp_fifo_enable_ce(fifo: int) -> None:
    _check(_lib.xp_fifo_enable_ce(fifo), "xp_fifo_enable_ce")


def xp_send_recv_ce(fifo: int, src, dst, nbytes: int, stream=None) -> None:
    _check(_lib.xp_send_recv_ce(fifo, _ptr(src), _ptr(dst), nbytes, _stream(stream)), "xp_send_recv_ce")


def xp_send_recv_staged(fifo: int, host_src, host_dst, dev_src, dev_dst, nbytes: int, chunk_bytes: int = 0,
                        stream=None) -> None:
    _check(_lib.xp_send_recv_staged(fifo, _ptr(host_src), _ptr(host_dst), _ptr(dev_src), _ptr(dev_dst), nbytes,
                                    chunk_bytes, _stream(stream)), "xp_send_recv_staged")


def xp_send_recv_posted(fifo: int, src, dst, nbytes: int, direct: bool = False, stream=None) -> None:
    _check(_lib.xp_send_recv_posted(fifo, _ptr(src), _ptr(dst), nbytes, 1 if direct else 0, _stream(stream)),
           "xp_send_recv_posted")


def xp_fifo_status(fifo: int, sync: bool = True) -> tuple[int, xp_report]:
    rep = xp_report()
    st = _lib.xp_fifo_status(fifo, 1 if sync else 0, ctypes.byref(rep))
    return st, rep


def xp_fifo_reset(fifo: int) -> None:
    _check(_lib.xp_fifo_reset(fifo), "xp_fifo_reset")


def xp_ll_pingpong(ab: int, ba: int, iters: int, stream=None) -> int:
    ns = ctypes.c_uint64()
    _check(_lib.xp_ll_pingpong(ab, ba, iters, ctypes.byref(ns), _stream(stream)), "xp_ll_pingpong")
    return ns.value


def xp_ring_create(nranks: int, nchannels: int, nslots: int, slot_bytes: int,
                   place: int = XP_PLACE_DEVICE) -> int:
    out = ctypes.c_void_p()
    _check(_lib.xp_ring_create(nranks, nchannels, nslots, slot_bytes, place, ctypes.byref(out)), "xp_ring_create")
    return out.value


def xp_ring_destroy(ring: int) -> None:
    _check(_lib.xp_ring_destroy(ring), "xp_ring_destroy")


def xp_ring_set_lanes(ring: int, lanes: int) -> None:
    _check(_lib.xp_ring_set_lanes(ring, lanes), "xp_ring_set_lanes")


def xp_ring_allreduce_virtual(ring: int, send_bufs, recv_bufs, count: int, dtype: int, stream=None) -> None:
    n = len(send_bufs)
    sb = (ctypes.c_void_p * n)(*[_ptr(b) for b in send_bufs])
    rb = (ctypes.c_void_p * len(recv_bufs))(*[_ptr(b) for b in recv_bufs])
    _check(_lib.xp_ring_allreduce_virtual(ring, sb, rb, count, dtype, _stream(stream)), "xp_ring_allreduce_virtual")


def xp_ring_status(ring: int, sync: bool = True) -> tuple[int, xp_report]:
    rep = xp_report()
    st = _lib.xp_ring_status(ring, 1 if sync else 0, ctypes.byref(rep))
    return st, rep


def xp_ring_reset(ring: int) -> None:
    _check(_lib.xp_ring_reset(ring), "xp_ring_reset")


def xp_set_spin_timeout_ns(ns: int) -> None:
    _check(_lib.xp_set_spin_timeout_ns(ns), "xp_set_spin_timeout_ns")


def xp_abort(value: int) -> None:
    _check(_lib.xp_abort(value), "xp_abort")


def xp_send_recv_noalloc(src, dst, nbytes: int, nchannels: int, nslots: int, slot_bytes: int,
                         dev_status=None, stream=None) -> None:
    """SIMPLE transfer through the library's static FIFO: allocates nothing."""
    _check(_lib.xp_send_recv_noalloc(_ptr(src), _ptr(dst), nbytes, nchannels, nslots, slot_bytes, _ptr(dev_status),
                                     _stream(stream)), "xp_send_recv_noalloc")


def library_path() -> str:
    return _LIB_PATH
