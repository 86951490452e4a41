"""Failure detection without a GPU fault: every device wait is bounded, so a
wait on a counter that nothing will ever advance ends with a status the host
reads; the host abort word stops waits early; an object that saw an error
refuses work until it is reset."""
import numpy as np
import pytest

import workloads
from tests.gpu_util import from_dev, raw_view, to_dev, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = torch_cuda()
    from collective_transport_plane_gb300 import build
    build.build()
    import collective_transport_plane_gb300.xp as xp
    yield torch, xp
    xp.xp_abort(0)
    xp.xp_set_spin_timeout_ns(2_000_000_000)


def _stall(torch, xp, fifo):
    # move the channel's step base far ahead of its head: the sender's first
    # step needs credit that no receiver will ever return, and the receiver
    # waits for a tail that no sender will publish
    d = xp.xp_fifo_describe(fifo, 0)
    raw_view(torch, d.ctl, 128, "<u8")[48] = 1000
    torch.cuda.synchronize()


def test_wait_times_out_and_reports(env):
    torch, xp = env
    xp.xp_set_spin_timeout_ns(50_000_000)
    fifo = xp.xp_fifo_create(1, 2, 1024)
    _stall(torch, xp, fifo)
    src = torch.ones(8192, dtype=torch.uint8, device="cuda")
    dst = torch.zeros_like(src)
    xp.xp_send_recv(fifo, src, dst, 8192)
    st, rep = xp.xp_fifo_status(fifo, True)
    assert st == xp.XP_ERR_TIMEOUT
    assert rep.where in (xp.XP_WAIT_HEAD, xp.XP_WAIT_TAIL, xp.XP_WAIT_SLOT_BARRIER)
    assert rep.channel == 0
    # sticky: the next operations are refused on the device, each claiming
    # the status block for itself (the timeout's counters are not repeated)
    for _ in range(2):
        xp.xp_send_recv(fifo, src, dst, 8192)
        st, rep = xp.xp_fifo_status(fifo, True)
        assert st == xp.XP_ERR_ABORTED and rep.where == xp.XP_WAIT_STICKY
        assert rep.observed == 0 and rep.expected == 0 and rep.channel == 0
    # reset restores it; a good operation reports no failure and its own
    # occupancy
    xp.xp_fifo_reset(fifo)
    xp.xp_set_spin_timeout_ns(2_000_000_000)
    for _ in range(2):
        xp.xp_send_recv(fifo, src, dst, 8192)
        st, rep = xp.xp_fifo_status(fifo, True)
        assert st == xp.XP_OK and bool((dst == 1).all())
        assert rep.channel == -1 and 1 <= rep.max_occupancy <= 2
    xp.xp_fifo_destroy(fifo)


def test_abort_word_stops_waits(env):
    torch, xp = env
    xp.xp_set_spin_timeout_ns(20_000_000_000)
    fifo = xp.xp_fifo_create(1, 2, 1024)
    _stall(torch, xp, fifo)
    xp.xp_abort(1)
    src = torch.ones(4096, dtype=torch.uint8, device="cuda")
    dst = torch.zeros_like(src)
    xp.xp_send_recv(fifo, src, dst, 4096)
    st, _ = xp.xp_fifo_status(fifo, True)
    xp.xp_abort(0)
    xp.xp_set_spin_timeout_ns(2_000_000_000)
    assert st == xp.XP_ERR_ABORTED
    xp.xp_fifo_destroy(fifo)


def test_ll_flag_wait_times_out(env):
    # an LL receiver whose flags never arrive: the sender is held back by
    # a head that never advances
    torch, xp = env
    xp.xp_set_spin_timeout_ns(50_000_000)
    fifo = xp.xp_fifo_create(1, 1, 64, xp.XP_PROTO_LL)
    _stall(torch, xp, fifo)
    words = to_dev(torch, workloads.uniform_u32(64, seed=1))
    out = torch.zeros_like(words)
    xp.xp_send_recv(fifo, words, out, 256)
    st, rep = xp.xp_fifo_status(fifo, True)
    assert st == xp.XP_ERR_TIMEOUT
    xp.xp_fifo_reset(fifo)
    xp.xp_set_spin_timeout_ns(2_000_000_000)
    xp.xp_send_recv(fifo, words, out, 256)
    st, _ = xp.xp_fifo_status(fifo, True)
    assert st == xp.XP_OK and np.array_equal(from_dev(out), from_dev(words))
    xp.xp_fifo_destroy(fifo)


def test_spin_timeout_from_environment(env):
    # XP_SPIN_TIMEOUT_NS sets the starting timeout of a fresh process: a
    # stalled wait gives up after ~50 ms instead of the default 2 s
    import os
    import subprocess
    import sys
    code = (
        "import time, torch\n"
        "import collective_transport_plane_gb300.xp as xp\n"
        "from tests.gpu_util import raw_view\n"
        "f = xp.xp_fifo_create(1, 2, 1024)\n"
        "raw_view(torch, xp.xp_fifo_describe(f, 0).ctl, 128, '<u8')[48] = 1000\n"
        "torch.cuda.synchronize()\n"
        "a = torch.ones(4096, dtype=torch.uint8, device='cuda'); b = torch.zeros_like(a)\n"
        "t = time.time(); xp.xp_send_recv(f, a, b, 4096); st, _ = xp.xp_fifo_status(f, True)\n"
        "print(st, time.time() - t)\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True, timeout=120,
                         env=dict(os.environ, XP_SPIN_TIMEOUT_NS="50000000"))
    st, secs = out.stdout.split()
    assert int(st) == 3 and float(secs) < 1.0, out.stdout + out.stderr


def test_zero_copy_wait_times_out_and_recovers(env):
    # zero copy with the channel's step base moved past head: the receiver
    # posts dst and waits for a tail that never comes, the sender waits for
    # credit; both give up, the FIFO refuses work until reset, then works
    torch, xp = env
    xp.xp_set_spin_timeout_ns(50_000_000)
    fifo = xp.xp_fifo_create(1, 2, 1024)
    xp.xp_fifo_set_lanes(fifo, 2)
    _stall(torch, xp, fifo)
    src = to_dev(torch, workloads.uniform_bytes(8192, seed=5))
    dst = torch.zeros_like(src)
    xp.xp_send_recv_zero_copy(fifo, src, dst, 8192)
    st, rep = xp.xp_fifo_status(fifo, True)
    assert st == xp.XP_ERR_TIMEOUT
    assert rep.where in (xp.XP_WAIT_HEAD, xp.XP_WAIT_TAIL, xp.XP_WAIT_SLOT_BARRIER)
    assert bool((dst == 0).all())   # no credit, so nothing was written
    xp.xp_send_recv_zero_copy(fifo, src, dst, 8192)
    st, rep = xp.xp_fifo_status(fifo, True)
    assert st == xp.XP_ERR_ABORTED and rep.where == xp.XP_WAIT_STICKY
    xp.xp_fifo_reset(fifo)
    xp.xp_set_spin_timeout_ns(2_000_000_000)
    xp.xp_send_recv_zero_copy(fifo, src, dst, 8192)
    st, _ = xp.xp_fifo_status(fifo, True)
    assert st == xp.XP_OK and np.array_equal(from_dev(dst), from_dev(src))
    xp.xp_fifo_destroy(fifo)


def test_create_and_destroy_return_device_memory(env):
    # every kind of object, with one operation each (lazily created streams
    # and events included), created and destroyed repeatedly: the device's
    # free memory comes back
    torch, xp = env
    src = to_dev(torch, workloads.uniform_bytes(1 << 20, seed=6))
    dst = torch.zeros_like(src)
    hsrc = torch.from_numpy(workloads.uniform_bytes(1 << 20, seed=7)).pin_memory()
    hdst = torch.zeros_like(hsrc).pin_memory()
    rin = [torch.ones(4096, dtype=torch.float32, device="cuda") for _ in range(4)]
    rout = [torch.zeros_like(t) for t in rin]

    def cycle():
        fifos = [xp.xp_fifo_create(16, 8, 512 << 10), xp.xp_fifo_create(2, 4, 32768, xp.XP_PROTO_LL),
                 xp.xp_fifo_create(2, 4, 32768, xp.XP_PROTO_LL128),
                 xp.xp_fifo_create(2, 2, 4096, xp.XP_PROTO_SIMPLE, xp.XP_PLACE_HOST_MAPPED)]
        for f in fifos:
            xp.xp_send_recv(f, src, dst, 1 << 20)
        xp.xp_send_recv_staged(fifos[0], hsrc, hdst, src, dst, 1 << 20, 1 << 18)
        ce = xp.xp_fifo_create(2, 4, 65536)
        xp.xp_fifo_enable_ce(ce)
        xp.xp_send_recv_ce(ce, src, dst, 1 << 20)
        fifos.append(ce)
        ring = xp.xp_ring_create(4, 2, 4, 65536)
        xp.xp_ring_allreduce_virtual(ring, rin, rout, 4096, xp.XP_F32)
        torch.cuda.synchronize()
        for i, f in enumerate(fifos):
            st, rep = xp.xp_fifo_status(f, True)
            assert st == xp.XP_OK, (i, st, rep.where, rep.channel, rep.observed, rep.expected, xp.xp_last_error())
            xp.xp_fifo_destroy(f)
        assert xp.xp_ring_status(ring, True)[0] == xp.XP_OK
        xp.xp_ring_destroy(ring)
        torch.cuda.synchronize()

    cycle()   # first use: module loading, kernel attributes
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        cycle()
    free1 = torch.cuda.mem_get_info()[0]
    assert free0 - free1 < (4 << 20), (free0, free1)
    assert bool((rout[0] == 4).all())
