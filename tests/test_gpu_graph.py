"""CUDA-graph replay: the step counters live on the device, so a captured
operation replayed with new inputs gives the oracle's result every time."""
import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_util import from_dev, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = torch_cuda()
    from collective_transport_plane_gb300 import build
    build.build()
    import collective_transport_plane_gb300.xp as xp
    xp.xp_set_spin_timeout_ns(2_000_000_000)
    return torch, xp


def _capture(torch, fn):
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fn(s)                                   # first call outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fn(s)
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("mode", ["simple", "zero_copy", "posted_copy", "posted_direct", "ce", "ll", "ll128"])
def test_p2p_graph_replay(env, mode):
    torch, xp = env
    nchan, nslots, slot = 4, 4, 8192
    n = 300008 if mode in ("ll", "ll128") else 300007
    proto = {"ll": xp.XP_PROTO_LL, "ll128": xp.XP_PROTO_LL128}.get(mode, xp.XP_PROTO_SIMPLE)
    fifo = xp.xp_fifo_create(nchan, nslots, slot, proto)
    if mode != "ll":
        xp.xp_fifo_set_lanes(fifo, 2)
    if mode == "ce":
        xp.xp_fifo_enable_ce(fifo)       # the pump keeps serving replays
    src = torch.zeros(n, dtype=torch.uint8, device="cuda")
    dst = torch.zeros_like(src)

    def op(s):
        if mode in ("simple", "ll", "ll128"):
            xp.xp_send_recv(fifo, src, dst, n, s)
        elif mode == "zero_copy":
            xp.xp_send_recv_zero_copy(fifo, src, dst, n, s)
        elif mode == "ce":
            xp.xp_send_recv_ce(fifo, src, dst, n, s)
        else:
            xp.xp_send_recv_posted(fifo, src, dst, n, mode == "posted_direct", s)

    g = _capture(torch, op)
    for i in range(3):
        src_np = workloads.uniform_bytes(n, seed=80 + i)
        if mode == "simple":
            want = oracle.simple_transfer(src_np, nchan, nslots, slot, seed=i)[0]
        elif mode == "ll":
            want = oracle.ll_transfer(src_np.view(np.uint32), nchan, nslots, slot, seed=i)[0].view(np.uint8)
        elif mode == "ll128":
            want = oracle.ll128_transfer(src_np, nchan, nslots, slot, seed=i)[0].view(np.uint8)
        elif mode == "zero_copy":
            want = oracle.zero_copy_transfer(src_np, nchan, nslots, slot, seed=i)[0]
        elif mode == "ce":
            want = oracle.ce_transfer(src_np, nchan, nslots, slot, seed=i)[0]
        else:
            want = oracle.posted_transfer(src_np, nchan, nslots, slot, seed=i, direct=mode == "posted_direct")[0]
        src.copy_(torch.from_numpy(src_np))
        dst.zero_()
        g.replay()
        torch.cuda.synchronize()
        st, rep = xp.xp_fifo_status(fifo, True)
        assert st == xp.XP_OK, (st, rep.where, rep.observed, rep.expected)
        assert rep.channel == -1
        if mode in ("simple", "zero_copy", "ce", "posted_direct"):
            # the replay's own occupancy: status words carry the captured
            # operation's id, which the replay also writes as it starts
            assert 1 <= rep.max_occupancy <= nslots
        assert np.array_equal(from_dev(dst), want)
    xp.xp_fifo_destroy(fifo)


def test_ring_graph_replay(env):
    torch, xp = env
    P, n, nchan, nslots, slot = 4, 100003, 3, 4, 4096
    ring = xp.xp_ring_create(P, nchan, nslots, slot)
    ins = [torch.zeros(n, dtype=torch.float32, device="cuda") for _ in range(P)]
    outs = [torch.zeros_like(t) for t in ins]
    g = _capture(torch, lambda s: xp.xp_ring_allreduce_virtual(ring, ins, outs, n, xp.XP_F32, s))
    for i in range(3):
        xs = workloads.ring_inputs(P, n, "f32", 30 + i)
        want = oracle.ring_order_sum(xs, nchan, nslots, slot)
        for t, x in zip(ins, xs):
            t.copy_(torch.from_numpy(x))
        g.replay()
        torch.cuda.synchronize()
        st, rep = xp.xp_ring_status(ring, True)
        assert st == xp.XP_OK and 1 <= rep.max_occupancy <= nslots
        for t in outs:
            assert np.array_equal(from_dev(t), want)
    xp.xp_ring_destroy(ring)
