"""Proxy (copy-engine) mode on the GPU: sender CTAs fill the send ring, the
library's host pump copies each slot-step with cudaMemcpyAsync (one hop for a
device FIFO, two hops through the host-placed FIFO), receiver CTAs drain the
last ring.  Compared with the oracle on the same seeded inputs: the delivered
bytes, the bytes left in every ring, and the tail/head counters."""
import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_util import from_dev, raw_view, to_dev, torch_cuda

pytestmark = pytest.mark.gpu

TAIL0, HEAD, BASE = 0, 384 // 8, 512 // 8


@pytest.fixture(scope="module")
def env():
    torch = torch_cuda()
    from collective_transport_plane_gb300 import build
    build.build()
    import collective_transport_plane_gb300.xp as xp
    xp.xp_set_spin_timeout_ns(2_000_000_000)
    return torch, xp


def _fifo(xp, nchan, nslots, slot, place, lanes=1, rlanes=None, discard=False):
    # ring contents are checked against the oracle's: no discard unless asked
    f = xp.xp_fifo_create(nchan, nslots, slot, xp.XP_PROTO_SIMPLE, place)
    xp.xp_fifo_set_discard(f, discard)
    xp.xp_fifo_set_lanes(f, lanes)
    if rlanes is not None:
        xp.xp_fifo_set_recv_lanes(f, rlanes)
    xp.xp_fifo_enable_ce(f)
    return f


def _ce(torch, xp, fifo, src_np):
    src = to_dev(torch, src_np)
    dst = torch.zeros_like(src)
    xp.xp_send_recv_ce(fifo, src, dst, src_np.nbytes, torch.cuda.current_stream())
    st, rep = xp.xp_fifo_status(fifo, True)
    assert st == xp.XP_OK, (st, rep.channel, rep.where, rep.observed, rep.expected, xp.xp_last_error())
    return dst, rep


def _check_state(torch, xp, fifo, fifos, nslots, slot, hops, rings=True):
    for c, f in enumerate(fifos):
        d = xp.xp_fifo_describe(fifo, c)
        w = raw_view(torch, d.ce, 2048 // 8, "<u8").cpu().numpy()
        assert [int(w[TAIL0 + 16 * h]) for h in range(hops + 1)] == f.tails
        assert int(w[HEAD]) == f.head == int(w[BASE])
        if rings:
            views = [d.send_ring] + ([d.slots] if hops == 2 else []) + [d.recv_ring]
            for r, ptr in zip(f.rings, views):
                got = raw_view(torch, ptr, nslots * slot, "|u1").cpu().numpy()
                assert np.array_equal(got, r.slots.reshape(-1))


SWEEP = [(1, 1, 1, 16, 1, 1), (15, 2, 2, 16, 1, 1), (17, 3, 1, 16, 2, 1), (4095, 3, 2, 64, 1, 2),
         (65537, 4, 2, 4096, 2, 3), (1000003, 16, 8, 16384, 1, 1), (1000003, 5, 3, 65536, 4, 4),
         (3 << 20, 2, 8, 65536, 8, 8), (12345, 1, 1, 4096, 3, 2)]


@pytest.mark.parametrize("place", [0, 1], ids=["device-1hop", "host-2hops"])
@pytest.mark.parametrize("n,nchan,nslots,slot,lanes,rlanes", SWEEP)
def test_ce_sweep(env, n, nchan, nslots, slot, lanes, rlanes, place):
    torch, xp = env
    hops = 1 + place
    src_np = workloads.uniform_bytes(n, seed=n % 997 + 11)
    want, fifos, _ = oracle.ce_transfer(src_np, nchan, nslots, slot, hops=hops, seed=4)
    fifo = _fifo(xp, nchan, nslots, slot, place, lanes, rlanes)
    dst, rep = _ce(torch, xp, fifo, src_np)
    assert np.array_equal(from_dev(dst), want)
    assert 1 <= rep.max_occupancy <= nslots
    _check_state(torch, xp, fifo, fifos, nslots, slot, hops)
    xp.xp_fifo_destroy(fifo)


@pytest.mark.parametrize("place", [0, 1], ids=["device-1hop", "host-2hops"])
def test_ce_operations_continue(env, place):
    # proxy operations keep their own counters; SIMPLE and posted operations
    # in between use the FIFO's other counters and leave them alone
    torch, xp = env
    hops = 1 + place
    nchan, nslots, slot = 3, 2, 1024
    fifo = _fifo(xp, nchan, nslots, slot, place, lanes=2)
    fifos = None
    for i in range(4):
        src_np = workloads.uniform_bytes(9000 + 1234 * i, seed=70 + i)
        want, fifos, _ = oracle.ce_transfer(src_np, nchan, nslots, slot, hops=hops, seed=i, fifos=fifos)
        dst, _ = _ce(torch, xp, fifo, src_np)
        assert np.array_equal(from_dev(dst), want)
        _check_state(torch, xp, fifo, fifos, nslots, slot, hops, rings=False)
        s_np = workloads.uniform_bytes(5000 + i, seed=90 + i)
        s = to_dev(torch, s_np)
        out = torch.zeros_like(s)
        xp.xp_send_recv(fifo, s, out, s_np.nbytes, torch.cuda.current_stream())
        assert xp.xp_fifo_status(fifo, True)[0] == xp.XP_OK
        assert np.array_equal(from_dev(out), s_np)
    xp.xp_fifo_destroy(fifo)


def test_ce_device_workload(env):
    # 1 GiB of bf16 normals, 16 channels of 8 x 512 KiB, one copy-engine hop
    torch, xp = env
    w = workloads.SIMPLE_MULTI
    src_np = workloads.normal_bf16_bits(w["nelems"], w["seed"]).view(np.uint8)
    fifo = _fifo(xp, w["nchannels"], w["nslots"], w["slot_bytes"], 0, lanes=4)
    dst, rep = _ce(torch, xp, fifo, src_np)
    assert np.array_equal(from_dev(dst), src_np)
    assert rep.max_occupancy <= w["nslots"]
    xp.xp_fifo_destroy(fifo)


def test_ce_host_workload(env):
    # 256 MiB fp32 through the host-placed FIFO of 8 channels x 8 x 1 MiB:
    # device -> host -> device copies by the copy engines
    torch, xp = env
    w = workloads.HOST_FIFO
    src_np = workloads.uniform_f32(w["nelems"], w["seed"]).view(np.uint8)
    want, fifos, _ = oracle.ce_transfer(src_np, w["nchannels"], w["nslots"], w["slot_bytes"], hops=2, seed=5)
    fifo = _fifo(xp, w["nchannels"], w["nslots"], w["slot_bytes"], 1, lanes=2)
    dst, _ = _ce(torch, xp, fifo, src_np)
    assert np.array_equal(from_dev(dst), want)
    _check_state(torch, xp, fifo, fifos, w["nslots"], w["slot_bytes"], 2)
    xp.xp_fifo_destroy(fifo)


def test_ce_needs_enable_and_survives_reset(env):
    torch, xp = env
    src = torch.arange(50000, dtype=torch.int32, device="cuda")
    dst = torch.zeros_like(src)
    f = xp.xp_fifo_create(2, 2, 4096)
    with pytest.raises(xp.XpError) as e:
        xp.xp_send_recv_ce(f, src, dst, src.numel() * 4, torch.cuda.current_stream())
    assert e.value.status == xp.XP_ERR_INVALID
    xp.xp_fifo_enable_ce(f)
    xp.xp_fifo_enable_ce(f)          # no-op
    for _ in range(2):
        xp.xp_send_recv_ce(f, src, dst, src.numel() * 4, torch.cuda.current_stream())
        assert xp.xp_fifo_status(f, True)[0] == xp.XP_OK
        assert torch.equal(dst, src)
        dst.zero_()
        xp.xp_fifo_reset(f)           # the pump restarts on zeroed counters
        d = xp.xp_fifo_describe(f, 0)
        assert not raw_view(torch, d.ce, 2048 // 8, "<u8").cpu().numpy().any()
    xp.xp_fifo_destroy(f)
    ll = xp.xp_fifo_create(1, 2, 4096, xp.XP_PROTO_LL)
    with pytest.raises(xp.XpError) as e:
        xp.xp_fifo_enable_ce(ll)
    assert e.value.status == xp.XP_ERR_INVALID
    xp.xp_fifo_destroy(ll)


def test_pump_refuses_a_bad_size_word(env):
    # Failure on the host side of the proxy mode, made on the host: a size
    # word larger than a slot appears with tail[0] (written into the mapped
    # control block while no kernel runs).  The pump stops instead of copying
    # out of bounds, the next transfer's wait runs out, xp_fifo_status reports
    # it with the pump's message, and a reset restarts the pump.
    import time
    torch, xp = env
    f = _fifo(xp, 1, 2, 4096, 0)
    d = xp.xp_fifo_describe(f, 0)
    w = raw_view(torch, d.ce, 2048 // 8, "<u8")
    w[640 // 8] = 1 << 30          # size word of slot 0
    w[TAIL0] = 1
    torch.cuda.synchronize()
    time.sleep(0.2)                # the pump polls at least every 50 us
    xp.xp_set_spin_timeout_ns(50_000_000)
    try:
        w[TAIL0] = 0               # leave the sender's counters consistent
        torch.cuda.synchronize()
        src = torch.ones(8192, dtype=torch.uint8, device="cuda")
        dst = torch.zeros_like(src)
        xp.xp_send_recv_ce(f, src, dst, 8192, torch.cuda.current_stream())
        st, rep = xp.xp_fifo_status(f, True)
        assert st == xp.XP_ERR_TIMEOUT, st
        assert "size word 1073741824" in xp.xp_last_error()
        xp.xp_fifo_reset(f)
        xp.xp_set_spin_timeout_ns(2_000_000_000)
        xp.xp_send_recv_ce(f, src, dst, 8192, torch.cuda.current_stream())
        assert xp.xp_fifo_status(f, True)[0] == xp.XP_OK and bool((dst == 1).all())
    finally:
        xp.xp_set_spin_timeout_ns(2_000_000_000)
    xp.xp_fifo_destroy(f)


def test_objects_created_while_a_proxy_transfer_runs(env):
    # FIFOs and rings are set up on streams of their own, so creating,
    # resetting and destroying them while a proxy transfer waits for the
    # pump's copies neither waits for that transfer nor holds the copies up
    torch, xp = env
    xp.xp_set_spin_timeout_ns(500_000_000)
    try:
        f = _fifo(xp, 2, 4, 65536, 0)
        src = to_dev(torch, workloads.uniform_bytes(1 << 20, seed=21))
        dst = torch.zeros_like(src)
        for make in (lambda: xp.xp_fifo_destroy(xp.xp_fifo_create(2, 2, 4096)),
                     lambda: xp.xp_ring_destroy(xp.xp_ring_create(4, 2, 4, 65536)),
                     lambda: xp.xp_fifo_destroy(xp.xp_fifo_create(2, 2, 4096, xp.XP_PROTO_LL128))):
            dst.zero_()
            torch.cuda.synchronize()
            xp.xp_send_recv_ce(f, src, dst, 1 << 20, torch.cuda.current_stream())
            make()
            st, rep = xp.xp_fifo_status(f, True)
            assert st == xp.XP_OK, (st, rep.where)
            assert torch.equal(src, dst)
        xp.xp_fifo_destroy(f)
    finally:
        xp.xp_set_spin_timeout_ns(2_000_000_000)
