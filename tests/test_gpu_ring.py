"""Virtual ring allreduce on the GPU: every rank's output bit-exact against
the oracle's ring-order sum (fp32 and int32)."""
import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_util import from_dev, to_dev, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = torch_cuda()
    from collective_transport_plane_gb300 import build
    build.build()
    import collective_transport_plane_gb300.xp as xp
    xp.xp_set_spin_timeout_ns(2_000_000_000)
    return torch, xp


def _inputs(P, n, dtype, seed_base=10):
    return workloads.ring_inputs(P, n, dtype, seed_base)


def _ring(torch, xp, xs, nchan, nslots, slot, lanes=1, in_place=False, place=0, ring=None):
    P = len(xs)
    own = ring is None
    if own:
        ring = xp.xp_ring_create(P, nchan, nslots, slot, place)
        xp.xp_ring_set_lanes(ring, lanes)
    ins = [to_dev(torch, x) for x in xs]
    outs = ins if in_place else [torch.zeros_like(t) for t in ins]
    dt = xp.XP_F32 if xs[0].dtype == np.float32 else xp.XP_I32
    xp.xp_ring_allreduce_virtual(ring, ins, outs, len(xs[0]), dt, torch.cuda.current_stream())
    st, rep = xp.xp_ring_status(ring, True)
    assert st == xp.XP_OK, (st, rep.channel, rep.where, rep.observed, rep.expected)
    assert rep.max_occupancy <= nslots
    res = [from_dev(t) for t in outs]
    if own:
        xp.xp_ring_destroy(ring)
    return res


@pytest.mark.parametrize("P,n,nchan,nslots,slot", [
    (2, 1, 1, 2, 16), (2, 100, 1, 2, 16), (3, 257, 2, 2, 32), (4, 1000, 3, 4, 64), (8, 4099, 2, 8, 64),
    (5, 7, 4, 3, 16), (8, 1 << 16, 8, 8, 4096), (3, 300001, 3, 4, 8192), (16, 5000, 2, 2, 256)])
@pytest.mark.parametrize("dtype", ["f32", "i32"])
def test_ring_sweep(env, P, n, nchan, nslots, slot, dtype):
    torch, xp = env
    xs = _inputs(P, n, dtype, seed_base=n % 50)
    want = oracle.ring_order_sum(xs, nchan, nslots, slot)
    if n <= 5000:
        sim, _ = oracle.ring_allreduce(xs, nchan, nslots, slot, seed=1)
        assert all(np.array_equal(s, want) for s in sim)
    for got in _ring(torch, xp, xs, nchan, nslots, slot):
        assert np.array_equal(got, want)


def test_ring_in_place_and_repeated(env):
    torch, xp = env
    P, n, nchan, nslots, slot = 4, 123457, 3, 4, 4096
    ring = xp.xp_ring_create(P, nchan, nslots, slot)
    for i in range(3):
        xs = _inputs(P, n, "f32", seed_base=20 + i)
        want = oracle.ring_order_sum(xs, nchan, nslots, slot)
        for got in _ring(torch, xp, xs, nchan, nslots, slot, in_place=(i % 2 == 1), ring=ring):
            assert np.array_equal(got, want)
    xp.xp_ring_destroy(ring)


@pytest.mark.parametrize("lanes", [2, 3, 4, 8])
@pytest.mark.parametrize("P,n,nchan,nslots,slot", [(8, (1 << 18) + 5, 2, 8, 4096), (3, 100003, 3, 4, 1024),
                                                   (5, 77, 2, 2, 16)])
def test_ring_lanes(env, lanes, P, n, nchan, nslots, slot):
    # lanes split every slot-step into stripes with counters of their own:
    # the result is the same ring-order sum for any lane count
    torch, xp = env
    for dtype in ("f32", "i32"):
        xs = _inputs(P, n, dtype, seed_base=lanes)
        want = oracle.ring_order_sum(xs, nchan, nslots, slot)
        for got in _ring(torch, xp, xs, nchan, nslots, slot, lanes=lanes):
            assert np.array_equal(got, want)


def test_ring_lanes_repeated_and_host_placed(env):
    # counters of every lane carry over between operations; host-placed rings
    # share one counter set among a rank's lanes
    torch, xp = env
    P, n, nchan, nslots, slot = 4, 54321, 2, 4, 2048
    for place in (0, 1):
        ring = xp.xp_ring_create(P, nchan, nslots, slot, place)
        for i, lanes in enumerate((2, 1, 3, 2)):
            xp.xp_ring_set_lanes(ring, lanes)
            xs = _inputs(P, n, "f32", seed_base=40 + i)
            want = oracle.ring_order_sum(xs, nchan, nslots, slot)
            for got in _ring(torch, xp, xs, nchan, nslots, slot, ring=ring):
                assert np.array_equal(got, want)
        xp.xp_ring_destroy(ring)


@pytest.mark.parametrize("P,n,nchan,nslots,slot", [(3, 15000017, 2, 4, 4 << 20), (2, 18000023, 3, 2, 8 << 20)])
@pytest.mark.parametrize("dtype", ["f32", "i32"])
def test_ring_channel_groups(env, P, n, nchan, nslots, slot, dtype):
    # automatic lanes run the channels in groups whose live FIFO data (P x
    # nslots/2 x slot bytes per channel) fits 32 MiB, one launch per group:
    # here one channel per launch (24 MiB per channel), and groups of 2 and 1
    # (16 MiB per channel)
    torch, xp = env
    xs = _inputs(P, n, dtype, seed_base=P)
    want = oracle.ring_order_sum(xs, nchan, nslots, slot)
    for got in _ring(torch, xp, xs, nchan, nslots, slot, lanes=0):
        assert np.array_equal(got, want)


@pytest.mark.parametrize("dtype,lanes", [("f32", 1), ("i32", 1), ("f32", 0), ("i32", 0)])
def test_ring_workload(env, dtype, lanes):
    # 8 ranks x 256 MiB, 8 channels of 8 x 512 KiB per rank-FIFO; lanes 1 runs
    # every channel in one launch, lanes 0 lets the library pick (groups of 2
    # channels at 8 lanes, four cooperative grids of 128 CTAs)
    torch, xp = env
    w = workloads.RING
    xs = _inputs(w["nranks"], w["nelems"], dtype, w["seed_base"])
    want = oracle.ring_order_sum(xs, w["nchannels"], w["nslots"], w["slot_bytes"])
    for got in _ring(torch, xp, xs, w["nchannels"], w["nslots"], w["slot_bytes"], lanes=lanes):
        assert np.array_equal(got, want)


@pytest.mark.parametrize("dtype", ["f32", "i32"])
def test_ring_host_placed(env, dtype):
    # FIFOs in mapped host memory: the vector-copy ring kernel
    torch, xp = env
    xs = _inputs(4, 100003, dtype, seed_base=3)
    want = oracle.ring_order_sum(xs, 3, 4, 4096)
    for got in _ring(torch, xp, xs, 3, 4, 4096, place=xp.XP_PLACE_HOST_MAPPED):
        assert np.array_equal(got, want)
