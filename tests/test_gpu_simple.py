"""SIMPLE, zero-copy and host-placed FIFO transfers on the GPU, element by
element against the CPU oracle on the same seeded inputs."""
import functools

import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_util import ctl_words, from_dev, raw_view, to_dev, torch_cuda

pytestmark = pytest.mark.gpu


@functools.lru_cache(maxsize=2)
def _multi_input():
    w = workloads.SIMPLE_MULTI
    return workloads.normal_bf16_bits(w["nelems"], w["seed"]).view(np.uint8)


@pytest.fixture(scope="module")
def env():
    torch = torch_cuda()
    from collective_transport_plane_gb300 import build
    build.build()
    import collective_transport_plane_gb300.xp as xp
    xp.xp_set_spin_timeout_ns(2_000_000_000)
    return torch, xp


def _run_simple(torch, xp, src_np, nchan, nslots, slot, lanes=1, place=0, zero_copy=False, fifo=None, discard=None):
    own = fifo is None
    if own:
        fifo = xp.xp_fifo_create(nchan, nslots, slot, xp.XP_PROTO_SIMPLE, place)
        xp.xp_fifo_set_lanes(fifo, lanes)
        xp.xp_fifo_set_discard(fifo, discard)   # None: by the FIFO's size
    src = to_dev(torch, src_np)
    dst = torch.zeros_like(src)
    s = torch.cuda.current_stream()
    if zero_copy:
        xp.xp_send_recv_zero_copy(fifo, src, dst, src_np.nbytes, s)
    else:
        xp.xp_send_recv(fifo, src, dst, src_np.nbytes, s)
    st, rep = xp.xp_fifo_status(fifo, True)
    assert st == xp.XP_OK, (st, rep.where, rep.observed, rep.expected)
    assert rep.max_occupancy <= nslots
    out = from_dev(dst)
    if own:
        xp.xp_fifo_destroy(fifo)
    return out, rep


def test_simple_loopback_workload(env):
    # 1 MiB of uniform bytes, one sender CTA and one receiver CTA, 8 x 64 KiB
    torch, xp = env
    w = workloads.SIMPLE_LOOPBACK
    src = workloads.uniform_bytes(w["nbytes"], w["seed"])
    want, fifos, _ = oracle.simple_transfer(src, w["nchannels"], w["nslots"], w["slot_bytes"], seed=0)
    got, rep = _run_simple(torch, xp, src, w["nchannels"], w["nslots"], w["slot_bytes"])
    assert np.array_equal(got, want)
    assert 1 <= rep.max_occupancy <= w["nslots"]


@pytest.mark.parametrize("n,nchan,nslots,slot,lanes", [
    (1, 1, 1, 16, 1), (15, 2, 2, 16, 1), (17, 3, 1, 16, 2), (4095, 3, 2, 64, 1), (65537, 4, 2, 4096, 2),
    (1000003, 16, 8, 16384, 1), (1000003, 5, 3, 65536, 4), (3 << 20, 2, 8, 65536, 8), (777777, 64, 2, 1024, 1),
    (12345, 1, 1, 4096, 3)])
@pytest.mark.parametrize("discard", [True, None])
def test_simple_sweep(env, n, nchan, nslots, slot, lanes, discard):
    # line drops forced on, and the automatic choice (off for FIFOs this small)
    torch, xp = env
    src = workloads.uniform_bytes(n, seed=n % 1000)
    want, _, _ = oracle.simple_transfer(src, nchan, nslots, slot, seed=1)
    got, _ = _run_simple(torch, xp, src, nchan, nslots, slot, lanes=lanes, discard=discard)
    assert np.array_equal(got, want)


def test_simple_counters_continue(env):
    # several operations through one FIFO: device counters end where the
    # oracle's do, and every result is exact
    torch, xp = env
    nchan, nslots, slot = 3, 2, 1024
    fifo = xp.xp_fifo_create(nchan, nslots, slot)
    xp.xp_fifo_set_lanes(fifo, 2)
    fifos = None
    for i, n in enumerate([5000, 1, 70001, 4096, 3 * 1024 * 7 + 5]):
        src = workloads.uniform_bytes(n, seed=100 + i)
        want, fifos, _ = oracle.simple_transfer(src, nchan, nslots, slot, seed=i, fifos=fifos)
        got, _ = _run_simple(torch, xp, src, nchan, nslots, slot, fifo=fifo)
        assert np.array_equal(got, want)
    for c in range(nchan):
        tail, head, ptrx, base = ctl_words(torch, xp, fifo, c)
        assert tail == head == base == fifos[c].tail
        assert ptrx == 0
    xp.xp_fifo_destroy(fifo)


@pytest.mark.parametrize("lanes,rlanes", [(1, 1), (4, 4), (9, 9), (9, 10), (10, 8)])
def test_simple_multichannel_workload(env, lanes, rlanes):
    # 1 GiB of bf16 N(0,1), 16 channels of 8 x 512 KiB; 9 + 10 lanes with
    # discards on is the configuration bench.py times, twice in a row
    torch, xp = env
    w = workloads.SIMPLE_MULTI
    src = _multi_input()
    want, _, _ = oracle.simple_transfer(src, w["nchannels"], w["nslots"], w["slot_bytes"], seed=2)
    fifo = xp.xp_fifo_create(w["nchannels"], w["nslots"], w["slot_bytes"])
    xp.xp_fifo_set_lanes(fifo, lanes)
    xp.xp_fifo_set_recv_lanes(fifo, rlanes)
    for _ in range(2):
        got, rep = _run_simple(torch, xp, src, w["nchannels"], w["nslots"], w["slot_bytes"], fifo=fifo)
        assert np.array_equal(got, want)
        assert rep.max_occupancy <= w["nslots"]
    xp.xp_fifo_destroy(fifo)


@pytest.mark.parametrize("n,nchan,nslots,slot,lanes", [
    (1, 1, 1, 16, 1), (100, 3, 2, 32, 2), (65536 + 7, 4, 2, 4096, 1), (1000003, 16, 8, 16384, 4)])
def test_zero_copy_sweep(env, n, nchan, nslots, slot, lanes):
    torch, xp = env
    src_np = workloads.uniform_bytes(n, seed=7 + n % 100)
    want, chans, _ = oracle.zero_copy_transfer(src_np, nchan, nslots, slot, seed=3)
    fifo = xp.xp_fifo_create(nchan, nslots, slot)
    xp.xp_fifo_set_lanes(fifo, lanes)
    # poison the staging slots: zero copy must leave them alone
    views = []
    for c in range(nchan):
        d = xp.xp_fifo_describe(fifo, c)
        v = raw_view(torch, d.slots, nslots * slot, "|u1")
        v.fill_(0xA5)
        views.append(v)
    for rep_i in range(2):
        got, _ = _run_simple(torch, xp, src_np, nchan, nslots, slot, zero_copy=True, fifo=fifo)
        assert np.array_equal(got, want)
    for v in views:
        assert bool((v == 0xA5).all())
    for c in range(nchan):
        tail, head, ptrx, base = ctl_words(torch, xp, fifo, c)
        assert ptrx == 0 and tail == head == base == 2 * chans[c].tail
    xp.xp_fifo_destroy(fifo)


@pytest.mark.parametrize("lanes", [6, 7, 8, 12])
def test_zero_copy_workload(env, lanes):
    # 1 GiB; 7 and 8 lanes are the bench.py rows
    torch, xp = env
    w = workloads.SIMPLE_MULTI
    src = _multi_input()
    want, _, _ = oracle.zero_copy_transfer(src, w["nchannels"], w["nslots"], w["slot_bytes"], seed=2)
    got, _ = _run_simple(torch, xp, src, w["nchannels"], w["nslots"], w["slot_bytes"], lanes=lanes, zero_copy=True)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("n,nchan,nslots,slot,lanes", [(4097, 2, 2, 1024, 1), (1 << 20, 8, 8, 65536, 2)])
def test_host_placed_sweep(env, n, nchan, nslots, slot, lanes):
    torch, xp = env
    src = workloads.uniform_bytes(n, seed=11)
    want, _, _ = oracle.simple_transfer(src, nchan, nslots, slot, seed=4)
    got, _ = _run_simple(torch, xp, src, nchan, nslots, slot, lanes=lanes, place=xp.XP_PLACE_HOST_MAPPED)
    assert np.array_equal(got, want)


def test_host_placed_workload(env):
    # 256 MiB fp32 uniform[-1,1), 8 channels of 8 x 1 MiB in pinned host memory
    torch, xp = env
    w = workloads.HOST_FIFO
    src = workloads.uniform_f32(w["nelems"], w["seed"]).view(np.uint8)
    want, _, _ = oracle.simple_transfer(src, w["nchannels"], w["nslots"], w["slot_bytes"], seed=5)
    got, _ = _run_simple(torch, xp, src, w["nchannels"], w["nslots"], w["slot_bytes"], lanes=2,
                         place=xp.XP_PLACE_HOST_MAPPED)
    assert np.array_equal(got, want)


def test_argument_errors(env):
    torch, xp = env
    fifo = xp.xp_fifo_create(2, 2, 1024)
    a = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    b = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    for args in [(a[1:], b, 16), (a, b[3:], 16), (a, a[16:], 64)]:
        with pytest.raises(xp.XpError) as e:
            xp.xp_send_recv(fifo, *args)
        assert e.value.status == xp.XP_ERR_INVALID
    xp.xp_send_recv(fifo, a, b, 0)            # no-op
    ll = xp.xp_fifo_create(1, 2, 1024, xp.XP_PROTO_LL)
    with pytest.raises(xp.XpError):
        xp.xp_send_recv(ll, a, b, 12)
    with pytest.raises(xp.XpError):
        xp.xp_send_recv_zero_copy(ll, a, b, 16)
    with pytest.raises(xp.XpError):
        xp.xp_fifo_set_lanes(ll, 2)
    xp.xp_fifo_destroy(ll)
    xp.xp_fifo_destroy(fifo)


@pytest.mark.parametrize("lanes", [1, 2])
def test_zero_copy_host_placed(env, lanes):
    # control block (ptrExchange, head, tail) in mapped host memory
    torch, xp = env
    src = workloads.uniform_bytes(300007, seed=12)
    want, _, _ = oracle.zero_copy_transfer(src, 3, 2, 4096, seed=6)
    got, _ = _run_simple(torch, xp, src, 3, 2, 4096, lanes=lanes, place=xp.XP_PLACE_HOST_MAPPED, zero_copy=True)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("n,nchan,nslots,slot,lanes,rlanes,place", [
    (1000003, 3, 4, 65536, 2, 5, 0), (777777, 16, 2, 16384, 6, 7, 0), (65537, 2, 1, 4096, 3, 1, 0),
    (300007, 4, 2, 8192, 1, 3, 1), (1 << 20, 2, 8, 65536, 3, 2, 1)])
def test_simple_receiver_lanes(env, n, nchan, nslots, slot, lanes, rlanes, place):
    # the receiver cuts each published slot-step into its own number of stripes
    torch, xp = env
    src = workloads.uniform_bytes(n, seed=n % 91)
    want, _, _ = oracle.simple_transfer(src, nchan, nslots, slot, seed=7)
    fifo = xp.xp_fifo_create(nchan, nslots, slot, xp.XP_PROTO_SIMPLE, place)
    xp.xp_fifo_set_lanes(fifo, lanes)
    xp.xp_fifo_set_recv_lanes(fifo, rlanes)
    d = xp.xp_fifo_describe(fifo, 0)
    assert (d.lanes, d.recv_lanes) == (lanes, rlanes)
    for discard in (True, None):
        xp.xp_fifo_set_discard(fifo, discard)
        got, _ = _run_simple(torch, xp, src, nchan, nslots, slot, fifo=fifo)
        assert np.array_equal(got, want)
    xp.xp_fifo_destroy(fifo)


@pytest.mark.parametrize("mode", ["simple", "zero_copy", "posted_copy", "posted_direct"])
def test_wide_sender_lanes(env, mode):
    # 12 sender lanes: SIMPLE and copy-mode posts pair them with 4 receiver
    # lanes (a 16-CTA cluster), zero copy and direct posts with one
    torch, xp = env
    src_np = workloads.uniform_bytes((3 << 20) + 4099, seed=12)
    nchan, nslots, slot = 5, 4, 65536
    f = xp.xp_fifo_create(nchan, nslots, slot)
    xp.xp_fifo_set_lanes(f, 12)
    src = to_dev(torch, src_np)
    dst = torch.zeros_like(src)
    s = torch.cuda.current_stream()
    if mode == "simple":
        want = oracle.simple_transfer(src_np, nchan, nslots, slot, seed=2)[0]
        xp.xp_send_recv(f, src, dst, src_np.nbytes, s)
    elif mode == "zero_copy":
        want = oracle.zero_copy_transfer(src_np, nchan, nslots, slot, seed=2)[0]
        xp.xp_send_recv_zero_copy(f, src, dst, src_np.nbytes, s)
    else:
        direct = mode == "posted_direct"
        want = oracle.posted_transfer(src_np, nchan, nslots, slot, seed=2, direct=direct)[0]
        xp.xp_send_recv_posted(f, src, dst, src_np.nbytes, direct, s)
    st, rep = xp.xp_fifo_status(f, True)
    assert st == xp.XP_OK, (st, rep.where)
    assert np.array_equal(from_dev(dst), want)
    assert xp.xp_fifo_describe(f, 0).recv_lanes == 4
    with pytest.raises(xp.XpError):
        xp.xp_fifo_set_recv_lanes(f, 33)
    xp.xp_fifo_destroy(f)


def test_lanes_beyond_a_cluster_and_the_cluster_fallback(env):
    # 12 + 10 CTAs per channel: more than a cluster holds, fine while the whole
    # grid is resident (cooperative launch); 64 channels of 4 + 4 CTAs do not
    # fit at once and run as clusters; 64 x (12 + 10) fits neither way
    torch, xp = env
    for nchan, lanes, rl in ((5, 12, 10), (64, 4, 4)):
        src_np = workloads.uniform_bytes((5 << 20) + 77, seed=nchan)
        want = oracle.simple_transfer(src_np, nchan, 4, 16384, seed=3)[0]
        f = xp.xp_fifo_create(nchan, 4, 16384)
        xp.xp_fifo_set_lanes(f, lanes)
        xp.xp_fifo_set_recv_lanes(f, rl)
        src = to_dev(torch, src_np)
        dst = torch.zeros_like(src)
        xp.xp_send_recv(f, src, dst, src_np.nbytes, torch.cuda.current_stream())
        st, rep = xp.xp_fifo_status(f, True)
        assert st == xp.XP_OK, (nchan, st, rep.where)
        assert np.array_equal(from_dev(dst), want)
        xp.xp_fifo_destroy(f)
    f = xp.xp_fifo_create(64, 4, 16384)
    xp.xp_fifo_set_lanes(f, 12)
    xp.xp_fifo_set_recv_lanes(f, 10)
    with pytest.raises(xp.XpError) as e:
        xp.xp_send_recv(f, src, dst, 4096, torch.cuda.current_stream())
    assert e.value.status == xp.XP_ERR_INVALID
    xp.xp_fifo_destroy(f)


@pytest.mark.parametrize("proto,place", [(0, 0), (0, 1), (1, 0)])
def test_channel_stats(env, proto, place):
    # per-channel records: the slot-steps the oracle's partition gives, device
    # timestamps in order, watcher polls where a side has a watcher
    torch, xp = env
    C, N, S = 5, 4, 4096
    n = 3 * 4096 * 4 + 48 if proto == 0 else 40000
    f = xp.xp_fifo_create(C, N, S, proto, place)
    src = to_dev(torch, workloads.uniform_bytes(n, seed=9))
    dst = torch.zeros_like(src)
    xp.xp_send_recv(f, src, dst, n, torch.cuda.current_stream())
    assert xp.xp_fifo_status(f, True)[0] == xp.XP_OK
    per_step = S if proto == 0 else S // 2       # LL lines carry 8 payload bytes per 16
    for c, (lo, hi) in enumerate(oracle.channel_byte_ranges(n, C)):
        st = xp.xp_fifo_stats(f, c)
        assert st.steps == -(-(hi - lo) // per_step)
        assert st.t_end_ns >= st.t_start_ns > 0
        if st.steps and proto == 0 and place == 0:
            assert st.recv_polls >= 1
    xp.xp_fifo_destroy(f)


@pytest.mark.parametrize("discard", [True, False])
def test_slot_contents_only_without_discard(env, discard):
    # slot sizes that are not multiples of 128 bytes put line boundaries inside
    # stripes and across slots; delivered bytes are exact either way, and with
    # discard off the slots keep the oracle's last slot-steps
    torch, xp = env
    n, nchan, nslots, slot = 777777, 3, 4, 4096 + 80
    src_np = workloads.uniform_bytes(n, seed=17)
    want, fifos, _ = oracle.simple_transfer(src_np, nchan, nslots, slot, seed=5)
    f = xp.xp_fifo_create(nchan, nslots, slot)
    xp.xp_fifo_set_lanes(f, 3)
    xp.xp_fifo_set_discard(f, discard)
    src = to_dev(torch, src_np)
    dst = torch.zeros_like(src)
    xp.xp_send_recv(f, src, dst, n, torch.cuda.current_stream())
    assert xp.xp_fifo_status(f, True)[0] == xp.XP_OK
    assert np.array_equal(from_dev(dst), want)
    if not discard:
        for c, fo in enumerate(fifos):
            d = xp.xp_fifo_describe(f, c)
            got = raw_view(torch, d.slots, nslots * slot, "|u1").cpu().numpy()
            assert np.array_equal(got, fo.slots.reshape(-1))
    xp.xp_fifo_destroy(f)


def test_discard_automatic_choice(env):
    # by default a FIFO drops read slot lines only when its slots take at
    # least XP_DISCARD_AUTO_BYTES; an explicit setting overrides the choice
    torch, xp = env
    T = xp.XP_DISCARD_AUTO_BYTES
    for (C, N, S), want in (((16, 8, T // 128), 1), ((16, 8, T // 128 - 16), 0), ((1, 8, 65536), 0), ((1, 1, T), 1)):
        f = xp.xp_fifo_create(C, N, S)
        assert xp.xp_fifo_describe(f, 0).discard == want
        for setting, got in ((True, 1), (False, 0), (None, want)):
            xp.xp_fifo_set_discard(f, setting)
            assert xp.xp_fifo_describe(f, C - 1).discard == got
        xp.xp_fifo_destroy(f)
    # the choice takes effect: a small FIFO left at its default keeps the
    # oracle's last slot-steps in its slots
    n, nchan, nslots, slot = 300007, 2, 4, 8192 + 48
    src_np = workloads.uniform_bytes(n, seed=23)
    want, fifos, _ = oracle.simple_transfer(src_np, nchan, nslots, slot, seed=4)
    f = xp.xp_fifo_create(nchan, nslots, slot)
    xp.xp_fifo_set_lanes(f, 2)
    src = to_dev(torch, src_np)
    dst = torch.zeros_like(src)
    xp.xp_send_recv(f, src, dst, n, torch.cuda.current_stream())
    assert xp.xp_fifo_status(f, True)[0] == xp.XP_OK
    assert np.array_equal(from_dev(dst), want)
    for c, fo in enumerate(fifos):
        d = xp.xp_fifo_describe(f, c)
        got = raw_view(torch, d.slots, nslots * slot, "|u1").cpu().numpy()
        assert np.array_equal(got, fo.slots.reshape(-1))
    xp.xp_fifo_destroy(f)
