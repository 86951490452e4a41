"""Receiver-driven credit transfers (posts {addr, size, idx}, completions
{size, idx}) on the GPU, against the CPU oracle on the same seeded inputs:
the delivered bytes, the final post and completion entries, the step base
and, in copy mode, the bytes left in every staging slot."""
import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_util import from_dev, raw_view, to_dev, torch_cuda

pytestmark = pytest.mark.gpu

POST_WORDS, COMPL_WORD, BASE_WORD = 8, 4096 // 8, 5120 // 8


@pytest.fixture(scope="module")
def env():
    torch = torch_cuda()
    from collective_transport_plane_gb300 import build
    build.build()
    import collective_transport_plane_gb300.xp as xp
    xp.xp_set_spin_timeout_ns(2_000_000_000)
    return torch, xp


def _fifo(xp, nchan, nslots, slot, lanes=1, rlanes=None):
    # slots keep their last bytes (checked against the oracle's): no discard
    f = xp.xp_fifo_create(nchan, nslots, slot, xp.XP_PROTO_SIMPLE, xp.XP_PLACE_DEVICE)
    xp.xp_fifo_set_discard(f, False)
    xp.xp_fifo_set_lanes(f, lanes)
    if rlanes is not None:
        xp.xp_fifo_set_recv_lanes(f, rlanes)
    return f


def _posted(torch, xp, fifo, src_np, direct):
    src = to_dev(torch, src_np)
    dst = torch.zeros_like(src)
    xp.xp_send_recv_posted(fifo, src, dst, src_np.nbytes, direct, torch.cuda.current_stream())
    st, rep = xp.xp_fifo_status(fifo, True)
    assert st == xp.XP_OK, (st, rep.channel, rep.where, rep.observed, rep.expected)
    return src, dst, rep


def _check_state(torch, xp, fifo, chans, nslots, slot, dst_ptr, direct, base_before, check_slots=False):
    """Post and completion entries, step base (and staging slots) of every
    channel equal the oracle's channel state."""
    for c, ch in enumerate(chans):
        d = xp.xp_fifo_describe(fifo, c)
        w = raw_view(torch, d.posted, BASE_WORD + 1, "<u8").cpu().numpy()
        assert int(w[BASE_WORD]) == ch.completed == ch.posted
        for k in range(nslots):
            q = ch.posts[k]
            addr, size, idx = (int(x) for x in w[POST_WORDS * k:POST_WORDS * k + 3])
            if q is None:
                assert idx == 0
            else:
                assert (idx, size) == (q.idx, q.size)
                if idx > base_before[c]:
                    want = (dst_ptr if direct else d.slots) + q.offset
                    assert addr == want
            cq = ch.cq[k]
            csize, cidx = int(w[COMPL_WORD + 2 * k]), int(w[COMPL_WORD + 2 * k + 1])
            assert (cidx, csize) == ((0, 0) if cq is None else cq)
        if check_slots:
            got = raw_view(torch, d.slots, nslots * slot, "|u1").cpu().numpy()
            assert np.array_equal(got, ch.slots)


SWEEP = [(1, 1, 1, 16, 1, 1), (15, 2, 2, 16, 1, 1), (17, 3, 1, 16, 2, 1), (4095, 3, 2, 64, 1, 2),
         (65537, 4, 2, 4096, 2, 3), (1000003, 16, 8, 16384, 1, 1), (1000003, 5, 3, 65536, 4, 4),
         (3 << 20, 2, 8, 65536, 8, 8), (777777, 64, 2, 1024, 1, 1), (12345, 1, 1, 4096, 3, 2)]


@pytest.mark.parametrize("direct", [False, True])
@pytest.mark.parametrize("n,nchan,nslots,slot,lanes,rlanes", SWEEP)
def test_posted_sweep(env, n, nchan, nslots, slot, lanes, rlanes, direct):
    torch, xp = env
    src_np = workloads.uniform_bytes(n, seed=n % 1000 + 7)
    want, chans, _ = oracle.posted_transfer(src_np, nchan, nslots, slot, seed=2, direct=direct)
    fifo = _fifo(xp, nchan, nslots, slot, lanes, rlanes)
    if direct:
        # the staging slots must stay untouched: poison them first
        for c in range(nchan):
            d = xp.xp_fifo_describe(fifo, c)
            raw_view(torch, d.slots, nslots * slot, "|u1").fill_(0xA5)
    _, dst, rep = _posted(torch, xp, fifo, src_np, direct)
    assert np.array_equal(from_dev(dst), want)
    assert 1 <= rep.max_occupancy <= nslots
    _check_state(torch, xp, fifo, chans, nslots, slot, dst.data_ptr(), direct, [0] * nchan,
                 check_slots=not direct)
    if direct:
        for c in range(nchan):
            d = xp.xp_fifo_describe(fifo, c)
            assert bool((raw_view(torch, d.slots, nslots * slot, "|u1") == 0xA5).all())
    xp.xp_fifo_destroy(fifo)


def test_posted_operations_continue(env):
    # copy, direct and SIMPLE operations alternate on one FIFO: the posted
    # step base carries over and the SIMPLE counters are not disturbed
    torch, xp = env
    nchan, nslots, slot = 3, 2, 1024
    fifo = _fifo(xp, nchan, nslots, slot, lanes=2, rlanes=3)
    chans = None
    for i, direct in enumerate([False, True, False, True, False]):
        src_np = workloads.uniform_bytes(9000 + 1111 * i, seed=40 + i)
        before = [0] * nchan if chans is None else [ch.completed for ch in chans]
        want, chans, _ = oracle.posted_transfer(src_np, nchan, nslots, slot, seed=i, chans=chans, direct=direct)
        _, dst, _ = _posted(torch, xp, fifo, src_np, direct)
        assert np.array_equal(from_dev(dst), want)
        _check_state(torch, xp, fifo, chans, nslots, slot, dst.data_ptr(), direct, before)
        # a SIMPLE transfer in between uses head/tail, not the posted FIFO
        s_np = workloads.uniform_bytes(5000 + i, seed=60 + i)
        s = to_dev(torch, s_np)
        out = torch.zeros_like(s)
        xp.xp_send_recv(fifo, s, out, s_np.nbytes, torch.cuda.current_stream())
        assert xp.xp_fifo_status(fifo, True)[0] == xp.XP_OK
        assert np.array_equal(from_dev(out), s_np)
    xp.xp_fifo_destroy(fifo)


@pytest.mark.parametrize("direct,lanes,rlanes,discard", [(False, 6, 7, False), (False, 9, 9, True),
                                                       (True, 6, None, False), (True, 8, None, False)])
def test_posted_workload(env, direct, lanes, rlanes, discard):
    # 1 GiB of bf16 normals through 16 channels of 8 x 512 KiB; 9 + 9 lanes
    # with discards on and direct at 6 lanes are the bench.py rows
    torch, xp = env
    w = workloads.SIMPLE_MULTI
    src_np = workloads.normal_bf16_bits(w["nelems"], w["seed"]).view(np.uint8)
    want, chans, _ = oracle.posted_transfer(src_np, w["nchannels"], w["nslots"], w["slot_bytes"], seed=3,
                                            direct=direct)
    fifo = _fifo(xp, w["nchannels"], w["nslots"], w["slot_bytes"], lanes, rlanes)
    xp.xp_fifo_set_discard(fifo, discard)
    src, dst, rep = _posted(torch, xp, fifo, src_np, direct)
    assert np.array_equal(from_dev(dst), want)
    assert rep.max_occupancy == w["nslots"]
    _check_state(torch, xp, fifo, chans, w["nslots"], w["slot_bytes"], dst.data_ptr(), direct,
                 [0] * w["nchannels"], check_slots=not (direct or discard))
    xp.xp_fifo_destroy(fifo)


def test_posted_refused_after_error_and_bad_fifos(env):
    # Both endpoints of a posted channel read one step base, so the host
    # cannot stall one side alone; a SIMPLE wait is made to time out instead
    # (its step base moved past head), and the posted operation that follows
    # on the FIFO must be refused until the FIFO is reset.
    torch, xp = env
    fifo = _fifo(xp, 2, 2, 4096)
    src = torch.ones(100000, dtype=torch.uint8, device="cuda")
    dst = torch.zeros_like(src)
    xp.xp_set_spin_timeout_ns(50_000_000)
    try:
        d = xp.xp_fifo_describe(fifo, 0)
        raw_view(torch, d.ctl, 128, "<u8")[48] = 1000
        torch.cuda.synchronize()
        xp.xp_send_recv(fifo, src, dst, 8192, torch.cuda.current_stream())
        assert xp.xp_fifo_status(fifo, True)[0] == xp.XP_ERR_TIMEOUT
        dst.zero_()   # channel 1 of that transfer was not stalled and delivered its half
        for direct in (False, True):
            xp.xp_send_recv_posted(fifo, src, dst, src.numel(), direct, torch.cuda.current_stream())
            st, rep = xp.xp_fifo_status(fifo, True)
            assert st == xp.XP_ERR_ABORTED and rep.where == xp.XP_WAIT_STICKY
        assert not bool(dst.any())
    finally:
        xp.xp_set_spin_timeout_ns(2_000_000_000)
    xp.xp_fifo_reset(fifo)
    xp.xp_send_recv_posted(fifo, src, dst, src.numel(), True, torch.cuda.current_stream())
    assert xp.xp_fifo_status(fifo, True)[0] == xp.XP_OK
    assert bool((dst == 1).all())
    xp.xp_fifo_destroy(fifo)
    # LL or host-placed FIFOs have no posted mode
    for proto, place in [(xp.XP_PROTO_LL, xp.XP_PLACE_DEVICE), (xp.XP_PROTO_SIMPLE, xp.XP_PLACE_HOST_MAPPED)]:
        f = xp.xp_fifo_create(1, 2, 4096, proto, place)
        with pytest.raises(xp.XpError) as e:
            xp.xp_send_recv_posted(f, src, dst, 64, False, torch.cuda.current_stream())
        assert e.value.status == xp.XP_ERR_INVALID
        xp.xp_fifo_destroy(f)


@pytest.mark.parametrize("lanes,rlanes", [(1, 1), (3, 5), (10, 8)])
def test_posted_copy_with_discard(env, lanes, rlanes):
    # with the receivers dropping read slot lines from L2, the delivered bytes,
    # posts and completions still equal the oracle's (the slots' final bytes
    # are undefined and not compared)
    torch, xp = env
    n, nchan, nslots, slot = 1000003, 5, 3, 65536 + 48
    src_np = workloads.uniform_bytes(n, seed=91)
    want, chans, _ = oracle.posted_transfer(src_np, nchan, nslots, slot, seed=2)
    fifo = _fifo(xp, nchan, nslots, slot, lanes, rlanes)
    xp.xp_fifo_set_discard(fifo, True)
    _, dst, _ = _posted(torch, xp, fifo, src_np, False)
    assert np.array_equal(from_dev(dst), want)
    _check_state(torch, xp, fifo, chans, nslots, slot, dst.data_ptr(), False, [0] * nchan)
    xp.xp_fifo_destroy(fifo)
