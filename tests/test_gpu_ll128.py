"""LL128 transfers on the GPU against the CPU oracle: delivered bytes, the
lines left in every slot, and the counters."""
import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_util import ctl_words, from_dev, raw_view, to_dev, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = torch_cuda()
    from collective_transport_plane_gb300 import build
    build.build()
    import collective_transport_plane_gb300.xp as xp
    xp.xp_set_spin_timeout_ns(2_000_000_000)
    yield torch, xp
    xp.xp_set_spin_timeout_ns(2_000_000_000)


def _ll128(torch, xp, fifo, src_np):
    src = to_dev(torch, src_np)
    dst = torch.zeros_like(src)
    xp.xp_send_recv(fifo, src, dst, src_np.nbytes, torch.cuda.current_stream())
    st, rep = xp.xp_fifo_status(fifo, True)
    assert st == xp.XP_OK, (st, rep.channel, rep.where, rep.observed, rep.expected)
    return from_dev(dst)


def _slots(torch, xp, fifo, channel, nslots, slot):
    d = xp.xp_fifo_describe(fifo, channel)
    assert d.slot_stride == slot
    return raw_view(torch, d.slots, nslots * slot // 8, "<u8").cpu().numpy().reshape(nslots, slot // 128, 16)


def _check_slots(torch, xp, fifo, fifos, nslots, slot):
    for c, f in enumerate(fifos):
        assert np.array_equal(_slots(torch, xp, fifo, c, nslots, slot), f.lines), c
        _, head, _, base = ctl_words(torch, xp, fifo, c)
        assert head == base == f.head


def _slots_by_definition(words, lo, hi, nslots, L):
    """Slot contents after one transfer of words[lo:hi] through a fresh
    channel: line i of step s holds payload words 15 (s L + i) ... + 14 of
    the channel (zeros past the end) and s + 1 in word 15; each slot keeps
    the lines of the last step that wrote them."""
    want = np.zeros((nslots, L, 16), np.uint64)
    n = hi - lo
    per = 15 * L
    for s in range(-(-n // per)):
        seg = words[lo + s * per:lo + min(n, (s + 1) * per)]
        nl = -(-len(seg) // 15)
        pad = np.zeros(nl * 15, np.uint64)
        pad[:len(seg)] = seg
        want[s % nslots, :nl, :15] = pad.reshape(nl, 15)
        want[s % nslots, :nl, 15] = s + 1
    return want


def test_ll128_size_sweep_workload(env):
    # uint32 words, 8 B ... 256 KiB in powers of two, through one LL128 FIFO
    # of 8 slots x 32 KiB of lines: counters and flags carry over
    torch, xp = env
    w = workloads.LL_SWEEP
    fifo = xp.xp_fifo_create(1, w["nslots"], w["slot_bytes"], xp.XP_PROTO_LL128)
    fifos = None
    for n in w["sizes"]:
        words = workloads.uniform_u32(n // 4, w["seed"])
        want, fifos, _ = oracle.ll128_transfer(words, 1, w["nslots"], w["slot_bytes"], seed=n, fifos=fifos)
        got = _ll128(torch, xp, fifo, words)
        assert np.array_equal(got, want.view(np.uint32)), n
    _check_slots(torch, xp, fifo, fifos, w["nslots"], w["slot_bytes"])
    xp.xp_fifo_destroy(fifo)


# sizes, channels and slots that give partial lines, partial steps, one-line
# slots, slots of more lines than one pass of the copy warps covers, and
# empty channels
SWEEP = [(8, 3, 1, 128), (120, 1, 1, 128), (1000, 3, 2, 256), (4096 + 8, 5, 3, 384), (65536 + 8, 4, 2, 1024),
         (300008, 5, 3, 4096), (1 << 20, 2, 8, 32768), ((2 << 20) + 24, 1, 2, 512 << 10), (129 * 120, 2, 4, 128)]


@pytest.mark.parametrize("lanes", [1, 3])
@pytest.mark.parametrize("n,nchan,nslots,slot", SWEEP)
def test_ll128_sweep(env, n, nchan, nslots, slot, lanes):
    torch, xp = env
    src = workloads.uniform_bytes(n, seed=n % 97)
    fifo = xp.xp_fifo_create(nchan, nslots, slot, xp.XP_PROTO_LL128)
    xp.xp_fifo_set_lanes(fifo, lanes)
    fifos = None
    for k in range(2):
        want, fifos, _ = oracle.ll128_transfer(src, nchan, nslots, slot, seed=k, fifos=fifos)
        assert np.array_equal(_ll128(torch, xp, fifo, src), want.view(np.uint8))
        _check_slots(torch, xp, fifo, fifos, nslots, slot)
    xp.xp_fifo_destroy(fifo)


@pytest.mark.parametrize("lanes,rlanes", [(1, 2), (2, 1), (3, 5), (4, 5), (5, 3), (1, 8), (8, 3)])
@pytest.mark.parametrize("n,nchan,nslots,slot", [SWEEP[2], SWEEP[3], SWEEP[5], SWEEP[7], SWEEP[8]])
def test_ll128_receiver_lanes(env, n, nchan, nslots, slot, lanes, rlanes):
    # sender and receiver sides cut each slot into different stripes: a
    # sender lane waits for the credit of every receiver lane its stripe
    # meets; twice through the same FIFO
    torch, xp = env
    src = workloads.uniform_bytes(n, seed=n % 89)
    fifo = xp.xp_fifo_create(nchan, nslots, slot, xp.XP_PROTO_LL128)
    xp.xp_fifo_set_lanes(fifo, lanes)
    xp.xp_fifo_set_recv_lanes(fifo, rlanes)
    d = xp.xp_fifo_describe(fifo, 0)
    assert (d.lanes, d.recv_lanes) == (lanes, rlanes)
    fifos = None
    for k in range(2):
        want, fifos, _ = oracle.ll128_transfer(src, nchan, nslots, slot, seed=k, fifos=fifos)
        assert np.array_equal(_ll128(torch, xp, fifo, src), want.view(np.uint8))
        _check_slots(torch, xp, fifo, fifos, nslots, slot)
    xp.xp_fifo_destroy(fifo)


@pytest.mark.parametrize("lanes", [1, 2])
def test_ll128_host_placed(env, lanes):
    torch, xp = env
    src = workloads.uniform_bytes(200000, seed=5)
    fifo = xp.xp_fifo_create(2, 4, 4096, xp.XP_PROTO_LL128, xp.XP_PLACE_HOST_MAPPED)
    xp.xp_fifo_set_lanes(fifo, lanes)
    want, fifos, _ = oracle.ll128_transfer(src, 2, 4, 4096, seed=2)
    assert np.array_equal(_ll128(torch, xp, fifo, src), want.view(np.uint8))
    _check_slots(torch, xp, fifo, fifos, 4, 4096)
    xp.xp_fifo_destroy(fifo)


def test_ll128_lanes_change_between_operations(env):
    # the lanes share the channel's head and step base, so the stripes may
    # be cut differently from one operation to the next
    torch, xp = env
    fifo = xp.xp_fifo_create(3, 2, 1024, xp.XP_PROTO_LL128)
    fifos = None
    for i, (lanes, rlanes) in enumerate(((1, 1), (4, 4), (2, 5), (8, 8), (3, 3), (1, 1), (6, 2), (2, 7))):
        src = workloads.uniform_bytes(20000 + 968 * i, seed=30 + i)
        xp.xp_fifo_set_lanes(fifo, lanes)
        xp.xp_fifo_set_recv_lanes(fifo, rlanes)
        want, fifos, _ = oracle.ll128_transfer(src, 3, 2, 1024, seed=i, fifos=fifos)
        assert np.array_equal(_ll128(torch, xp, fifo, src), want.view(np.uint8)), lanes
        _check_slots(torch, xp, fifo, fifos, 2, 1024)
    xp.xp_fifo_destroy(fifo)


@pytest.mark.parametrize("lanes,rlanes", [(1, 1), (4, 4), (4, 5)])
def test_ll128_workload(env, lanes, rlanes):
    # 1 GiB of bf16 normals through 16 channels of 8 x 512 KiB LL128 slots:
    # identity, and the slots of the first and last channel by the format's
    # definition (4 + 5 lanes is the configuration bench.py times)
    torch, xp = env
    w = workloads.SIMPLE_MULTI
    src_np = workloads.normal_bf16_bits(w["nelems"], w["seed"]).view(np.uint8)
    fifo = xp.xp_fifo_create(w["nchannels"], w["nslots"], w["slot_bytes"], xp.XP_PROTO_LL128)
    xp.xp_fifo_set_lanes(fifo, lanes)
    xp.xp_fifo_set_recv_lanes(fifo, rlanes)
    assert np.array_equal(_ll128(torch, xp, fifo, src_np), src_np)
    words = src_np.view(np.uint64)
    ranges = oracle.channel_byte_ranges(src_np.nbytes, w["nchannels"])
    L = w["slot_bytes"] // 128
    for c in (0, w["nchannels"] - 1):
        lo, hi = ranges[c]
        want = _slots_by_definition(words, lo // 8, hi // 8, w["nslots"], L)
        assert np.array_equal(_slots(torch, xp, fifo, c, w["nslots"], w["slot_bytes"]), want)
        _, head, _, base = ctl_words(torch, xp, fifo, c)
        assert head == base == -(-(hi - lo) // (120 * L))
    xp.xp_fifo_destroy(fifo)


def test_ll128_argument_errors(env):
    torch, xp = env
    with pytest.raises(xp.XpError) as e:
        xp.xp_fifo_create(1, 2, 192, xp.XP_PROTO_LL128)
    assert e.value.status == xp.XP_ERR_INVALID
    f = xp.xp_fifo_create(1, 2, 256, xp.XP_PROTO_LL128)
    a = torch.zeros(64, dtype=torch.uint8, device="cuda")
    b = torch.zeros_like(a)
    for call in (lambda: xp.xp_send_recv(f, a, b, 12, torch.cuda.current_stream()),
                 lambda: xp.xp_send_recv_zero_copy(f, a, b, 64, torch.cuda.current_stream()),
                 lambda: xp.xp_send_recv_posted(f, a, b, 64, False, torch.cuda.current_stream()),
                 lambda: xp.xp_fifo_enable_ce(f),
                 lambda: xp.xp_fifo_set_lanes(f, 9),
                 lambda: xp.xp_fifo_set_recv_lanes(f, 9),
                 lambda: xp.xp_fifo_set_recv_lanes(f, 0)):
        with pytest.raises(xp.XpError) as e:
            call()
        assert e.value.status == xp.XP_ERR_INVALID
    xp.xp_fifo_destroy(f)


def test_ll128_flag_wait_times_out(env):
    # the sender is held back by a head that never advances (the channel's
    # step base moved far ahead), so the receiver's flags never arrive; both
    # waits end with a status, and after a reset the FIFO works again
    torch, xp = env
    xp.xp_set_spin_timeout_ns(50_000_000)
    fifo = xp.xp_fifo_create(1, 1, 128, xp.XP_PROTO_LL128)
    d = xp.xp_fifo_describe(fifo, 0)
    raw_view(torch, d.ctl, 128, "<u8")[48] = 1000
    torch.cuda.synchronize()
    src = to_dev(torch, workloads.uniform_bytes(4096, seed=1))
    out = torch.zeros_like(src)
    xp.xp_send_recv(fifo, src, out, 4096)
    st, rep = xp.xp_fifo_status(fifo, True)
    assert st == xp.XP_ERR_TIMEOUT
    # whichever of the three stuck waits runs out first reports
    assert rep.where in (xp.XP_WAIT_HEAD, xp.XP_WAIT_LL_FLAG, xp.XP_WAIT_SLOT_BARRIER)
    xp.xp_fifo_reset(fifo)
    xp.xp_set_spin_timeout_ns(2_000_000_000)
    xp.xp_send_recv(fifo, src, out, 4096)
    st, _ = xp.xp_fifo_status(fifo, True)
    assert st == xp.XP_OK and torch.equal(out, src)
    xp.xp_fifo_destroy(fifo)
