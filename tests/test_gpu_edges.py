"""Edge cases at the limits of the interface, against the oracle: the largest
channel and slot counts, a 1 GiB slot, 16 ranks, and LL flags crossing the
2^32 wrap of the step counter."""
import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_util import from_dev, raw_view, to_dev, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = torch_cuda()
    from collective_transport_plane_gb300 import build
    build.build()
    import collective_transport_plane_gb300.xp as xp
    xp.xp_set_spin_timeout_ns(2_000_000_000)
    return torch, xp


@pytest.mark.parametrize("mode", ["simple", "zero_copy", "posted_copy", "posted_direct", "ce", "ll"])
def test_max_channels_and_slots(env, mode):
    # 64 channels x 64 slots of 16 bytes: every channel wraps its FIFO 3 times
    torch, xp = env
    C, N, S = 64, 64, 16
    n = C * N * S * 3 + (8 if mode == "ll" else 5)
    f = xp.xp_fifo_create(C, N, S, xp.XP_PROTO_LL if mode == "ll" else xp.XP_PROTO_SIMPLE)
    s = torch.cuda.current_stream()
    if mode == "ll":
        src_np = workloads.uniform_u32(n // 4, seed=64)
        want = oracle.ll_transfer(src_np, C, N, S, seed=1)[0]
    else:
        src_np = workloads.uniform_bytes(n, seed=64)
        if mode == "simple":
            want = oracle.simple_transfer(src_np, C, N, S, seed=1)[0]
        elif mode == "zero_copy":
            want = oracle.zero_copy_transfer(src_np, C, N, S, seed=1)[0]
        elif mode == "ce":
            xp.xp_fifo_enable_ce(f)
            want = oracle.ce_transfer(src_np, C, N, S, seed=1)[0]
        else:
            want = oracle.posted_transfer(src_np, C, N, S, seed=1, direct=mode == "posted_direct")[0]
    src = to_dev(torch, src_np)
    dst = torch.zeros_like(src)
    {"simple": xp.xp_send_recv, "ll": xp.xp_send_recv, "zero_copy": xp.xp_send_recv_zero_copy,
     "ce": xp.xp_send_recv_ce,
     "posted_copy": lambda *a: xp.xp_send_recv_posted(*a[:4], False, a[4]),
     "posted_direct": lambda *a: xp.xp_send_recv_posted(*a[:4], True, a[4])}[mode](f, src, dst, n, s)
    st, rep = xp.xp_fifo_status(f, True)
    assert st == xp.XP_OK, (st, rep.channel, rep.where)
    assert np.array_equal(from_dev(dst), want)
    xp.xp_fifo_destroy(f)


@pytest.mark.parametrize("lanes", [1, 8])
def test_ll128_max_channels_and_slots(env, lanes):
    # 64 channels x 64 one-line slots, every channel wrapping its FIFO 3
    # times; at 8 lanes most lanes own no line, and the 1024 CTAs run in
    # waves (the lanes never wait for one another)
    torch, xp = env
    C, N, S = 64, 64, 128
    n = C * N * 120 * 3 + 8
    f = xp.xp_fifo_create(C, N, S, xp.XP_PROTO_LL128)
    xp.xp_fifo_set_lanes(f, lanes)
    src_np = workloads.uniform_bytes(n, seed=65)
    want = oracle.ll128_transfer(src_np, C, N, S, seed=1)[0].view(np.uint8)
    src = to_dev(torch, src_np)
    dst = torch.zeros_like(src)
    xp.xp_send_recv(f, src, dst, n, torch.cuda.current_stream())
    st, rep = xp.xp_fifo_status(f, True)
    assert st == xp.XP_OK, (st, rep.channel, rep.where)
    assert np.array_equal(from_dev(dst), want)
    xp.xp_fifo_destroy(f)


def test_ll128_large_slot(env):
    # one channel of 2 slots of 512 MiB of lines (480 MiB of payload each)
    # at 8 lanes: 1.5 GiB moves in four slot-steps, the last one short, and
    # wraps the FIFO; identity is the oracle's result for a copy of any size
    torch, xp = env
    S = 512 << 20
    n = (3 << 29) - 8
    src = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda",
                        generator=torch.Generator(device="cuda").manual_seed(7))
    dst = torch.zeros_like(src)
    f = xp.xp_fifo_create(1, 2, S, xp.XP_PROTO_LL128)
    xp.xp_fifo_set_lanes(f, 8)
    xp.xp_send_recv(f, src, dst, n, torch.cuda.current_stream())
    st, rep = xp.xp_fifo_status(f, True)
    assert st == xp.XP_OK, (st, rep.where)
    assert torch.equal(dst, src)
    xp.xp_fifo_destroy(f)


def test_one_gib_slot(env):
    # a single channel of 2 slots of 1 GiB: 64-bit offsets inside one slot-step
    torch, xp = env
    S = 1 << 30
    n = S + (S >> 1) + 3
    src_np = workloads.uniform_bytes(n, seed=30)
    want = oracle.simple_transfer(src_np, 1, 2, S, seed=0)[0]
    f = xp.xp_fifo_create(1, 2, S)
    xp.xp_fifo_set_lanes(f, 8)
    src = to_dev(torch, src_np)
    dst = torch.zeros_like(src)
    xp.xp_send_recv(f, src, dst, n, torch.cuda.current_stream())
    st, rep = xp.xp_fifo_status(f, True)
    assert st == xp.XP_OK, (st, rep.where)
    assert np.array_equal(from_dev(dst), want)
    xp.xp_fifo_destroy(f)


@pytest.mark.parametrize("dtype", ["f32", "i32"])
def test_sixteen_ranks_automatic_lanes(env, dtype):
    torch, xp = env
    P, n, C, N, S = 16, 300007, 2, 4, 4096
    xs = workloads.ring_inputs(P, n, dtype, 60)
    want = oracle.ring_order_sum(xs, C, N, S)
    r = xp.xp_ring_create(P, C, N, S)          # lanes 0: chosen by the library
    ins = [to_dev(torch, x) for x in xs]
    outs = [torch.zeros_like(t) for t in ins]
    xp.xp_ring_allreduce_virtual(r, ins, outs, n, xp.XP_F32 if dtype == "f32" else xp.XP_I32,
                                 torch.cuda.current_stream())
    st, _ = xp.xp_ring_status(r, True)
    assert st == xp.XP_OK
    for t in outs:
        assert np.array_equal(from_dev(t), want)
    xp.xp_ring_destroy(r)


def test_ll_flags_cross_the_32_bit_wrap(env):
    # LL flags are (step + 1) mod 2^32.  Start the step counters 2N + 3 steps
    # below 2^32 (every slot is used once before the wrap, as after a long
    # run) and run across it: the flag of step 2^32 - 1 is 0.
    torch, xp = env
    C, N, S = 2, 4, 64
    B = (1 << 32) - 2 * N - 3
    f = xp.xp_fifo_create(C, N, S, xp.XP_PROTO_LL)
    for c in range(C):
        ctl = raw_view(torch, xp.xp_fifo_describe(f, c).ctl, 128, "<u8")
        ctl[16] = B          # head
        ctl[48] = B          # step base
    torch.cuda.synchronize()
    words = workloads.uniform_u32(1000, seed=32)
    fifos = [oracle.LLFifo(N, S, step0=B) for _ in range(C)]
    want, fifos, _ = oracle.ll_transfer(words, C, N, S, seed=3, fifos=fifos)
    src = to_dev(torch, words)
    dst = torch.zeros_like(src)
    xp.xp_send_recv(f, src, dst, words.nbytes, torch.cuda.current_stream())
    st, rep = xp.xp_fifo_status(f, True)
    assert st == xp.XP_OK, (st, rep.where, rep.observed, rep.expected)
    assert np.array_equal(from_dev(dst), want)
    for c in range(C):
        ctl = raw_view(torch, xp.xp_fifo_describe(f, c).ctl, 128, "<u8").cpu().numpy()
        assert int(ctl[48]) == int(ctl[16]) == fifos[c].head > (1 << 32)
    xp.xp_fifo_destroy(f)
