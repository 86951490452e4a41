"""LL transfers and the LL ping-pong on the GPU against the CPU oracle."""
import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_util import ctl_words, from_dev, to_dev, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = torch_cuda()
    from collective_transport_plane_gb300 import build
    build.build()
    import collective_transport_plane_gb300.xp as xp
    xp.xp_set_spin_timeout_ns(2_000_000_000)
    return torch, xp


def _ll(torch, xp, fifo, words):
    src = to_dev(torch, words)
    dst = torch.zeros_like(src)
    xp.xp_send_recv(fifo, src, dst, words.nbytes, torch.cuda.current_stream())
    st, rep = xp.xp_fifo_status(fifo, True)
    assert st == xp.XP_OK, (st, rep.where, rep.observed, rep.expected)
    return from_dev(dst)


def test_ll_size_sweep_workload(env):
    # uint32 words, 8 B ... 256 KiB in powers of two, through one LL FIFO of
    # 8 slots x 32 KiB of lines: counters and flags carry over between sizes
    torch, xp = env
    w = workloads.LL_SWEEP
    fifo = xp.xp_fifo_create(1, w["nslots"], w["slot_bytes"], xp.XP_PROTO_LL)
    fifos = None
    for n in w["sizes"]:
        words = workloads.uniform_u32(n // 4, w["seed"])
        want, fifos, _ = oracle.ll_transfer(words, 1, w["nslots"], w["slot_bytes"], seed=n, fifos=fifos)
        got = _ll(torch, xp, fifo, words)
        assert np.array_equal(got, want), n
    tail, head, _, base = ctl_words(torch, xp, fifo, 0)
    assert head == base == fifos[0].head
    xp.xp_fifo_destroy(fifo)


@pytest.mark.parametrize("n,nchan,nslots,slot", [(8, 3, 1, 16), (1000, 3, 2, 32), (65536 + 8, 4, 2, 1024),
                                                 (1 << 20, 2, 8, 32768)])
def test_ll_sweep(env, n, nchan, nslots, slot):
    torch, xp = env
    words = workloads.uniform_u32(n // 4, seed=n % 97)
    want, _, _ = oracle.ll_transfer(words, nchan, nslots, slot, seed=1)
    fifo = xp.xp_fifo_create(nchan, nslots, slot, xp.XP_PROTO_LL)
    for _ in range(2):
        assert np.array_equal(_ll(torch, xp, fifo, words), want)
    xp.xp_fifo_destroy(fifo)


def test_ll_host_placed(env):
    torch, xp = env
    words = workloads.uniform_u32(50000, seed=5)
    fifo = xp.xp_fifo_create(2, 4, 4096, xp.XP_PROTO_LL, xp.XP_PLACE_HOST_MAPPED)
    want, _, _ = oracle.ll_transfer(words, 2, 4, 4096, seed=2)
    assert np.array_equal(_ll(torch, xp, fifo, words), want)
    xp.xp_fifo_destroy(fifo)


def test_ll_pingpong(env):
    torch, xp = env
    ab = xp.xp_fifo_create(1, 8, 32768, xp.XP_PROTO_LL)
    ba = xp.xp_fifo_create(1, 8, 32768, xp.XP_PROTO_LL)
    for iters in (1, 1000, 20000):
        ns = xp.xp_ll_pingpong(ab, ba, iters, torch.cuda.current_stream())
        one_way = ns / (2 * iters)
        assert 10 < one_way < 100_000, one_way
    # the FIFOs are still consistent for ordinary transfers afterwards
    words = workloads.uniform_u32(4096, seed=9)
    assert np.array_equal(_ll(torch, xp, ab, words), words)
    xp.xp_fifo_destroy(ab)
    xp.xp_fifo_destroy(ba)
