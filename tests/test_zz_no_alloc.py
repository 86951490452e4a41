"""xp_send_recv_noalloc, the transfer for callers that cannot allocate device
memory while they run (allocator hooks, hard memory budgets): its FIFO is the
library's static device array, and its result must be byte for byte the one
xp_send_recv gives, call after call."""
import pytest

import workloads
from tests.gpu_util import to_dev, torch_cuda

pytestmark = pytest.mark.gpu


def test_noalloc_matches_send_recv_on_consecutive_calls():
    torch = torch_cuda()
    from collective_transport_plane_gb300 import build
    build.build()
    import collective_transport_plane_gb300.xp as xp

    nchan, nslots, slot = 3, 4, 64 << 10
    fifo = xp.xp_fifo_create(nchan, nslots, slot)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call, n in enumerate([(1 << 20) + 5, 777777]):
        src = to_dev(torch, workloads.uniform_bytes(n, seed=40 + call))
        ref = torch.zeros_like(src)
        out = torch.zeros_like(src)
        xp.xp_send_recv(fifo, src, ref, n)
        st, _ = xp.xp_fifo_status(fifo, True)
        assert st == xp.XP_OK
        status.fill_(-1)
        xp.xp_send_recv_noalloc(src, out, n, nchan, nslots, slot, status)
        torch.cuda.synchronize()
        assert int(status.item()) == xp.XP_OK
        assert torch.equal(out, ref)
    xp.xp_fifo_destroy(fifo)


def test_noalloc_refuses_a_fifo_larger_than_its_array():
    torch = torch_cuda()
    import collective_transport_plane_gb300.xp as xp
    a = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    b = torch.zeros_like(a)
    with pytest.raises(xp.XpError) as e:
        xp.xp_send_recv_noalloc(a, b, 4096, 16, 8, 1 << 20)
    assert e.value.status == xp.XP_ERR_INVALID and "8 MiB" in str(e.value)
