"""xp_send_recv_noalloc, the transfer for callers that cannot allocate device
memory while they run (allocator and memory-pool hooks, hard memory budgets).
Its FIFO is the library's static device array.  Checked here: the bytes it
delivers equal the oracle's SIMPLE transfer on two calls in a row, and, after
the first call has set the device up, later calls leave the device's free
memory and torch's allocations exactly as they were."""
import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_util import to_dev, torch_cuda

pytestmark = pytest.mark.gpu


def test_noalloc_equals_the_oracle_on_consecutive_calls():
    torch = torch_cuda()
    from collective_transport_plane_gb300 import build
    build.build()
    import collective_transport_plane_gb300.xp as xp

    nchan, nslots, slot = 3, 4, 64 << 10
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call, n in enumerate([(1 << 20) + 5, 777777]):
        src_np = workloads.uniform_bytes(n, seed=40 + call)
        want, _, _ = oracle.simple_transfer(src_np, nchan, nslots, slot, seed=call)
        src = to_dev(torch, src_np)
        out = torch.zeros_like(src)
        status.fill_(-1)
        xp.xp_send_recv_noalloc(src, out, n, nchan, nslots, slot, status)
        torch.cuda.synchronize()
        assert int(status.item()) == xp.XP_OK
        assert np.array_equal(out.cpu().numpy(), want)


def test_noalloc_calls_leave_device_memory_unchanged():
    torch = torch_cuda()
    import collective_transport_plane_gb300.xp as xp

    nchan, nslots, slot = 16, 8, 64 << 10   # the largest FIFO the array holds
    n = (3 << 20) + 48
    src_np = workloads.uniform_bytes(n, seed=44)
    want, _, _ = oracle.simple_transfer(src_np, nchan, nslots, slot, seed=7)
    src = to_dev(torch, src_np)
    outs = [torch.zeros_like(src) for _ in range(4)]
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    # first call: the device's set-up (module load, kernel attribute)
    xp.xp_send_recv_noalloc(src, outs[0], n, nchan, nslots, slot, status)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for out in outs[1:]:
        xp.xp_send_recv_noalloc(src, out, n, nchan, nslots, slot, status)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert free1 == free0
    assert int(status.item()) == xp.XP_OK
    for out in outs:
        assert np.array_equal(out.cpu().numpy(), want)


def test_noalloc_refuses_a_fifo_larger_than_its_array():
    torch = torch_cuda()
    import collective_transport_plane_gb300.xp as xp
    a = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    b = torch.zeros_like(a)
    with pytest.raises(xp.XpError) as e:
        xp.xp_send_recv_noalloc(a, b, 4096, 16, 8, 1 << 20)
    assert e.value.status == xp.XP_ERR_INVALID and "8 MiB" in str(e.value)
