"""Host-to-host transfers staged through device buffers (xp_send_recv_staged):
chunked copies in, SIMPLE transfers, copies out, overlapped on three streams;
the host result equals the oracle's, chunk by chunk."""
import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_util import torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = torch_cuda()
    from collective_transport_plane_gb300 import build
    build.build()
    import collective_transport_plane_gb300.xp as xp
    xp.xp_set_spin_timeout_ns(2_000_000_000)
    return torch, xp


def _pinned(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


@pytest.mark.parametrize("n,chunk,nchan,nslots,slot,lanes", [
    (1, 0, 1, 1, 16, 1), (1000003, 65536, 3, 2, 4096, 2), (5 << 20, 1 << 20, 4, 4, 65536, 3),
    ((3 << 20) + 17, 999984, 16, 8, 16384, 1), (12345, 16, 2, 2, 64, 1)])
def test_staged_matches_oracle(env, n, chunk, nchan, nslots, slot, lanes):
    torch, xp = env
    src_np = workloads.uniform_bytes(n, seed=n % 101)
    # the oracle moves the same chunks through the same FIFO geometry
    c = chunk or (64 << 20)
    want = np.concatenate([oracle.simple_transfer(src_np[o:o + c], nchan, nslots, slot, seed=o % 7)[0]
                           for o in range(0, n, c)])
    f = xp.xp_fifo_create(nchan, nslots, slot)
    xp.xp_fifo_set_lanes(f, lanes)
    hs = _pinned(torch, src_np)
    hd = _pinned(torch, np.zeros_like(src_np))
    ds = torch.empty(n, dtype=torch.uint8, device="cuda")
    dd = torch.empty_like(ds)
    s = torch.cuda.Stream()
    xp.xp_send_recv_staged(f, hs, hd, ds, dd, n, chunk, s)
    s.synchronize()
    st, rep = xp.xp_fifo_status(f, True)
    assert st == xp.XP_OK, (st, rep.where)
    assert np.array_equal(hd.numpy(), want)
    xp.xp_fifo_destroy(f)


def test_staged_orders_after_prior_work_and_rejects_bad_chunks(env):
    torch, xp = env
    f = xp.xp_fifo_create(2, 4, 4096)
    n = 1 << 20
    hs = _pinned(torch, workloads.uniform_bytes(n, seed=5))
    hd = _pinned(torch, np.zeros(n, np.uint8))
    ds = torch.empty(n, dtype=torch.uint8, device="cuda")
    dd = torch.empty_like(ds)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dd.fill_(7)                      # prior work on the stream: overwritten afterwards
    xp.xp_send_recv_staged(f, hs, hd, ds, dd, n, 1 << 18, s)
    s.synchronize()
    assert torch.equal(hd, hs) and bool(dd.cpu().eq(hs).all())
    with pytest.raises(xp.XpError) as e:
        xp.xp_send_recv_staged(f, hs, hd, ds, dd, n, 1000, s)
    assert e.value.status == xp.XP_ERR_INVALID
    xp.xp_fifo_destroy(f)
