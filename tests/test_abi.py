"""The C ABI library builds, loads and exports every entry point include/xp.h
declares; argument errors that need no GPU are reported without a launch."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "xp.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(xp_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def xp():
    from collective_transport_plane_gb300 import build
    build.build()
    import collective_transport_plane_gb300.xp as xp
    return xp


def test_every_declared_symbol_is_exported(xp):
    names = _declared()
    assert len(names) == 28, names
    out = subprocess.run(["nm", "-D", "--defined-only", xp.library_path()], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (xp_[a-z0-9_]+)", out))
    assert set(names) <= exported
    assert sorted(xp.EXPORTS) == names
    for n in names:
        assert callable(getattr(xp._lib, n))


def test_status_strings(xp):
    assert xp.xp_version() == 1
    assert xp.xp_status_string(xp.XP_OK) == "ok"
    assert "timed out" in xp.xp_status_string(xp.XP_ERR_TIMEOUT)


@pytest.mark.parametrize("args", [
    (0, 8, 1024, 0, 0), (65, 8, 1024, 0, 0), (1, 0, 1024, 0, 0), (1, 65, 1024, 0, 0),
    (1, 8, 0, 0, 0), (1, 8, 24, 0, 0), (1, 8, 1024, 3, 0), (1, 8, 1024, 0, 5), (64, 64, 1 << 31, 0, 0),
    (1, 8, 192, 2, 0)])
def test_fifo_create_rejects_bad_arguments(xp, args):
    with pytest.raises(xp.XpError) as e:
        xp.xp_fifo_create(*args)
    assert e.value.status == xp.XP_ERR_INVALID


@pytest.mark.parametrize("args", [(1, 1, 8, 1024, 0), (17, 1, 8, 1024, 0), (8, 1, 1, 1024, 0), (8, 1, 8, 8, 0)])
def test_ring_create_rejects_bad_arguments(xp, args):
    with pytest.raises(xp.XpError) as e:
        xp.xp_ring_create(*args)
    assert e.value.status == xp.XP_ERR_INVALID


def test_null_handles_are_rejected(xp):
    for fn in (xp._lib.xp_fifo_set_lanes, xp._lib.xp_ring_set_lanes):
        assert fn(None, 1) == xp.XP_ERR_INVALID
    assert xp._lib.xp_send_recv(None, None, None, 16, None) == xp.XP_ERR_INVALID
    assert xp._lib.xp_send_recv_posted(None, None, None, 16, 0, None) == xp.XP_ERR_INVALID
    assert xp._lib.xp_fifo_destroy(None) == xp.XP_OK
    assert xp._lib.xp_ring_destroy(None) == xp.XP_OK
    with pytest.raises(xp.XpError):
        xp.xp_set_spin_timeout_ns(10)


def test_binding_mirrors_the_header(xp):
    # the automatic drop threshold and the channel descriptor's last field
    src = open(HEADER).read()
    m = re.search(r"#define XP_DISCARD_AUTO_BYTES \(\(size_t\)(\d+) << (\d+)\)", src)
    assert m and int(m.group(1)) << int(m.group(2)) == xp.XP_DISCARD_AUTO_BYTES
    body = re.search(r"typedef struct \{((?:(?!typedef struct).)*?)\} xp_channel_desc;", src, flags=re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"\b([a-z_]+);", body)
    assert fields == [f for f, _ in xp.xp_channel_desc._fields_]
