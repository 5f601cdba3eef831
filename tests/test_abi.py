"""The C-ABI library loads and exports every entry point of include/mla.h (CPU).

No compute call is made: only host-side argument checks that return before
any CUDA work is enqueued.
"""

import ctypes
import os
import re

import pytest

from paged_mla_decode_gb300 import binding
from paged_mla_decode_gb300 import build as mbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "mla.h")


def _declared():
    text = open(HEADER).read()
    return re.findall(r"MLA_API\s+[\w\s\*]+?\b(mla_\w+)\s*\(", text)


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return binding.load_library()


def test_header_and_binding_agree():
    assert sorted(_declared()) == sorted(binding.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version_and_status_strings(lib):
    assert lib.mla_abi_version() == 1
    for code in range(5):
        assert lib.mla_status_string(code)
    assert b"UNKNOWN" in lib.mla_status_string(99)


def test_host_validation_returns_codes(lib):
    # negative token count / bad dtype / bad scale: rejected before any CUDA call
    assert lib.mla_kv_append(None, None, None, -1, None, 10, 64, 0, 1.0, None) == 1
    assert lib.mla_kv_append(None, None, None, 1, None, 10, 64, 7, 1.0, None) == 1
    assert lib.mla_kv_append(None, None, None, 1, None, 10, 64, 0, 0.0, None) == 1
    assert lib.mla_kv_append(None, None, None, 1, None, 10, 32, 0, 1.0, None) == 2
    assert lib.mla_kv_append(None, None, None, 1, None, 10, 64, 1, 0.5, None) == 1
    assert lib.mla_kv_append(None, None, None, 0, None, 10, 64, 0, 1.0, None) == 0
    # decode: unsupported heads, bad queries, empty batch
    args = dict(q=None, kv=None, npages=10, ps=64, dt=0, bt=None, mp=4, sl=None)
    def dec(batch, nq, heads, ps=64, scale=1.0):
        return lib.mla_decode(None, None, 10, ps, 0, None, 4, None, batch, nq, heads, 0.1,
                              scale, 0, None, 0, None, None, None)
    assert dec(1, 1, 48) == 2
    assert dec(1, 5, 64) == 1
    assert dec(1, 0, 64) == 1
    assert dec(1, 1, 64, ps=16) == 2
    assert dec(1, 1, 64, scale=-1.0) == 1
    assert dec(0, 1, 64) == 0
    assert dec(1, 1, 64) == 1            # null pointers
    assert lib.mla_decode_combine(None, None, 3, 0, None, None, None) == 0
    assert lib.mla_decode_combine(None, None, 3, 5, None, None, None) == 1
    # integrity check: bad sizes, page size, missing buffers; empty batch is a no-op
    assert lib.mla_kv_check(None, 10, None, None, 4, None, -1, 64, None, None, None) == 1
    assert lib.mla_kv_check(None, -1, None, None, 4, None, 1, 64, None, None, None) == 1
    assert lib.mla_kv_check(None, 10, None, None, 4, None, 1, 32, None, None, None) == 2
    assert lib.mla_kv_check(None, 10, None, None, 4, None, 0, 64, None, None, None) == 0
    assert lib.mla_kv_check(None, 10, None, None, 4, None, 1, 64, None, None, None) == 1
    del args


def test_workspace_size_grows_with_ctas(lib):
    a = lib.mla_decode_workspace_size(1, 1, 64, 100)
    b = lib.mla_decode_workspace_size(1, 1, 64, 200)
    assert 0 < a < b
    # per piece: 64 heads x (512 + 1) floats
    assert b - a >= 100 * 64 * 513 * 4
    assert lib.mla_decode_workspace_size(1, 9, 64, 100) == 0


def test_grouped_decode_checks_group_shape(lib):
    """Group shapes the grouped decode cannot cut are refused before any launch."""
    fake = ctypes.c_void_p(1 << 20)        # never dereferenced: the checks fail first
    args = lambda batch, forks, ctas: (fake, fake, 100, 64, 0, fake, 4, fake, batch, 1, 64,
                                       forks, fake, 0.1, 1.0, ctas, fake, 1 << 30, fake, fake,
                                       None)
    assert lib.mla_decode_grouped(*args(8, 3, 16)) == 1      # batch not a multiple of forks
    assert lib.mla_decode_grouped(*args(8, 8, 4)) == 1       # more forks than CTAs
    assert lib.mla_decode_grouped(*args(8, 0, 16)) == 1      # no forks
    assert lib.mla_decode_grouped_workspace_size(8, 1, 64, 16) > \
        lib.mla_decode_workspace_size(8, 1, 64, 16)
