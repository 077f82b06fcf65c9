"""All-or-nothing registration of host ranges ([D5] "Registered mmap
transport" and "Validation coverage": registration is all-or-nothing, a
partial registration that cannot be rolled back is fatal, unregistration
is retryable), checked on the host against fakes of the CUDA calls."""
import ctypes
import os

import numpy as np
import pytest

from layerwise_weight_offload_gb300 import dlo

PAGE = os.sysconf("SC_PAGE_SIZE")


@pytest.fixture(autouse=True)
def _fakes():
    yield
    dlo.debug_fake_host_register(0)


def _ranges(n):
    bufs = [np.zeros(3 * PAGE, dtype=np.uint8) for _ in range(n)]
    # an unaligned start and length inside each buffer
    return bufs, [b.ctypes.data + 100 for b in bufs], [PAGE + 7 for _ in bufs]


def test_all_registered_then_unregistered():
    dlo.debug_fake_host_register(1)
    bufs, ptrs, sizes = _ranges(4)
    got = dlo.host_register_ranges(ptrs, sizes)
    assert dlo.debug_fake_host_register_log() == [1, 2, 3, 4]
    # every range widened to whole pages
    exp = 0
    for p, n in zip(ptrs, sizes):
        exp += ((p + n + PAGE - 1) // PAGE - p // PAGE) * PAGE
    assert got == exp
    dlo.debug_fake_host_register(1)
    dlo.host_unregister_ranges(ptrs, sizes)
    assert dlo.debug_fake_host_register_log() == [-1, -2, -3, -4]


def test_failure_rolls_back_newest_first():
    dlo.debug_fake_host_register(1, fail_register_at=2)
    bufs, ptrs, sizes = _ranges(4)
    with pytest.raises(dlo.DLOError) as ei:
        dlo.host_register_ranges(ptrs, sizes)
    assert ei.value.status == dlo.ERR_CUDA
    assert dlo.debug_fake_host_register_log() == [1, 2, 3, -2, -1]


def test_failed_rollback_is_reported_as_partial():
    dlo.debug_fake_host_register(1, fail_register_at=3, fail_unregister_at=1)
    bufs, ptrs, sizes = _ranges(5)
    with pytest.raises(dlo.DLOError) as ei:
        dlo.host_register_ranges(ptrs, sizes)
    assert ei.value.status == dlo.ERR_PARTIAL
    # every rollback is still attempted
    assert dlo.debug_fake_host_register_log() == [1, 2, 3, 4, -3, -2, -1]


def test_first_range_failing_registers_nothing():
    dlo.debug_fake_host_register(1, fail_register_at=0)
    bufs, ptrs, sizes = _ranges(3)
    with pytest.raises(dlo.DLOError) as ei:
        dlo.host_register_ranges(ptrs, sizes)
    assert ei.value.status == dlo.ERR_CUDA
    assert dlo.debug_fake_host_register_log() == [1]


def test_limit_is_a_preflight():
    dlo.debug_fake_host_register(1)
    bufs, ptrs, sizes = _ranges(3)
    with pytest.raises(dlo.DLOError) as ei:
        dlo.host_register_ranges(ptrs, sizes, limit_bytes=2 * PAGE)
    assert ei.value.status == dlo.ERR_NOMEM
    assert dlo.debug_fake_host_register_log() == []
    assert dlo.host_register_ranges(ptrs, sizes, limit_bytes=100 * PAGE) > 0


def test_unregister_continues_past_a_failure():
    dlo.debug_fake_host_register(1, fail_unregister_at=1)
    bufs, ptrs, sizes = _ranges(4)
    with pytest.raises(dlo.DLOError) as ei:
        dlo.host_unregister_ranges(ptrs, sizes)
    assert ei.value.status == dlo.ERR_CUDA
    assert dlo.debug_fake_host_register_log() == [-1, -2, -3, -4]
    dlo.debug_fake_host_register(1)                  # retryable
    dlo.host_unregister_ranges(ptrs, sizes)


def test_bad_arguments():
    with pytest.raises(dlo.DLOError):
        dlo.host_register_ranges([0], [16])
    with pytest.raises(dlo.DLOError):
        dlo.host_register_ranges([1 << 20], [0])
    L = dlo.lib()
    assert L.dlo_host_register_ranges(None, None, 2, 0, 0, None) == dlo.ERR_INVALID


def test_engine_host_staging_arguments_fail_closed():
    L = dlo.lib()
    out = ctypes.c_void_p()
    d = dlo.EngineDesc()
    d.n_blocks = 2
    d.slot[0], d.slot[1] = 4096, 4096 * 3
    d.slot_bytes = 100
    d.compute_stream, d.copy_stream = 8, 16
    d.host_staging[0] = 4096 * 8                      # only one buffer
    d.host_staging_bytes = 100
    assert L.dlo_engine_create(ctypes.byref(d), ctypes.byref(out)) == dlo.ERR_INVALID
    d.host_staging[1] = 4096 * 8                      # the same buffer twice
    assert L.dlo_engine_create(ctypes.byref(d), ctypes.byref(out)) == dlo.ERR_INVALID
    d.host_staging[1] = 4096 * 9
    d.pack_threads = 65
    assert L.dlo_engine_create(ctypes.byref(d), ctypes.byref(out)) == dlo.ERR_INVALID


def test_ranges_sharing_pages_are_merged():
    dlo.debug_fake_host_register(1)
    buf = np.zeros(8 * PAGE, dtype=np.uint8)
    base = (buf.ctypes.data + PAGE - 1) // PAGE * PAGE
    # three ranges: the first two share a page, the third is apart
    ptrs = [base + 10, base + PAGE - 5, base + 5 * PAGE]
    sizes = [100, 200, 50]
    got = dlo.host_register_ranges(ptrs, sizes)
    assert dlo.debug_fake_host_register_log() == [1, 2]
    assert got == 3 * PAGE
