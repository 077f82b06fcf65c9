"""Placement of pinned host pieces into surveyed huge-page ranges (host
logic only: the ranges' states are set by hand, nothing is registered)."""
import random

import pytest

from layerwise_weight_offload_gb300.stack import PinnedBuffer, _HUGE


def _buf(n_ranges):
    b = PinnedBuffer(n_ranges * _HUGE, spare=0.0, defer=True)
    n = b.capacity // _HUGE
    b.good = [True] * n
    b.fast = [True] * n
    b.rate = [211.0] * n
    b.segments = [(0, n)]
    return b


def _check(b, sizes, offs, align):
    spans = sorted((o, o + n) for o, n in zip(offs, sizes))
    for (s0, e0), (s1, _) in zip(spans, spans[1:]):
        assert e0 <= s1, "pieces overlap"
    for o, n in zip(offs, sizes):
        assert o % align == 0
        first, last = o // _HUGE, (o + n - 1) // _HUGE
        for r in range(first, last + 1):
            assert b.good[r] and b.fast[r], "piece on a slow or non-huge range"
        assert any(a <= first and last < e for a, e in b.segments), "piece crosses a segment"


def test_fit_skips_slow_and_bad_ranges():
    b = _buf(12)
    b.fast[2] = False
    b.good[5] = False
    b.fast[6] = False
    sizes = [int(0.7 * _HUGE)] * 6
    offs = b._fit(sizes, 256)
    assert offs is not None
    _check(b, sizes, offs, 256)


def test_fit_respects_segments():
    b = _buf(10)
    b.segments = [(0, 3), (3, b.capacity // _HUGE)]
    sizes = [2 * _HUGE, 2 * _HUGE]          # the first cannot start in range 2
    offs = b._fit(sizes, 256)
    _check(b, sizes, offs, 256)
    assert offs[0] == 0 and offs[1] >= 3 * _HUGE


def test_fit_reports_no_room():
    b = _buf(4)
    n = b.capacity // _HUGE
    for r in range(n):
        b.fast[r] = r % 2 == 0               # no two adjacent fast ranges
    assert b._fit([_HUGE + 1], 256) is None
    offs = b._fit([_HUGE + 1], 256, any_range=True)
    assert offs == [0]


@pytest.mark.parametrize("seed", range(5))
def test_fit_random_states(seed):
    rng = random.Random(seed)
    b = _buf(40)
    n = b.capacity // _HUGE
    for r in range(n):
        b.good[r] = rng.random() > 0.1
        b.fast[r] = rng.random() > 0.2
    cuts = sorted(rng.sample(range(1, n), 3))
    b.segments = list(zip([0] + cuts, cuts + [n]))
    sizes = [rng.randrange(1 << 20, int(1.3 * _HUGE)) for _ in range(12)]
    offs = b._fit(sizes, 4096)
    if offs is not None:
        _check(b, sizes, offs, 4096)
