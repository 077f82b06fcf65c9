"""dlo_check_pieces on CPU: the copies a prefetch issues, given by offsets,
against the block layout of the pages (shard r of dtype group g holds the
group's flat elements [r*S_g, (r+1)*S_g) and lands at base_g +
r*shard_bytes_g of the slot, the place all_gather_into_tensor gives it).

The correct piece lists — one copy per shard, shards split in two, the
staged H2D rows with and without their padding, the gather out of staging —
pass; each planted mistake (a byte off, two shards swapped, a piece missing
or doubled, a read past the shard, a write past the target, an unknown
group) fails and names the piece."""
import numpy as np
import pytest

import oracle
from tests._util import build_lib
from layerwise_weight_offload_gb300 import dlo

SLOT = dlo.PIECES_SLOT_FROM_SHARDS
STAGE = dlo.PIECES_STAGING_FROM_SHARDS
GATHER = dlo.PIECES_SLOT_FROM_STAGING


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_lib()


def _plan(seed):
    """A plan of 2-4 dtype groups with odd sizes (misaligned shard ends) and
    the slot layout the oracle gives for it."""
    rng = np.random.default_rng(seed)
    codes = [dlo.F32, dlo.BF16, dlo.U8, dlo.F16]
    descs = []
    for i in range(int(rng.integers(2, 6))):
        descs.append(("p%d" % i, (int(rng.integers(1, 40)), int(rng.integers(1, 9))),
                      codes[int(rng.integers(0, len(codes)))]))
    s = int(rng.integers(1, 5))
    plan = dlo.Plan(descs, s)
    numels = [int(np.prod(d[1])) for d in descs]
    raw = [np.zeros(n * dlo.ESIZE[d[2]], np.uint8) for n, d in zip(numels, descs)]
    _, gdt, gbase, used = oracle.slot_image(raw, numels, [d[2] for d in descs],
                                            [dlo.ESIZE[d[2]] for d in descs], s, 256)
    return plan, s, gbase, used


def _slot_pieces(plan, s, gbase, split=False):
    out = []
    for g, grp in enumerate(plan.groups()):
        sb = grp.shard_bytes
        for r in range(s):
            if split and sb > 1:
                h = sb // 2
                out.append((g, r, gbase[g] + r * sb, 0, h))
                out.append((g, r, gbase[g] + r * sb + h, h, sb - h))
            else:
                out.append((g, r, gbase[g] + r * sb, 0, sb))
    return out


def _stage_pieces(plan, s, padded):
    return [(g, r, grp.stage_base + r * grp.shard_alloc_bytes, 0,
             grp.shard_alloc_bytes if padded else grp.shard_bytes)
            for g, grp in enumerate(plan.groups()) for r in range(s)]


def _gather_pieces(plan, s, gbase):
    return [(g, r, gbase[g] + r * grp.shard_bytes, grp.stage_base + r * grp.shard_alloc_bytes,
             grp.shard_bytes) for g, grp in enumerate(plan.groups()) for r in range(s)]


@pytest.mark.parametrize("seed", range(12))
def test_correct_pieces_pass(seed):
    plan, s, gbase, used = _plan(seed)
    info = plan.info()
    assert info.slot_bytes == used
    assert dlo.check_pieces(plan, SLOT, _slot_pieces(plan, s, gbase), used) is None
    split = _slot_pieces(plan, s, gbase, split=True)
    assert dlo.check_pieces(plan, SLOT, split[::-1], used) is None      # any order
    for padded in (False, True):
        assert dlo.check_pieces(plan, STAGE, _stage_pieces(plan, s, padded),
                                info.staging_bytes) is None
    assert dlo.check_pieces(plan, GATHER, _gather_pieces(plan, s, gbase), used) is None


def _fails(plan, phase, pieces, target, bad):
    got = dlo.check_pieces(plan, phase, pieces, target)
    assert got is not None, "planted mistake passed"
    assert got[0] == bad, got
    return got[1]


@pytest.mark.parametrize("seed", range(12))
def test_planted_mistakes_fail(seed):
    plan, s, gbase, used = _plan(seed)
    base = _slot_pieces(plan, s, gbase)
    last = len(base) - 1
    # a destination one byte off
    p = list(base)
    g, r, d, x, n = p[last]
    p[last] = (g, r, d + 1, x, n)
    assert "belong at" in _fails(plan, SLOT, p, used + 64, last)
    # a piece read from the wrong end of its shard (source offset shifted)
    p = list(base)
    p[0] = (p[0][0], p[0][1], p[0][2] + 1, 1, p[0][4] - 1) if p[0][4] > 1 else p[0]
    if p[0] != base[0]:
        assert dlo.check_pieces(plan, SLOT, p, used) is not None        # byte 0 left uncopied
    # two shards of one group swapped (when the group has two)
    if s > 1:
        p = list(base)
        g, r, d, x, n = p[0]
        p[0] = (g, r + 1, d, x, n)
        assert "belong at" in _fails(plan, SLOT, p, used, 0)
    # a piece missing: a shard not copied
    msg = _fails(plan, SLOT, base[:-1], used, -1)
    assert "not copied" in msg
    # a piece doubled: two writes of the same bytes
    p = base + [base[last]]
    assert "both write" in _fails(plan, SLOT, p, used, len(base))
    # a read past the shard's bytes
    p = list(base)
    g, r, d, x, n = p[last]
    p[last] = (g, r, d, x, n + 1)
    assert "reads shard bytes" in _fails(plan, SLOT, p, used + 64, last)
    # a write past the target
    assert "past the target" in _fails(plan, SLOT, base, used - 1, last)
    # an unknown group / shard, an empty piece
    p = list(base)
    p[0] = (len(plan.groups()), 0, 0, 0, 1)
    _fails(plan, SLOT, p, used, 0)
    p = list(base)
    p[0] = (p[0][0], s, p[0][2], 0, p[0][4])
    _fails(plan, SLOT, p, used, 0)
    p = list(base)
    p[0] = (p[0][0], p[0][1], p[0][2], 0, 0)
    _fails(plan, SLOT, p, used, 0)
    # staged: a row past its padded shard, a gather from the wrong staging offset
    st = _stage_pieces(plan, s, True)
    g, r, d, x, n = st[last]
    st[last] = (g, r, d, x, n + 1)
    _fails(plan, STAGE, st, plan.info().staging_bytes + 64, last)
    ga = _gather_pieces(plan, s, gbase)
    g, r, d, x, n = ga[last]
    ga[last] = (g, r, d, x + 16, n)
    _fails(plan, GATHER, ga, used, last)


def test_bad_arguments():
    plan, s, gbase, used = _plan(0)
    with pytest.raises(dlo.DLOError) as ei:
        dlo.check_pieces(plan, 7, _slot_pieces(plan, s, gbase), used)
    assert ei.value.status == dlo.ERR_INVALID
    # no pieces at all: every shard uncopied
    assert dlo.check_pieces(plan, SLOT, [], used)[0] == -1
