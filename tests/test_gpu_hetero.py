"""Heterogeneous blocks of 1-byte and 2-byte dtype groups through the engine
([D5] "Request and loading constraints": an int8 weight with an fp32 scale,
an fp8 weight with an e8m0 block scale, each contiguous or a transposed
view, packed in physical order; "Validation coverage": heterogeneous-block
regression tests).  Every slot the compute stream reads holds the oracle's
image of its block byte for byte, the schedule is the oracle's, and a
transposed view rebuilt over the slot equals the original tensor.  The
engine runs with its `checks` option: every prefetch's copies pass the
offset checks against their block's plan before they are issued."""
import numpy as np
import pytest
import torch

import oracle
from tests._util import build_lib
from layerwise_weight_offload_gb300 import dlo
from layerwise_weight_offload_gb300.stack import PinnedBuffer

pytestmark = pytest.mark.gpu

MODES = [dlo.COPY_DMA, dlo.COPY_KERNEL, dlo.COPY_AUTO, dlo.COPY_STAGED]


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_lib()


def _block_specs():
    """Three blocks of different parameter sets; (name, shape, dtype[, strides])."""
    a = [("w_fp8", (96, 64), dlo.FP8_E4M3, (1, 96)),      # transposed finalized weight
         ("w_fp8.scale", (96, 2), dlo.E8M0),               # one scale per 32 weights
         ("norm", (64,), dlo.F32),
         ("proj", (32, 16), dlo.BF16)]
    b = [("w_int8", (128, 48), dlo.I8),
         ("w_int8.scale", (128,), dlo.F32),
         ("emb", (7, 5), dlo.F16),
         ("w2_fp8", (40, 33), dlo.FP8_E5M2, (1, 40)),
         ("w2_fp8.scale", (40,), dlo.F32)]
    c = [("w", (64, 64), dlo.BF16),
         ("flags", (13,), dlo.U8),
         ("w_int8", (17, 9), dlo.I8, (16, 1))]               # rows padded to 16 bytes
    return [a, b, c]


def _storage(d):
    return oracle.storage_extent(d[1], d[3]) if len(d) > 3 else int(np.prod(d[1]))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shards", [1, 3, 4])
def test_heterogeneous_blocks_stream_exact(mode, shards):
    rng = np.random.default_rng(shards * 10 + mode)
    specs = _block_specs()
    plans = [dlo.Plan(s, shards) for s in specs]
    raws = [[rng.integers(0, 256, size=_storage(d) * dlo.ESIZE[d[2]], dtype=np.uint8)
             for d in s] for s in specs]
    # pinned, device-mapped host shards of every block
    pieces = [(b, g) for b, p in enumerate(plans) for g in range(p.info().n_groups)
              for _ in range(shards)]
    sizes = [plans[b].group(g).shard_alloc_bytes for b, g in pieces]
    buf = PinnedBuffer(sum(-(-n // 256) * 256 for n in sizes) + 4096, defer=True)
    offs = buf.place(sizes, 256)
    buf.register()
    ptrs, at = [], 0
    for b, p in enumerate(plans):
        n = p.info().n_groups * shards
        ptrs.append([buf.ptr + o for o in offs[at:at + n]])
        at += n
        p.shard_host([r.ctypes.data for r in raws[b]], ptrs[b])
    images = []
    for b, s in enumerate(specs):
        img, _, _, _ = oracle.slot_image(raws[b], [_storage(d) for d in s], [d[2] for d in s],
                                         [dlo.ESIZE[d[2]] for d in s], shards, 256)
        images.append(img)
    slot_bytes = max(p.info().slot_bytes for p in plans)
    slot_bytes = -(-slot_bytes // 256) * 256
    slots = [torch.empty(slot_bytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream()
    n_blocks, steps = 3, 3
    staging, gather, staging_bytes = None, None, 0
    if mode == dlo.COPY_STAGED:
        staging_bytes = -(-max(p.info().staging_bytes for p in plans) // 256) * 256
        staging = [torch.empty(staging_bytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
        gather = torch.cuda.Stream()
    e = dlo.Engine(n_blocks, slots[0], slots[1], slot_bytes, compute, copy, mode,
                   staging=staging, staging_bytes=staging_bytes, gather_stream=gather,
                   checks=True)
    for b in range(n_blocks):
        e.register_block(b, plans[b], ptrs[b])
    e.prefetch(0, 0)
    snaps = []
    for k in range(n_blocks * steps):
        i = k % n_blocks
        slot = e.pre_forward(i)
        snap = torch.empty_like(slots[slot])
        with torch.cuda.stream(compute):
            snap.copy_(slots[slot])
        snaps.append((i, snap))
        e.post_forward(i)
    torch.cuda.synchronize()
    fetched = [0] + [(k + 1) % n_blocks for k in range(n_blocks * steps)]
    per_phase = 2 if mode == dlo.COPY_STAGED else 1
    assert e.query().checked_pieces == per_phase * shards * sum(
        plans[b].info().n_groups for b in fetched)
    log = e.schedule_log()
    ref = oracle.schedule(n_blocks, steps)
    assert [tuple(x[:6]) for x in log] == [tuple(int(v) for v in r[:6]) for r in ref]
    for i, snap in snaps:
        got = snap.cpu().numpy()
        for g in plans[i].groups():
            n = shards * g.shard_bytes
            assert np.array_equal(got[g.base:g.base + n], images[i][g.base:g.base + n]), (i, g.dtype)
    # the transposed fp8 weight of block 0, rebuilt over the slot on the GPU
    i0 = [k for k, (i, _) in enumerate(snaps) if i == 0][-1]
    pi = plans[0].param(0)
    dev = snaps[i0][1]
    view = torch.as_strided(dev, size=(96, 64), stride=tuple(pi.stride[:2]),
                            storage_offset=pi.slot_offset)
    want = raws[0][0].reshape(64, 96).T                  # the original transposed tensor
    assert np.array_equal(view.cpu().numpy(), want)
    e.destroy()
    buf.close()
