"""Moving a block's host shards while the stream runs (the defence against
host ranges that turn slow for the GPU to read):
- dlo_engine_copy_log reports completed prefetches in order, without
  waiting for one still in flight;
- dlo_replace_block_shards waits (bounded) for copies still reading the old
  shards, then later prefetches read the new ones;
- a host block moved by HostBlocks.relocate_block between two steps, and by
  the stack's healer, streams the same bytes: slot images equal the
  oracle's, and the streamed output stays bit-identical to the resident one;
- PinnedIO (a step's input and result buffers in huge-page pinned memory):
  its buffers round-trip through the device, a move that fails its rate
  check leaves a buffer where it was, and a move that passes keeps the
  contents.
"""
import numpy as np
import pytest
import torch

import oracle
from tests._util import build_lib, raw_bytes
from layerwise_weight_offload_gb300 import dlo, workloads as W
from layerwise_weight_offload_gb300.stack import (HostBlocks, StreamedStack, ResidentStack,
                                                  PinnedIO)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_lib()


def _workload():
    # 12 host blocks of 25 MB: a pinned footprint large enough for
    # huge-page ranges (and so for relocation)
    return W.custom("reloc", n_blocks=12, hidden=1024, heads=16, mlp=4096, tokens=256,
                    shards=3, steps=2, distinct=12)


def _image(host, hb):
    p = host.params[hb]
    numels = [int(np.prod(sh)) for _, sh, _ in host.descs]
    codes = [c for _, _, c in host.descs]
    raw = [raw_bytes(p[name]) for name, _, _ in host.descs]
    return oracle.slot_image(raw, numels, codes, [W.ESIZE[c] for c in codes], host.w.shards,
                             256)[0]


def test_copy_log_and_replace_wait_for_copies_in_flight():
    w = _workload()
    host = HostBlocks(w, seed=7, keep_params=True)
    st = StreamedStack(host, copy_mode=dlo.COPY_DMA, timing=True)
    e = st.engine
    st.prime()
    torch.cuda.synchronize()
    recs, nxt = e.copy_log(0)
    assert [r[0] for r in recs] == [0] and recs[0][1] == 0 and nxt == 1
    # hold the copy stream: the next prefetch (block 1, issued by forward 0)
    # is in flight, so neither the log nor a replace of block 1 may pass it
    with torch.cuda.stream(st.copy):
        torch.cuda._sleep(int(0.3 * 2.2e9))
    e.pre_forward(0)
    recs, nxt2 = e.copy_log(nxt)
    assert recs == [] and nxt2 == nxt
    with pytest.raises(dlo.DLOError) as ei:
        e.replace_block_shards(1, host.shard_ptrs(1), timeout_ms=5)
    assert ei.value.status == dlo.ERR_TIMEOUT
    e.replace_block_shards(1, host.shard_ptrs(1), timeout_ms=10000)
    e.post_forward(0)
    torch.cuda.synchronize()
    recs, nxt3 = e.copy_log(nxt)
    assert [(r[0], r[1], r[2]) for r in recs] == [(1, 1, 1)] and nxt3 == 2
    assert recs[0][3] > 0 and recs[0][4] == sum(g.shard_bytes * w.shards for g in host.groups)
    with pytest.raises(dlo.DLOError):
        e.replace_block_shards(1, [0] * len(host.shard_ptrs(1)))
    st.close()
    host.close()


@pytest.mark.parametrize("how", ["direct", "healer"])
def test_relocated_blocks_stream_the_same_bytes(how):
    w = _workload()
    host = HostBlocks(w, seed=8, keep_params=True)
    host.pretouch()
    assert host.buf.small is False
    report = host.verify()
    assert report["rounds"] >= 1
    st = StreamedStack(host, copy_mode=dlo.COPY_DMA, heal=(how == "healer"))
    x0 = W.gen_x(w, seed=8)
    xs = x0.clone().cuda()
    st.compute.wait_stream(torch.cuda.current_stream())
    st.step(xs)
    moved = [5, 11]
    old = {hb: list(host.shard_ptrs(hb)) for hb in moved}
    if how == "direct":
        for hb in moved:
            assert host.relocate_block(hb, 1.0)
            st.engine.replace_block_shards(hb, host.shard_ptrs(hb))
    else:
        # the healer names blocks 5 and 11 once, as if their copies had
        # turned slow; the stack moves them and re-points the engine
        names = [list(moved)]
        real = st.healer.observe
        st.healer.observe = lambda recs: (real(recs), names.pop() if names else [])[1]
        st.heal()
        assert [(hb, ok) for _, hb, ok in st.heal_log] == [(5, True), (11, True)]
    for hb in moved:
        assert host.shard_ptrs(hb) != old[hb]
    # every prefetch of the next step, moved blocks included, holds the
    # oracle's image of its block
    snaps = []
    st.step(xs)
    torch.cuda.synchronize()
    for k in range(w.n_blocks):
        i = k % w.n_blocks
        slot = st.engine.pre_forward(i)
        snap = torch.empty_like(st.slots[slot])
        with torch.cuda.stream(st.compute):
            snap.copy_(st.slots[slot])
        snaps.append((i, snap))
        st.engine.post_forward(i)
    torch.cuda.synchronize()
    for i, snap in snaps:
        exp = _image(host, i % w.distinct)
        got = snap.cpu().numpy()
        for g in host.plan.groups():
            n = w.shards * g.shard_bytes
            assert np.array_equal(got[g.base:g.base + n], exp[g.base:g.base + n]), (i, g.dtype)
    torch.cuda.current_stream().wait_stream(st.compute)
    rs = ResidentStack(host)
    xr = x0.clone().cuda()
    rs.stream.wait_stream(torch.cuda.current_stream())
    for _ in range(2):
        rs.step(xr)
    torch.cuda.current_stream().wait_stream(rs.stream)
    torch.cuda.synchronize()
    assert torch.equal(xs, xr)
    assert dlo.kernel_status() == 0
    st.close()
    host.close()


def test_pinned_io_buffers_round_trip_and_move():
    shape = (1000, 777)                       # fp32: 3,108,000 bytes, not a multiple of 256
    nbytes = 1000 * 777 * 4
    io = PinnedIO(nbytes, 3)
    assert io.buf.good_fraction() == 1.0      # huge-page ranges although the buffers are small
    rates = io.verify(1.0)
    assert len(rates) == 3 and all(a > 1.0 and b > 1.0 for a, b in rates)
    assert io.relocated == [] and io.failed == []
    x = torch.randn(shape, generator=torch.Generator().manual_seed(3))
    xh = io.tensor(0, shape, torch.float32)
    xh.copy_(x)
    d = xh.cuda()
    yh = io.tensor(1, shape, torch.float32)
    yh.copy_(d, non_blocking=True)
    torch.cuda.synchronize()
    assert torch.equal(yh, x)
    # a move whose new place misses the rate: refused, buffer unchanged
    off0 = io.offs[0]
    del xh, yh
    io.verify(1e12, rounds=1)
    assert io.failed == [0, 1, 2] and io.relocated == [] and io.offs[0] == off0
    assert torch.equal(io.tensor(0, shape, torch.float32), x)
    # a move that passes: a new address, the same contents
    new = io.buf.relocate([(io.offs[0], nbytes)], 1.0)
    assert new is not None and new[0] != off0
    io.offs[0] = new[0]
    assert torch.equal(io.tensor(0, shape, torch.float32), x)
    io.close()
