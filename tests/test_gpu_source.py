"""The rank-local source path ([D5] "Rank-local path without DLO
AllGather", "Registered mmap transport"): blocks registered by the host
addresses of their parameters, one shard.  Pageable parameters are packed
by CPU threads into two bounded pinned host staging slots; parameters in a
registered (read-only) mapping are copied straight into the slots.  Every
slot the compute stream reads equals the oracle's image of its block, and
the DiT forward through source blocks equals the all-resident forward bit
for bit."""
import os
import tempfile

import numpy as np
import pytest
import torch

import oracle
from tests._util import build_lib, raw_bytes
from layerwise_weight_offload_gb300 import dlo, workloads as W
from layerwise_weight_offload_gb300.stack import HostBlocks, PinnedBuffer, ResidentStack

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_lib()


def _specs():
    return [
        [("w_fp8", (96, 64), dlo.FP8_E4M3, (1, 96)), ("w_fp8.scale", (96, 2), dlo.E8M0),
         ("norm", (64,), dlo.F32), ("proj", (32, 16), dlo.BF16)],
        [("w_int8", (128, 48), dlo.I8), ("w_int8.scale", (128,), dlo.F32),
         ("emb", (7, 5), dlo.F16)],
        [("w", (64, 64), dlo.BF16), ("flags", (13,), dlo.U8)],
    ]


def _storage(d):
    return oracle.storage_extent(d[1], d[3]) if len(d) > 3 else int(np.prod(d[1]))


def _run_schedule(e, slots, compute, n_blocks, steps):
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
    return snaps


def _check(e, snaps, plans, images, n_blocks, steps):
    log = e.schedule_log()
    ref = oracle.schedule(n_blocks, steps)
    assert [tuple(x[:6]) for x in log] == [tuple(int(v) for v in r[:6]) for r in ref]
    for i, snap in snaps:
        got = snap.cpu().numpy()
        for g in plans[i].groups():
            n = g.shard_bytes
            assert np.array_equal(got[g.base:g.base + n], images[i][g.base:g.base + n]), (i, g.dtype)


def _images(specs, raws):
    out = []
    for s, r in zip(specs, raws):
        img, _, _, _ = oracle.slot_image(r, [_storage(d) for d in s], [d[2] for d in s],
                                         [dlo.ESIZE[d[2]] for d in s], 1, 256)
        out.append(img)
    return out


def _engine(plans, host_staging=True):
    slot_bytes = -(-max(p.info().slot_bytes for p in plans) // 256) * 256
    slots = [torch.empty(slot_bytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream()
    hs = None
    if host_staging:
        hs = PinnedBuffer(2 * slot_bytes, defer=True)
        offs = hs.place([slot_bytes, slot_bytes], 256)
        hs.register()
    e = dlo.Engine(len(plans), slots[0], slots[1], slot_bytes, compute, copy, dlo.COPY_DMA,
                   host_staging=[hs.ptr + o for o in offs] if hs else None,
                   host_staging_bytes=slot_bytes if hs else 0, pack_threads=3)
    return e, slots, compute, hs


@pytest.mark.parametrize("steps", [1, 3])
def test_pageable_sources_pack_through_host_staging(steps):
    rng = np.random.default_rng(steps)
    specs = _specs()
    plans = [dlo.Plan(s, 1) for s in specs]
    raws = [[rng.integers(0, 256, size=_storage(d) * dlo.ESIZE[d[2]], dtype=np.uint8)
             for d in s] for s in specs]
    e, slots, compute, hs = _engine(plans)
    for b, p in enumerate(plans):
        e.register_block_source(b, p, [r.ctypes.data for r in raws[b]])
    snaps = _run_schedule(e, slots, compute, 3, steps)
    _check(e, snaps, plans, _images(specs, raws), 3, steps)
    st = e.query()
    assert st.n_packed_prefetches == 3 * steps + 1 and st.n_direct_prefetches == 0
    e.destroy()
    hs.close()


def test_pageable_source_without_host_staging_is_refused():
    specs = _specs()
    plans = [dlo.Plan(s, 1) for s in specs]
    e, slots, compute, _ = _engine(plans, host_staging=False)
    r = np.zeros(1 << 16, dtype=np.uint8)
    with pytest.raises(dlo.DLOError):
        e.register_block_source(0, plans[0], [r.ctypes.data] * len(specs[0]))
    with pytest.raises(dlo.DLOError):                 # sharded plans are not rank-local
        e.register_block_source(0, dlo.Plan(specs[0], 2), [r.ctypes.data] * len(specs[0]))
    e.destroy()


def test_mapping_registered_or_staged():
    # the blocks' parameters back to back in a file, mapped: registered (read
    # only, else writable) and copied straight into the slots; where the
    # platform refuses the registration (rolled back), the same mapping
    # streams through the two host staging slots instead
    rng = np.random.default_rng(7)
    specs = _specs()
    plans = [dlo.Plan(s, 1) for s in specs]
    raws = [[rng.integers(0, 256, size=_storage(d) * dlo.ESIZE[d[2]], dtype=np.uint8)
             for d in s] for s in specs]
    offs, at = [], 0
    for r in raws:
        o = []
        for x in r:
            at = -(-at // 64) * 64
            o.append(at)
            at += x.size
        offs.append(o)
    with tempfile.TemporaryDirectory() as td:
        path = os.path.join(td, "blocks.bin")
        img = np.zeros(at, dtype=np.uint8)
        for r, o in zip(raws, offs):
            for x, p in zip(r, o):
                img[p:p + x.size] = x
        img.tofile(path)
        transport = None
        for mode, ro in (("r", True), ("r+", False)):
            mm = np.memmap(path, dtype=np.uint8, mode=mode)
            base = mm.ctypes.data
            try:
                dlo.host_register_ranges([base], [at], read_only=ro)
                transport = "registered-" + mode
                break
            except dlo.DLOError as err:
                assert err.status == dlo.ERR_CUDA          # rolled back, nothing left
                del mm
        if transport is None:
            mm = np.memmap(path, dtype=np.uint8, mode="r")
            base = mm.ctypes.data
            transport = "staged"
        e, slots, compute, hs = _engine(plans, host_staging=transport == "staged")
        for b, p in enumerate(plans):
            e.register_block_source(b, p, [base + o for o in offs[b]])
        snaps = _run_schedule(e, slots, compute, 3, 2)
        _check(e, snaps, plans, _images(specs, raws), 3, 2)
        st = e.query()
        print("mapping transport:", transport)
        if transport == "staged":
            assert st.n_packed_prefetches == 7 and st.n_direct_prefetches == 0
        else:
            assert st.n_direct_prefetches == 7 and st.n_packed_prefetches == 0
        e.destroy()
        if hs is not None:
            hs.close()
        if transport != "staged":
            dlo.host_unregister_ranges([base], [at])
            with pytest.raises(dlo.DLOError) as ei:    # over a ceiling: nothing registered
                dlo.host_register_ranges([base], [at], limit_bytes=4096)
            assert ei.value.status == dlo.ERR_NOMEM
        del mm


@pytest.mark.parametrize("registered", [False, True])
def test_dit_forward_through_source_blocks_equals_resident(registered):
    w = W.custom("src", n_blocks=4, hidden=256, heads=4, mlp=1024, tokens=128, shards=1,
                 steps=2, distinct=4)
    host = HostBlocks(w, seed=9, keep_params=True)      # the resident reference
    plan = host.plan
    params = [[raw_bytes(host.params[b][name]) for name, _, _ in host.descs]
              for b in range(w.distinct)]
    hs = None
    if registered:
        flat = [np.ascontiguousarray(np.concatenate(p)) for p in params]
        ptrs, sizes = [f.ctypes.data for f in flat], [f.size for f in flat]
        dlo.host_register_ranges(ptrs, sizes)
        srcs = []
        for f, p in zip(flat, params):
            cuts = np.cumsum([0] + [x.size for x in p[:-1]])
            srcs.append([f.ctypes.data + int(c) for c in cuts])
    else:
        srcs = [[x.ctypes.data for x in p] for p in params]
    slot_bytes = -(-plan.info().slot_bytes // 256) * 256
    slots = [torch.empty(slot_bytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream()
    if not registered:
        hs = PinnedBuffer(2 * slot_bytes, defer=True)
        o = hs.place([slot_bytes, slot_bytes], 256)
        hs.register()
    e = dlo.Engine(w.n_blocks, slots[0], slots[1], slot_bytes, compute, copy, dlo.COPY_DMA,
                   host_staging=[hs.ptr + x for x in o] if hs else None,
                   host_staging_bytes=slot_bytes if hs else 0)
    for b in range(w.n_blocks):
        e.register_block_source(b, plan, srcs[b % w.distinct])
    cfg = dlo.dit_cfg(w.batch, w.tokens, w.hidden, w.heads, w.mlp, w.eps)
    nb = dlo.forward_scratch_bytes(cfg)
    scratch = torch.empty(nb, dtype=torch.uint8, device="cuda")
    x0 = W.gen_x(w, 9, device="cuda")
    x = x0.clone()
    torch.cuda.synchronize()
    e.prefetch(0, 0)
    with torch.cuda.stream(compute):
        for _ in range(w.steps):
            for b in range(w.n_blocks):
                e.block_forward(b, cfg, x, scratch, nb)
    torch.cuda.synchronize()
    rs = ResidentStack(host)
    xr = x0.clone()
    torch.cuda.synchronize()
    with torch.cuda.stream(rs.stream):
        for _ in range(w.steps):
            rs.step(xr)
    torch.cuda.synchronize()
    assert torch.equal(x, xr)
    st = e.query()
    if registered:
        assert st.n_direct_prefetches > 0 and st.n_packed_prefetches == 0
        dlo.host_unregister_ranges(ptrs, sizes)
    else:
        assert st.n_packed_prefetches > 0 and st.n_direct_prefetches == 0
        hs.close()
    e.destroy()
    host.close()


@pytest.mark.parametrize("transport,pages", [("registered", "huge"), ("registered", "base"),
                                             ("pageable", "huge")])
def test_source_stack_streams_like_resident(transport, pages):
    # the stack the bench runs for --source: a footprint above the
    # huge-page threshold, so the "huge" form copies the parameters into a
    # huge-page arena and registers that
    from layerwise_weight_offload_gb300.stack import SourceStack
    w = W.custom("srcstack", n_blocks=12, hidden=1024, heads=16, mlp=4096, tokens=128,
                 shards=1, steps=2, distinct=12)
    host = HostBlocks(w, seed=12, keep_params=True)
    st = SourceStack(host, transport=transport, pages=pages)
    # a second stack over the same sources (the bench builds two): base
    # pages are registered once and shared, a huge-page arena is its own
    SourceStack(host, transport=transport, pages=pages).close()
    if transport == "registered" and pages == "huge":
        assert st.arena is not None and st.arena.good_fraction() is not None
        assert st.srcs[3][0] != host.params[3]["norm1.weight"].data_ptr()
    x0 = W.gen_x(w, 12, device="cuda")
    x = x0.clone()
    st.compute.wait_stream(torch.cuda.current_stream())
    for _ in range(w.steps):
        st.step(x)
    torch.cuda.current_stream().wait_stream(st.compute)
    rs = ResidentStack(host)
    xr = x0.clone()
    rs.stream.wait_stream(torch.cuda.current_stream())
    for _ in range(w.steps):
        rs.step(xr)
    torch.cuda.current_stream().wait_stream(rs.stream)
    torch.cuda.synchronize()
    assert torch.equal(x, xr)
    q = st.engine.query()
    if transport == "registered":
        assert q.n_direct_prefetches > 0 and q.n_packed_prefetches == 0
    else:
        assert q.n_packed_prefetches > 0
    st.close()
    host.close()
