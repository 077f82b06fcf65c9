"""The streamed stack on the GPU against the oracle:
- the engine's slot/event schedule equals the oracle's literal hook
  simulation, entry for entry;
- at every forward the slot the compute stream reads holds exactly the
  oracle's reassembled image of that block (the stream's read-after-write
  and write-after-read ordering);
- the streamed forward is bit-identical to the all-resident forward;
- the block forward matches the oracle within the acceptance bar, step by
  step (teacher-forced: the oracle's input at step s is the GPU's output of
  step s-1)."""
import numpy as np
import pytest
import torch

import oracle
from tests._util import (build_lib, raw_bytes, params_f32, assert_oracle_close,
                         assert_only_groups_written)
from layerwise_weight_offload_gb300 import dlo, workloads as W
from layerwise_weight_offload_gb300.stack import HostBlocks, StreamedStack, ResidentStack

pytestmark = pytest.mark.gpu

MODES = [dlo.COPY_DMA, dlo.COPY_KERNEL, dlo.COPY_AUTO, dlo.COPY_STAGED]


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_lib()


def _slot_image(host, hb):
    p = host.params[hb]
    numels = [int(np.prod(sh)) for _, sh, _ in host.descs]
    codes = [c for _, _, c in host.descs]
    esizes = [W.ESIZE[c] for c in codes]
    raw = [raw_bytes(p[name]) for name, _, _ in host.descs]
    image, _, _, _ = oracle.slot_image(raw, numels, codes, esizes, host.w.shards, 256)
    return image


def _small(name, **kw):
    base = W.CONFIGS[name].__dict__.copy()
    base.update(kw)
    return W.Workload(**base)


@pytest.mark.parametrize("two_streams", [False, True])
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n_blocks,steps", [(1, 3), (2, 2), (3, 2), (9, 3), (8, 1)])
def test_schedule_and_slot_contents(n_blocks, steps, mode, two_streams):
    # small blocks so that every slot can be snapshotted; with two_streams
    # slot 1's prefetches run on a second copy stream
    w = W.custom("sched", n_blocks=n_blocks, hidden=256, heads=4, mlp=1024, tokens=64,
                 shards=3, steps=steps, distinct=min(n_blocks, 3))
    host = HostBlocks(w, seed=5, keep_params=True)
    st = StreamedStack(host, copy_mode=mode, two_copy_streams=two_streams)
    images = [_slot_image(host, hb) for hb in range(w.distinct)]
    for sl in st.slots:
        sl.fill_(0xA5)                         # canary: prefetches write only the groups
    torch.cuda.synchronize()
    st.prime()
    snaps = []
    groups = host.plan.groups()
    for k in range(n_blocks * steps):
        i = k % n_blocks
        slot = st.engine.pre_forward(i)
        snap = torch.empty_like(st.slots[slot])
        with torch.cuda.stream(st.compute):
            snap.copy_(st.slots[slot])        # read on the compute stream, like a forward
        snaps.append((i, snap))
        st.engine.post_forward(i)
    torch.cuda.synchronize()
    log = st.engine.schedule_log()
    ref = oracle.schedule(n_blocks, steps)
    assert [tuple(e[:6]) for e in log] == [tuple(int(v) for v in r[:6]) for r in ref]
    for i, snap in snaps:
        got = snap.cpu().numpy()
        exp = images[i % w.distinct]
        for g in groups:
            n = w.shards * g.shard_bytes
            assert np.array_equal(got[g.base:g.base + n], exp[g.base:g.base + n]), (i, g.dtype)
        assert_only_groups_written(got, groups, w.shards, 0xA5, i)
    stats = st.engine.query()
    assert stats.n_forwards == n_blocks * steps
    assert stats.n_prefetches == n_blocks * steps + 1
    st.close()
    host.close()


def test_fail_closed_states():
    w = W.custom("fc", n_blocks=3, hidden=256, heads=4, mlp=1024, tokens=64, shards=2)
    host = HostBlocks(w, seed=1)
    st = StreamedStack(host, copy_mode=dlo.COPY_DMA)
    e = st.engine
    with pytest.raises(dlo.DLOError) as ei:
        e.pre_forward(0)                       # nothing prefetched yet
    assert ei.value.status == dlo.ERR_STATE
    with pytest.raises(dlo.DLOError):
        e.param_view(0, 0)                     # not resident
    st.prime()
    with pytest.raises(dlo.DLOError) as ei:
        e.pre_forward(1)                       # out of order
    assert ei.value.status == dlo.ERR_STATE
    slot = e.pre_forward(0)
    with pytest.raises(dlo.DLOError):
        e.prefetch(2, slot)                    # slot being read
    with pytest.raises(dlo.DLOError):
        e.pre_forward(1)                       # post_forward missing
    with pytest.raises(dlo.DLOError):
        e.register_block(0, host.plan, host.shard_ptrs(0))   # twice
    v = e.param_view(0, 4)
    assert v == st.slots[slot].data_ptr() + host.plan.param(4).slot_offset
    e.post_forward(0)
    e.wait_host(1, 10000)
    torch.cuda.synchronize()
    st.close()
    host.close()


def test_register_rejects_pageable_and_oversized():
    w = W.custom("rj", n_blocks=2, hidden=256, heads=4, mlp=1024, tokens=64, shards=2)
    host = HostBlocks(w, seed=1)
    st = StreamedStack(host, copy_mode=dlo.COPY_KERNEL)
    pageable = [torch.empty(g.shard_alloc_bytes, dtype=torch.uint8) for g in host.plan.groups()
                for _ in range(w.shards)]
    e2 = dlo.Engine(2, st.slots[0], st.slots[1], st.slot_bytes, st.compute, st.copy,
                    dlo.COPY_KERNEL)
    with pytest.raises(dlo.DLOError) as ei:
        e2.register_block(0, host.plan, [t.data_ptr() for t in pageable])
    assert ei.value.status == dlo.ERR_INVALID
    e3 = dlo.Engine(2, st.slots[0], st.slots[1], 1024, st.compute, st.copy, dlo.COPY_DMA)
    with pytest.raises(dlo.DLOError):
        e3.register_block(0, host.plan, host.shard_ptrs(0))
    e2.destroy()
    e3.destroy()
    st.close()
    host.close()


def _run_streamed(host, x0, steps, mode):
    st = StreamedStack(host, copy_mode=mode)
    x = x0.clone().cuda()
    outs = []
    for _ in range(steps):
        st.compute.wait_stream(torch.cuda.current_stream())
        st.step(x)
        torch.cuda.current_stream().wait_stream(st.compute)
        outs.append(x.clone())
    torch.cuda.synchronize()
    st.close()
    return outs


def _run_resident(host, x0, steps):
    rs = ResidentStack(host)
    x = x0.clone().cuda()
    outs = []
    per_block = []
    for _ in range(steps):
        rs.stream.wait_stream(torch.cuda.current_stream())
        for i in range(host.w.n_blocks):
            xin = x.clone()
            rs.block(i, x)
            torch.cuda.current_stream().wait_stream(rs.stream)
            per_block.append((i, xin, x.clone()))
        outs.append(x.clone())
    torch.cuda.synchronize()
    return outs, per_block


def _check_against_oracle(host, per_block, which):
    w = host.w
    for idx in which:
        i, xin, xout = per_block[idx]
        p = params_f32(host.params[i % w.distinct])
        xin_np = xin.cpu().numpy()
        ref = oracle.block_forward(xin_np, p, w.batch, w.tokens, w.hidden, w.heads, w.mlp, w.eps,
                                   rope_base=W.oracle_rope_base(w))
        got = xout.cpu().numpy()
        assert_oracle_close(got, ref, "block %d output" % idx)
        # the branch updates alone, which the residual would otherwise mask
        assert_oracle_close(got - xin_np, ref - xin_np, "block %d update" % idx, 2e-2, 1e-2)


@pytest.mark.parametrize("mode", MODES)
def test_tiny_streamed_vs_resident_vs_oracle(mode):
    w = W.CONFIGS["tiny"]
    host = HostBlocks(w, seed=0, keep_params=True)
    x0 = W.gen_x(w, seed=0)
    res, per_block = _run_resident(host, x0, w.steps)
    stm = _run_streamed(host, x0, w.steps, mode)
    for a, b in zip(res, stm):
        assert torch.equal(a, b)            # bit-identical
    _check_against_oracle(host, per_block, range(len(per_block)))
    assert dlo.kernel_status() == 0
    host.close()


def test_odd_streamed_vs_resident_vs_oracle():
    w = W.CONFIGS["odd"]
    host = HostBlocks(w, seed=0, keep_params=True)
    x0 = W.gen_x(w, seed=0)
    res, per_block = _run_resident(host, x0, w.steps)
    for mode in (dlo.COPY_AUTO, dlo.COPY_KERNEL):
        stm = _run_streamed(host, x0, w.steps, mode)
        for a, b in zip(res, stm):
            assert torch.equal(a, b)
    n = w.n_blocks
    # sampled, teacher-forced: blocks 0, 1, n-1 of step 0, block 0 of the last step
    _check_against_oracle(host, per_block, [0, 1, n - 1, (w.steps - 1) * n])
    assert dlo.kernel_status() == 0
    host.close()


def test_odd_full_streamed_vs_resident_vs_oracle():
    # the checkpoint-shaped block at the odd workload's shape (biases, q/k
    # norm, rotary embedding; 9 blocks, 3 misaligned shards, head dim 64)
    w = W.CONFIGS["odd-full"]
    host = HostBlocks(w, seed=0, keep_params=True)
    x0 = W.gen_x(w, seed=0)
    res, per_block = _run_resident(host, x0, w.steps)
    for mode in (dlo.COPY_AUTO, dlo.COPY_KERNEL):
        stm = _run_streamed(host, x0, w.steps, mode)
        for a, b in zip(res, stm):
            assert torch.equal(a, b)
    n = w.n_blocks
    _check_against_oracle(host, per_block, [0, 1, n - 1, (w.steps - 1) * n])
    assert dlo.kernel_status() == 0
    host.close()


@pytest.mark.parametrize("cfg", [
    dict(n_blocks=3, hidden=320, heads=5, mlp=1280, tokens=200, shards=3),   # ragged tiles
    dict(n_blocks=2, hidden=256, heads=2, mlp=1024, tokens=1, shards=2),     # one token
    dict(n_blocks=3, hidden=384, heads=3, mlp=1536, tokens=77, shards=5, batch=2),
])
def test_ragged_streamed_vs_resident_vs_oracle(cfg):
    w = W.custom("ragged", steps=2, **cfg)
    host = HostBlocks(w, seed=9, keep_params=True)
    x0 = W.gen_x(w, seed=9)
    res, per_block = _run_resident(host, x0, w.steps)
    stm = _run_streamed(host, x0, w.steps, dlo.COPY_AUTO)
    for a, b in zip(res, stm):
        assert torch.equal(a, b)
    _check_against_oracle(host, per_block, range(len(per_block)))
    host.close()


@pytest.mark.parametrize("mode", [dlo.COPY_DMA, dlo.COPY_KERNEL, dlo.COPY_STAGED])
@pytest.mark.parametrize("cfg", [
    dict(name="tiny-full"),
    dict(name="ragged-full", n_blocks=3, hidden=384, heads=3, mlp=1536, tokens=77, shards=5,
         batch=2),
    dict(name="hd64-full", n_blocks=2, hidden=512, heads=8, mlp=2048, tokens=300, shards=3),
])
def test_checkpoint_shaped_block_streamed_vs_resident_vs_oracle(cfg, mode):
    # biases on the four linears, per-head q/k RMSNorm, rotary embedding
    # (positions restart in the second batch item): streamed equals resident
    # bit for bit, both match the oracle's block with the same additions
    if cfg["name"] == "tiny-full":
        w = W.CONFIGS["tiny-full"]
    else:
        kw = dict(cfg)
        name = kw.pop("name")
        w = W.custom(name, steps=2, variant="full", **kw)
    host = HostBlocks(w, seed=13, keep_params=True)
    x0 = W.gen_x(w, seed=13)
    res, per_block = _run_resident(host, x0, w.steps)
    stm = _run_streamed(host, x0, w.steps, mode)
    for a, b in zip(res, stm):
        assert torch.equal(a, b)
    _check_against_oracle(host, per_block, range(len(per_block)))
    assert dlo.kernel_status() == 0
    host.close()


def test_forward_with_split_tails_vs_oracle():
    # tokens chosen so that the QKV linear's tiles (6 column blocks at
    # d = 512) leave a short last wave on this GPU: that tail runs as K slices
    # with the transposed-V epilogue in the reduction; the out-projection and
    # fc2 have fewer tiles than SMs and split every tile (all on the
    # single-CTA kernel: by shape the QKV linear would run on CTA pairs)
    dlo.set_gemm_pair_mode(dlo.GEMM_PAIR_OFF)
    try:
        _forward_with_split_tails_vs_oracle()
    finally:
        dlo.set_gemm_pair_mode(dlo.GEMM_PAIR_AUTO)


def _forward_with_split_tails_vs_oracle():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    num_m = -(-(sms + 1) // 6)
    assert 1 <= 6 * num_m - sms <= sms // 2
    w = W.custom("tails", n_blocks=1, hidden=512, heads=4, mlp=2048, tokens=128 * num_m - 28,
                 shards=2, steps=1)
    cfg = dlo.dit_cfg(w.batch, w.tokens, w.hidden, w.heads, w.mlp)
    assert dlo.forward_launches(cfg) == 11
    host = HostBlocks(w, seed=3, keep_params=True)
    x0 = W.gen_x(w, seed=3)
    res, per_block = _run_resident(host, x0, w.steps)
    _check_against_oracle(host, per_block, [0])
    assert dlo.kernel_status() == 0
    host.close()


def _forward_outputs(rs, w, x0, cfgs):
    # one x buffer (so a graph call with the same configuration replays the
    # cached graph), reset before each call; the outputs are copied out
    x = x0.clone()
    outs = []
    for cfg in cfgs:
        rs.cfg = cfg
        x.copy_(x0)
        rs.stream.wait_stream(torch.cuda.current_stream())
        rs.step(x)
        torch.cuda.current_stream().wait_stream(rs.stream)
        outs.append(x.clone())
    torch.cuda.synchronize()
    return outs


def test_graph_replay_equals_direct_launches():
    w = W.custom("graph", n_blocks=2, hidden=256, heads=4, mlp=1024, tokens=130, shards=2)
    host = HostBlocks(w, seed=4)
    rs = ResidentStack(host)
    x0 = W.gen_x(w, seed=4, device="cuda")
    cfg = lambda graph: dlo.dit_cfg(w.batch, w.tokens, w.hidden, w.heads, w.mlp, w.eps,
                                    graph=graph)
    # direct launches, a captured graph, then its replay
    outs = _forward_outputs(rs, w, x0, [cfg(False), cfg(True), cfg(True)])
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    host.close()


def test_graph_cache_keys_on_the_block_variant_flags():
    # the checkpoint-shaped block on the same plan, weights, x and scratch with
    # and without rotary embedding: each flag set gets its own graph (a graph
    # keyed without the flags would replay the other's launches)
    w = W.custom("graphfull", n_blocks=1, hidden=256, heads=4, mlp=1024, tokens=96, shards=2,
                 variant="full")
    host = HostBlocks(w, seed=6)
    rs = ResidentStack(host)
    x0 = W.gen_x(w, seed=6, device="cuda")
    cfg = lambda graph, rope: dlo.dit_cfg(w.batch, w.tokens, w.hidden, w.heads, w.mlp, w.eps,
                                          graph=graph, rope=rope, qk_norm=True)
    outs = _forward_outputs(rs, w, x0, [cfg(False, True), cfg(False, False), cfg(True, True),
                                        cfg(True, False), cfg(True, True), cfg(True, False)])
    assert torch.equal(outs[0], outs[2]) and torch.equal(outs[2], outs[4])
    assert torch.equal(outs[1], outs[3]) and torch.equal(outs[3], outs[5])
    assert not torch.equal(outs[0], outs[1])
    host.close()


@pytest.mark.parametrize("dma_streams", [1, 2, 8])
def test_dma_fan_out_bytes(dma_streams):
    w = W.custom("fan", n_blocks=3, hidden=256, heads=4, mlp=1024, tokens=64, shards=5,
                 distinct=3)
    host = HostBlocks(w, seed=2, keep_params=True)
    st = StreamedStack(host, copy_mode=dlo.COPY_DMA)
    st.engine.destroy()
    st.engine = dlo.Engine(w.n_blocks, st.slots[0], st.slots[1], st.slot_bytes, st.compute,
                           st.copy, dlo.COPY_DMA, 0, False, dma_streams)
    for i in range(w.n_blocks):
        st.engine.register_block(i, host.plan, host.shard_ptrs(i))
    st.prime()
    for k in range(2 * w.n_blocks):
        i = k % w.n_blocks
        slot = st.engine.pre_forward(i)
        snap = torch.empty_like(st.slots[slot])
        with torch.cuda.stream(st.compute):
            snap.copy_(st.slots[slot])
        st.engine.post_forward(i)
        torch.cuda.synchronize()
        exp = _slot_image(host, i)
        got = snap.cpu().numpy()
        for g in host.plan.groups():
            n = w.shards * g.shard_bytes
            assert np.array_equal(got[g.base:g.base + n], exp[g.base:g.base + n])
    st.close()
    host.close()


def test_auto_races_on_forward_time():
    w = W.custom("race", n_blocks=5, hidden=512, heads=4, mlp=2048, tokens=256, shards=2,
                 steps=7, distinct=5)
    host = HostBlocks(w, seed=3)
    st = StreamedStack(host, copy_mode=dlo.COPY_AUTO)
    x = W.gen_x(w, seed=3, device="cuda")
    st.compute.wait_stream(torch.cuda.current_stream())
    for _ in range(w.steps):
        st.step(x)
    torch.cuda.synchronize()
    s = st.engine.query()
    assert s.race_dma_us > 0 and s.race_kernel_us > 0
    assert s.chosen_mode in (dlo.COPY_DMA, dlo.COPY_KERNEL)
    assert s.chosen_mode == (dlo.COPY_KERNEL if s.race_kernel_us < s.race_dma_us
                             else dlo.COPY_DMA)
    modes = [e[6] for e in st.engine.schedule_log()]
    s0 = w.n_blocks + 2
    for win in range(4):
        want = dlo.COPY_KERNEL if win % 2 else dlo.COPY_DMA
        assert modes[s0 + 6 * win:s0 + 6 * win + 6] == [want] * 6
    assert s.n_kernel_prefetches >= 12
    st.close()
    host.close()


@pytest.mark.parametrize("two_streams", [False, True])
def test_copy_spans(two_streams):
    # the spans sit on one clock: per slot they follow one another, each
    # lasts what copy_times says, and their union is no longer than the sum
    w = W.custom("spans", n_blocks=4, hidden=512, heads=4, mlp=2048, tokens=64, shards=2,
                 steps=3)
    host = HostBlocks(w, seed=2)
    st = StreamedStack(host, copy_mode=dlo.COPY_DMA, timing=True, two_copy_streams=two_streams)
    x = W.gen_x(w, seed=2, device="cuda")
    torch.cuda.synchronize()
    for _ in range(w.steps):
        st.step(x)
    torch.cuda.synchronize()
    ms, _ = st.engine.copy_times()
    spans = st.engine.copy_spans()
    assert len(spans) == len(ms) == w.n_blocks * w.steps + 1
    assert spans[0][0] == 0.0
    for (s, e), d in zip(spans, ms):
        assert e >= s and abs((e - s) - d) <= 1e-3 + 1e-3 * d
    for slot in (0, 1):
        mine = spans[slot::2]                 # prefetch k fills slot k % 2
        for (s0, e0), (s1, e1) in zip(mine, mine[1:]):
            assert s1 >= e0 - 1e-3
    if not two_streams:
        for (s0, e0), (s1, e1) in zip(spans, spans[1:]):
            assert s1 >= e0 - 1e-3
    st.close()
    host.close()


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n_blocks,steps", [(1, 3), (9, 3)])
def test_poisoned_slots_stream_like_resident(n_blocks, steps, mode):
    # with every slot overwritten by 0xA5 right after the forward that read
    # it, a forward that read a released or not-yet-refilled slot would see
    # garbage: the streamed output must still equal the resident one bit for
    # bit (one block: both slots hold it; nine: the odd-count wrap)
    w = W.custom("poison", n_blocks=n_blocks, hidden=256, heads=4, mlp=1024, tokens=96,
                 shards=3, steps=steps, distinct=min(n_blocks, 3))
    host = HostBlocks(w, seed=13)
    x0 = W.gen_x(w, seed=13)
    st = StreamedStack(host, copy_mode=mode, poison=True)
    xs = x0.clone().cuda()
    st.compute.wait_stream(torch.cuda.current_stream())
    for _ in range(steps):
        st.step(xs)
    torch.cuda.current_stream().wait_stream(st.compute)
    torch.cuda.synchronize()
    # the last slot read now holds the poison
    last = (n_blocks * steps - 1) % 2
    assert (st.slots[last][:st.plan.info().slot_bytes] == 0xA5).all()
    st.close()
    rs = ResidentStack(host)
    xr = x0.clone().cuda()
    rs.stream.wait_stream(torch.cuda.current_stream())
    for _ in range(steps):
        rs.step(xr)
    torch.cuda.current_stream().wait_stream(rs.stream)
    torch.cuda.synchronize()
    assert torch.isfinite(xs).all()
    assert torch.equal(xs, xr)
    host.close()
