"""Fail-closed behaviour on the GPU, without faulting or hanging it ([B1]
"Fail-Closed Design"; [B2] "Validation Results": a partial wave that times
out fails closed; [D5] "Lease ownership": in-flight copies are drained
before a close):
- dlo_wait_host and dlo_engine_destroy give up after their host-side limit
  while a copy is held back (by a bounded GPU sleep on the copy stream),
  keep the engine intact, and succeed once the copy has landed;
- the kernels' bounded device waits give up on a phase nobody completes
  (limit shortened by the probe), record their code and leave the context
  usable;
- a one-block pass resolves dlo_wait / dlo_param_view to the slot the hook
  reads, not to the slot a copy is refilling;
- the schedule log and the timing record keep a bounded number of entries
  however many forwards run."""
import os
import time

import numpy as np
import pytest
import torch

from tests._util import build_lib
from layerwise_weight_offload_gb300 import dlo, workloads as W
from layerwise_weight_offload_gb300.stack import HostBlocks, StreamedStack

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_lib()


def _sleep_cycles(seconds):
    # torch.cuda._sleep spins for a number of SM clock cycles: take the
    # highest clock so the sleep lasts at least `seconds`
    return int(seconds * 2.2e9)


def test_wait_host_and_destroy_time_out_while_a_copy_is_held_back():
    w = W.custom("to", n_blocks=1, hidden=256, heads=4, mlp=1024, tokens=64, shards=2)
    host = HostBlocks(w, seed=2)
    st = StreamedStack(host, copy_mode=dlo.COPY_DMA)
    e = st.engine
    with torch.cuda.stream(st.copy):
        torch.cuda._sleep(_sleep_cycles(0.3))
    e.prefetch(0, 0)                    # queued behind the sleep
    t0 = time.perf_counter()
    with pytest.raises(dlo.DLOError) as ei:
        e.wait_host(0, 5)
    assert ei.value.status == dlo.ERR_TIMEOUT
    assert time.perf_counter() - t0 < 0.25
    e.wait_host(0, 10000)               # the copy lands: the same call succeeds
    # destroy while a copy is pending: times out, the engine stays usable
    with torch.cuda.stream(st.copy):
        torch.cuda._sleep(_sleep_cycles(0.3))
    st.engine = None
    st_handle = e.handle
    rc = dlo.lib().dlo_engine_destroy(st_handle, 5)
    assert rc == dlo.ERR_TIMEOUT
    slot = e.pre_forward(0)             # still a working engine
    e.post_forward(0)
    assert slot == 0
    e.destroy(10000)                    # drains, then releases
    torch.cuda.synchronize()
    host.close()


@pytest.mark.parametrize("spin", [0, 1])
def test_device_wait_gives_up_and_the_context_stays_usable(spin):
    limit = 50_000_000                  # 50 ms instead of the kernels' 4 s
    st, el, code = dlo.debug_wait_probe(spin, limit)
    assert st == dlo.ERR_TIMEOUT
    assert code == 7                    # timed out
    assert limit <= el < 2_000_000_000
    assert dlo.kernel_status() == 0     # the probe cleared the word
    # another role's abort flag ends the wait before its limit
    st, el, code = dlo.debug_wait_probe(spin, 1_000_000_000, abort_ns=20_000_000)
    assert st == dlo.ERR_TIMEOUT and code == 6
    assert 20_000_000 <= el < 1_000_000_000
    # the context still runs the library's kernels correctly
    x = torch.randn(37, 256, device="cuda")
    g = torch.ones(256, device="cuda")
    z = torch.zeros(256, device="cuda")
    h = torch.empty(37, 256, dtype=torch.bfloat16, device="cuda")
    dlo.op_rmsnorm_mod(x, 37, 256, g, z, z, 1e-6, h, None)
    torch.cuda.synchronize()
    ref = x / torch.sqrt((x * x).mean(dim=1, keepdim=True) + 1e-6)
    assert torch.allclose(h.float(), ref, atol=2e-2, rtol=1e-2)
    assert dlo.kernel_status() == 0
    with pytest.raises(dlo.DLOError):
        dlo._check(dlo.lib().dlo_debug_wait_probe(0, 3_000_000_000, 0, None, None), "probe")


def test_one_block_pass_resolves_views_to_the_hook_slot():
    w = W.custom("one", n_blocks=1, hidden=256, heads=4, mlp=1024, tokens=64, shards=2,
                 steps=4)
    host = HostBlocks(w, seed=3)
    st = StreamedStack(host, copy_mode=dlo.COPY_DMA)
    e = st.engine
    st.prime()
    off = host.plan.param(4).slot_offset
    for k in range(6):
        slot = e.pre_forward(0)
        assert slot == k % 2
        # both slots hold block 0 now (the hook refills the other one): the
        # forward's views and waits resolve to the slot it reads
        assert e.param_view(0, 4) == st.slots[slot].data_ptr() + off
        e.wait(0)
        e.post_forward(0)
        # between forwards: the newer copy, which the next forward reads
        assert e.param_view(0, 4) == st.slots[1 - slot].data_ptr() + off
    torch.cuda.synchronize()
    st.close()
    host.close()


def test_log_and_timing_records_are_bounded_rings():
    w = W.custom("ring", n_blocks=3, hidden=256, heads=4, mlp=1024, tokens=64, shards=2)
    host = HostBlocks(w, seed=4)
    cap = 64
    st = StreamedStack(host, copy_mode=dlo.COPY_DMA, timing=True, log_capacity=cap)
    e = st.engine
    st.prime()
    n = 1000
    for k in range(n):
        e.pre_forward(k % 3)
        e.post_forward(k % 3)
    torch.cuda.synchronize()
    log = e.schedule_log()
    assert len(log) == cap
    assert [ev[0] for ev in log] == list(range(n - cap, n))   # the newest, oldest first
    for ev in log:
        assert ev[1] == ev[0] % 3 and ev[2] == ev[0] % 2
    stats = e.query()
    assert stats.log_dropped == n - cap
    assert stats.timed_dropped == n + 1 - cap                  # + the setup prefetch
    ms, by = e.copy_times()
    assert len(ms) == cap and all(v > 0 for v in ms)
    spans = e.copy_spans()
    assert len(spans) == cap
    assert spans[0][0] == 0.0 and all(b >= a for a, b in spans)
    st.close()
    host.close()


def _rss_bytes():
    with open("/proc/self/statm") as fh:
        return int(fh.read().split()[1]) * os.sysconf("SC_PAGE_SIZE")


def test_a_million_forwards_hold_constant_host_memory():
    # hooks only (the caller's forward is empty), on a 4 KB block: the
    # schedule log must stop growing at its capacity
    descs = [("v", (1024,), W.F32)]
    plan = dlo.Plan(descs, 1)
    src = torch.arange(1024, dtype=torch.float32).pin_memory()
    shard = torch.empty(plan.groups()[0].shard_alloc_bytes, dtype=torch.uint8).pin_memory()
    plan.shard_host([src.data_ptr()], [shard.data_ptr()])
    slots = [torch.empty(4096, dtype=torch.uint8, device="cuda") for _ in range(2)]
    comp, copy = torch.cuda.Stream(), torch.cuda.Stream()
    e = dlo.Engine(2, slots[0], slots[1], 4096, comp, copy, dlo.COPY_DMA, log_capacity=1024)
    for b in range(2):
        e.register_block(b, plan, [shard.data_ptr()])
    e.prefetch(0, 0)
    n, warm = 1_000_000, 20_000
    rss0 = None
    for k in range(n):
        e.pre_forward(k & 1)
        e.post_forward(k & 1)
        if k == warm:
            torch.cuda.synchronize()
            rss0 = _rss_bytes()
    torch.cuda.synchronize()
    grown = _rss_bytes() - rss0
    # an unbounded log would have grown by 28 bytes x 980,000 entries (27 MB)
    assert grown < 8 << 20, grown
    stats = e.query()
    assert stats.n_forwards == n and stats.log_dropped == n - 1024
    assert len(e.schedule_log()) == 1024
    got = slots[0][:4096].view(torch.float32).cpu()
    assert torch.equal(got, src)
    e.destroy()
