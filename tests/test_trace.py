"""The library's NVTX ranges, seen by a recording NVTX tool (tests/nvtx_probe.c,
attached through NVTX_INJECTION64_PATH in a fresh process).

CPU: the plan and host-shard calls each emit one range in the "dlo" domain
with the number of parameters as payload, closed before they return (also
when they fail).  GPU: a streamed pass emits, per forward, block_forward ⊃
pre_forward ⊃ the prefetch of the next block into the slot the schedule log
names, then forward (rows as payload) and post_forward; explicit prefetches,
host waits and the engine's teardown emit their own ranges."""
import pytest

from tests._nvtx import build_probe, run_traced, ranges
from tests._util import build_lib


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    build_lib()
    return build_probe(tmp_path_factory.mktemp("nvtx"))


CPU_SNIPPET = r"""
import numpy as np
from layerwise_weight_offload_gb300 import dlo
descs = [("a", (3, 5), dlo.BF16), ("b", (7,), dlo.F32), ("c", (4, 2), dlo.BF16)]
plan = dlo.Plan(descs, 3)
raw = [np.arange(15 * 2, dtype=np.uint8), np.arange(7 * 4, dtype=np.uint8),
       np.arange(8 * 2, dtype=np.uint8)]
shards = [np.zeros(g.shard_alloc_bytes, np.uint8) for g in plan.groups() for _ in range(3)]
plan.shard_host([r.ctypes.data for r in raw], [s.ctypes.data for s in shards])
failed = False
try:
    dlo.Plan([("bad", (2,), 99)], 1)
except dlo.DLOError:
    failed = True
result = {"failed": failed, "groups": len(plan.groups())}
"""


def test_cpu_calls_emit_ranges(probe):
    result, rec = run_traced(CPU_SNIPPET, probe, timeout=300)
    assert result["failed"] and result["groups"] == 2
    assert rec["inits"] >= 1 and rec["dropped"] == 0
    got = [(n, p, d) for n, p, d, _ in ranges(rec["events"])]
    # two plans (the second fails its dtype check inside the range)
    assert got == [("plan_create", 3, 0), ("shard_host", 3, 0), ("plan_create", 1, 0)], got


GPU_SNIPPET = r"""
import torch
from layerwise_weight_offload_gb300 import dlo, workloads as W
from layerwise_weight_offload_gb300.stack import HostBlocks, StreamedStack
w = W.custom("trace", n_blocks=3, hidden=256, heads=4, mlp=1024, tokens=64, shards=2,
             distinct=3)
host = HostBlocks(w, seed=5)
st = StreamedStack(host, copy_mode=dlo.COPY_DMA)
x = W.gen_x(w, seed=5, device="cuda")
torch.cuda.synchronize()
for _ in range(2):
    st.step(x)
torch.cuda.synchronize()
log = [list(e[:5]) for e in st.engine.schedule_log()]   # k, block, read, prefetch block/slot
st.engine.wait_host(0, 10000)
st.close()
host.close()
result = {"log": log, "rows": w.batch * w.tokens, "n": w.n_blocks}
"""


@pytest.mark.gpu
def test_streamed_pass_emits_hook_ranges(probe):
    result, rec = run_traced(GPU_SNIPPET, probe)
    assert rec["dropped"] == 0
    got = ranges(rec["events"])
    threads = {t for _, _, _, t in got}
    assert len(threads) == 1, "hooks ran on one thread"
    got = [(n, p, d) for n, p, d, _ in got]
    log, rows, n = result["log"], result["rows"], result["n"]
    assert len(log) == 2 * n
    # the first fill: an explicit prefetch of block 0 into slot 0 before the first forward
    i = got.index(("block_forward", 0, 0))
    assert ("prefetch slot 0", 0, 0) in got[:i]
    fwd = got[i:]
    expect = []
    for k, block, read_slot, pb, ps in log:
        expect += [("block_forward", block, 0), ("pre_forward", block, 1),
                   ("prefetch slot %d" % ps, pb, 2), ("forward", rows, 1),
                   ("post_forward", block, 1)]
    assert fwd[:len(expect)] == expect, (fwd[:len(expect)], expect)
    tail = fwd[len(expect):]
    assert ("wait_host", 0, 0) in tail and ("engine_destroy", n, 0) in tail, tail
