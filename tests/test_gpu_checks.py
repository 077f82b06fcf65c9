"""The engine's `checks` option on the GPU: every prefetch lists its copies
(DMA pieces, 2-D copy rows, copy-kernel segments, staged H2D and gather)
without issuing them, checks their offsets against the plan with
dlo_check_pieces, then issues them.  In every copy mode, for the odd-count
wrap and a one-block pass, the checks pass for every prefetch (one piece
per (group, shard) and phase), parameter views pass their own check, and
the streamed output equals the resident one bit for bit."""
import pytest
import torch

from tests._util import build_lib
from layerwise_weight_offload_gb300 import dlo, workloads as W
from layerwise_weight_offload_gb300.stack import HostBlocks, StreamedStack, ResidentStack

pytestmark = pytest.mark.gpu

MODES = [dlo.COPY_DMA, dlo.COPY_KERNEL, dlo.COPY_AUTO, dlo.COPY_STAGED]


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_lib()


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n_blocks,steps", [(9, 4), (1, 3)])
def test_checked_prefetches_stream_like_resident(n_blocks, steps, mode):
    w = W.custom("checks", n_blocks=n_blocks, hidden=256, heads=4, mlp=1024, tokens=96,
                 shards=3, steps=steps, distinct=min(n_blocks, 3))
    host = HostBlocks(w, seed=17)
    x0 = W.gen_x(w, seed=17)
    st = StreamedStack(host, copy_mode=mode, checks=True)
    xs = x0.clone().cuda()
    st.compute.wait_stream(torch.cuda.current_stream())
    for _ in range(steps):
        st.step(xs)
    torch.cuda.current_stream().wait_stream(st.compute)
    torch.cuda.synchronize()
    q = st.engine.query()
    per = len(host.groups) * w.shards * (2 if mode == dlo.COPY_STAGED else 1)
    assert q.n_prefetches == n_blocks * steps + 1
    assert q.checked_pieces == q.n_prefetches * per
    # block 0 is in a slot again (the last forward prefetched it)
    bases = [t.data_ptr() for t in st.slots]
    for p in range(len(host.descs)):
        off = st.plan.param(p).slot_offset
        assert st.engine.param_view(0, p) in (bases[0] + off, bases[1] + off)
    st.close()
    rs = ResidentStack(host)
    xr = x0.clone().cuda()
    rs.stream.wait_stream(torch.cuda.current_stream())
    for _ in range(steps):
        rs.step(xr)
    torch.cuda.current_stream().wait_stream(rs.stream)
    torch.cuda.synchronize()
    assert torch.equal(xs, xr)
    assert dlo.kernel_status() == 0
    host.close()


def test_checked_dma_fan_out_and_views():
    # DMA spread over several streams: one piece per (group, shard)
    w = W.custom("checks-fan", n_blocks=3, hidden=256, heads=4, mlp=1024, tokens=64,
                 shards=4, steps=2, distinct=3)
    host = HostBlocks(w, seed=19)
    slot_bytes = (host.plan.info().slot_bytes + 255) // 256 * 256
    slots = [torch.empty(slot_bytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
    comp, copy = torch.cuda.Stream(), torch.cuda.Stream()
    e = dlo.Engine(w.n_blocks, slots[0], slots[1], slot_bytes, comp, copy, dlo.COPY_DMA,
                   dma_streams=3, checks=True)
    for i in range(w.n_blocks):
        e.register_block(i, host.plan, host.shard_ptrs(i))
    e.prefetch(0, 0)
    e.wait_host(0, 10000)
    for p in range(len(host.descs)):
        ptr = e.param_view(0, p)
        assert ptr == slots[0].data_ptr() + host.plan.param(p).slot_offset
    assert e.query().checked_pieces == len(host.groups) * w.shards
    e.destroy()
    host.close()
