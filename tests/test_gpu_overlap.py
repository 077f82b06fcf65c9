"""Launch overlap (programmatic dependent launch) of the block forward's
kernels changes when CTAs are scheduled, never what they compute: the
forward with overlap on equals the forward with it off bit for bit, as a
direct launch sequence and as the cached CUDA graph, at shapes that run the
one-CTA GEMM with K slices, the CTA-pair GEMM with split tails, attention
with KV slices and the checkpoint-shaped extras."""
import pytest
import torch

from tests._util import build_lib
from layerwise_weight_offload_gb300 import dlo, workloads as W
from layerwise_weight_offload_gb300.stack import HostBlocks, ResidentStack

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [
    dict(hidden=1024, heads=16, mlp=4096, tokens=1024),            # one-CTA GEMMs, K slices
    dict(hidden=1664, heads=13, mlp=6656, tokens=4096),            # pairs, split tails
    dict(hidden=512, heads=4, mlp=2048, tokens=777, variant="full"),  # ragged, q/k norm, RoPE
])
@pytest.mark.parametrize("graph", [True, False])
def test_overlap_on_equals_off(shape, graph):
    build_lib()
    w = W.custom("ovl", n_blocks=2, shards=2, distinct=2, **shape)
    host = HostBlocks(w, seed=31)
    rs = ResidentStack(host)
    cfg = dlo.dit_cfg(w.batch, w.tokens, w.hidden, w.heads, w.mlp, w.eps, graph=graph,
                      **W.cfg_flags(w))
    rs.cfg = cfg
    x0 = W.gen_x(w, seed=31, device="cuda")
    out = {}
    try:
        for on in (False, True, False, True):
            dlo.set_launch_overlap(on)
            x = x0.clone()
            torch.cuda.synchronize()
            rs.stream.wait_stream(torch.cuda.current_stream())
            rs.step(x)
            torch.cuda.current_stream().wait_stream(rs.stream)
            torch.cuda.synchronize()
            out.setdefault(on, []).append(x)
    finally:
        dlo.set_launch_overlap(-1)
    assert torch.equal(out[True][0], out[False][0])
    assert torch.equal(out[True][1], out[True][0]) and torch.equal(out[False][1], out[False][0])
    assert dlo.kernel_status() == 0
    host.close()
