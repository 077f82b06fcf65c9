"""dlo_forward_noalloc: the block forward for callers that cannot allocate
device memory (serving loops that must not allocate once warm, device
memory owned by another allocator with a fixed budget).  It takes its
scratch from the library's static device array; its output must match
dlo_forward with a caller-provided scratch buffer, on two calls in a row
(the second call finds the first call's leftovers in the shared array)."""
import pytest
import torch

from tests._util import build_lib, assert_oracle_close
from layerwise_weight_offload_gb300 import dlo, workloads as W
from layerwise_weight_offload_gb300.stack import HostBlocks, ResidentStack

pytestmark = pytest.mark.gpu


def test_noalloc_forward_matches_forward_on_two_calls():
    build_lib()
    w = W.custom("noalloc", n_blocks=2, hidden=256, heads=4, mlp=1024, tokens=200, shards=3,
                 distinct=2)
    host = HostBlocks(w, seed=21)
    rs = ResidentStack(host)
    cfg = dlo.dit_cfg(w.batch, w.tokens, w.hidden, w.heads, w.mlp, w.eps, graph=False)
    nbytes = dlo.forward_scratch_bytes(cfg)
    assert 0 < nbytes <= 32 << 20
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    x = W.gen_x(w, seed=21, device="cuda")
    torch.cuda.synchronize()
    for call in range(2):                      # two calls in a row, different blocks
        buf = rs.bufs[call % w.distinct]
        x_ref, x_na = x.clone(), x.clone()
        torch.cuda.synchronize()
        dlo.forward(cfg, host.plan, buf, x_ref, scratch, nbytes, stream)
        dlo.forward_noalloc(cfg, host.plan, buf, x_na, stream)
        stream.synchronize()
        assert_oracle_close(x_na.cpu().numpy(), x_ref.cpu().numpy(), "call %d" % call)
        assert torch.equal(x_na, x_ref)
        x = x_ref
    assert dlo.kernel_status() == 0
    # a shape whose scratch exceeds the static array is refused, not run
    big = dlo.dit_cfg(1, 16384, 1024, 16, 4096)
    with pytest.raises(dlo.DLOError) as ei:
        dlo.forward_noalloc(big, host.plan, rs.bufs[0], x, stream)
    assert ei.value.status == dlo.ERR_NOMEM
    host.close()
