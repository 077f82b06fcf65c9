"""Full-size checks at the shapes of the Nano workload (hidden 3840, 30
heads, MLP 15360, 4096 tokens, 4 shards), its checkpoint-shaped variant
(biases, per-head q/k RMSNorm, rotary embedding), the Super workload
(hidden 6144, 48 heads, MLP 24576, 8192 tokens, 2 shards) and the
longest-sequence sweep cell (hidden 1664, 13 heads, MLP 6656, 16384 tokens,
2 shards), in the
launch configuration bench.py times (two-slot engine, AUTO copy mode,
CUDA-graph forwards):
- every prefetched slot equals the oracle's reassembled block, byte for byte;
- the streamed output equals the all-resident output bit for bit;
- sampled output rows match the oracle's block forward for those rows.
Two distinct host blocks and three block forwards stand in for each
workload's full count (the per-block work and the launch shapes are the
workload's; only the number of blocks is smaller, to keep host memory and
run time small)."""
import numpy as np
import pytest
import torch

import oracle
from tests._util import build_lib, raw_bytes, params_f32, assert_oracle_close
from layerwise_weight_offload_gb300 import dlo, workloads as W
from layerwise_weight_offload_gb300.stack import HostBlocks, StreamedStack, ResidentStack

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,rows", [
    ("nano", [0, 1, 777, 2048, 4095]),
    ("nano-full", [0, 1, 1234, 3000, 4095]),
    ("super", [0, 1, 3333, 4096, 8191]),
    ("sweep-d1664-t16384-s2", [0, 1, 5000, 12345, 16383]),
])
def test_full_shapes_streamed_resident_and_sampled_oracle(name, rows):
    build_lib()
    base = W.CONFIGS[name]
    w = W.Workload(**{**base.__dict__, "n_blocks": 3, "distinct": 2, "steps": 2})
    host = HostBlocks(w, seed=0, gen_device="cuda", keep_params=True)
    # bytes: one-shot reassembly of each host block against the oracle image
    numels = [int(np.prod(sh)) for _, sh, _ in host.descs]
    codes = [c for _, _, c in host.descs]
    esizes = [W.ESIZE[c] for c in codes]
    slot = torch.empty(host.plan.info().slot_bytes, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    for hb in range(w.distinct):
        raw = [raw_bytes(host.params[hb][name]) for name, _, _ in host.descs]
        image, _, gbase, _ = oracle.slot_image(raw, numels, codes, esizes, w.shards, 256)
        for mode in (dlo.COPY_DMA, dlo.COPY_KERNEL):
            slot.fill_(0)
            dlo.reassemble(host.plan, host.shard_ptrs(hb), slot, mode, s)
            s.synchronize()
            got = slot.cpu().numpy()
            for g in host.plan.groups():
                n = w.shards * g.shard_bytes
                assert np.array_equal(got[g.base:g.base + n], image[g.base:g.base + n])
    del slot
    # streamed vs resident, two steps
    x0 = W.gen_x(w, seed=0)
    st = StreamedStack(host, copy_mode=dlo.COPY_AUTO)
    xs = x0.clone().cuda()
    st.compute.wait_stream(torch.cuda.current_stream())
    for _ in range(w.steps):
        st.step(xs)
    torch.cuda.current_stream().wait_stream(st.compute)
    rs = ResidentStack(host)
    xr = x0.clone().cuda()
    x_in_block0 = xr.clone()
    rs.stream.wait_stream(torch.cuda.current_stream())
    rs.block(0, xr)
    torch.cuda.current_stream().wait_stream(rs.stream)
    x_out_block0 = xr.clone()
    rs.stream.wait_stream(torch.cuda.current_stream())
    for i in range(1, w.n_blocks):
        rs.block(i, xr)
    for _ in range(w.steps - 1):
        rs.step(xr)
    torch.cuda.current_stream().wait_stream(rs.stream)
    torch.cuda.synchronize()
    assert torch.equal(xs, xr)
    assert dlo.kernel_status() == 0
    st.close()
    # sampled rows of block 0 against the oracle (K and V over all tokens)
    p = params_f32(host.params[0])
    ref = oracle.block_forward_rows(x_in_block0.cpu().numpy(), p, rows, w.batch, w.tokens,
                                    w.hidden, w.heads, w.mlp, w.eps,
                                    rope_base=W.oracle_rope_base(w))
    got = x_out_block0.cpu().numpy()[rows]
    assert_oracle_close(got, ref, name + " rows")
    xin = x_in_block0.cpu().numpy()[rows]
    assert_oracle_close(got - xin, ref - xin, name + " row updates", 2e-2, 1e-2)
    host.close()
