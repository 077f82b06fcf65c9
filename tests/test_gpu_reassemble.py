"""The prefetch's bytes: a slot reassembled on the GPU (DMA and the copy
kernel) equals the oracle's slot image byte for byte."""
import numpy as np
import pytest
import torch

import oracle
from tests._util import build_lib, raw_bytes, assert_only_groups_written
from layerwise_weight_offload_gb300 import dlo, workloads as W
from layerwise_weight_offload_gb300.stack import HostBlocks, PinnedBuffer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_lib()


def _expected_image(host, hb):
    w = host.w
    p = host.params[hb]
    numels = [int(np.prod(sh)) for _, sh, _ in host.descs]
    codes = [c for _, _, c in host.descs]
    esizes = [W.ESIZE[c] for c in codes]
    raw = [raw_bytes(p[name]) for name, _, _ in host.descs]
    image, _, _, used = oracle.slot_image(raw, numels, codes, esizes, w.shards, 256)
    return image


@pytest.mark.parametrize("mode", [dlo.COPY_DMA, dlo.COPY_KERNEL])
@pytest.mark.parametrize("name", ["tiny", "odd"])
def test_workload_slot_bit_exact(name, mode):
    w = W.CONFIGS[name]
    w = W.Workload(**{**w.__dict__, "distinct": 2, "n_blocks": 2})
    host = HostBlocks(w, seed=3, keep_params=True)
    info = host.plan.info()
    dst = torch.full((info.slot_bytes + 512,), 0xA5, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    for hb in range(2):
        dlo.reassemble(host.plan, host.shard_ptrs(hb), dst, mode, s)
        s.synchronize()
        got = dst.cpu().numpy()
        exp = _expected_image(host, hb)
        # every group's gathered range equals the image; nothing else written
        for g in host.plan.groups():
            n = w.shards * g.shard_bytes
            assert np.array_equal(got[g.base:g.base + n], exp[g.base:g.base + n]), (hb, g.dtype)
        assert_only_groups_written(got, host.plan.groups(), w.shards, 0xA5, (name, hb))
    host.close()


def _custom_plan_case(rng, s):
    """Random parameter sets whose shard byte lengths are not multiples of 16."""
    descs = []
    for i in range(int(rng.integers(1, 6))):
        code = int(rng.integers(0, 2))
        n = int(rng.integers(1, 5000))
        descs.append(("p%d" % i, (n,), code))
    return descs


@pytest.mark.parametrize("mode", [dlo.COPY_DMA, dlo.COPY_KERNEL])
def test_misaligned_shards_bit_exact(mode):
    rng = np.random.default_rng(11)
    s_stream = torch.cuda.Stream()
    n_cases = 0
    for trial in range(40):
        s = int(rng.integers(1, 9))
        descs = _custom_plan_case(rng, s)
        plan = dlo.Plan(descs, s)
        groups = plan.groups()
        numels = [d[1][0] for d in descs]
        codes = [d[2] for d in descs]
        esizes = [W.ESIZE[c] for c in codes]
        raw = [rng.integers(0, 256, size=n * e, dtype=np.uint8) for n, e in zip(numels, esizes)]
        sizes = [g.shard_alloc_bytes for g in groups for _ in range(s)]
        offs = np.cumsum([0] + [(x + 255) // 256 * 256 for x in sizes])
        buf = PinnedBuffer(int(offs[-1]))
        ptrs = [buf.ptr + int(o) for o in offs[:-1]]
        plan.shard_host([r.ctypes.data for r in raw], ptrs)
        info = plan.info()
        dst = torch.full((info.slot_bytes + 256,), 0x5A, dtype=torch.uint8, device="cuda")
        dlo.reassemble(plan, ptrs, dst, mode, s_stream)
        s_stream.synchronize()
        got = dst.cpu().numpy()
        exp, _, gbase, used = oracle.slot_image(raw, numels, codes, esizes, s, 256)
        for g in groups:
            n = s * g.shard_bytes
            assert np.array_equal(got[g.base:g.base + n], exp[g.base:g.base + n]), (trial, s)
            if g.shard_bytes % 16:
                n_cases += 1
        assert_only_groups_written(got, groups, s, 0x5A, (trial, s))
        buf.close()
    assert n_cases > 10        # the misaligned paths were exercised


@pytest.mark.parametrize("same_stream", [False, True])
@pytest.mark.parametrize("name", ["tiny", "odd"])
def test_staged_reassembly_bit_exact(name, same_stream):
    # the two-phase form: H2D into device staging, then the device gather
    w = W.CONFIGS[name]
    w = W.Workload(**{**w.__dict__, "distinct": 2, "n_blocks": 2})
    host = HostBlocks(w, seed=4, keep_params=True)
    info = host.plan.info()
    dst = torch.full((info.slot_bytes + 512,), 0xA5, dtype=torch.uint8, device="cuda")
    staging = torch.full((info.staging_bytes,), 0x5A, dtype=torch.uint8, device="cuda")
    cs = torch.cuda.Stream()
    gs = cs if same_stream else torch.cuda.Stream()
    for hb in range(2):
        dlo.reassemble_staged(host.plan, host.shard_ptrs(hb), staging, info.staging_bytes, dst,
                              cs, gs)
        torch.cuda.synchronize()
        got = dst.cpu().numpy()
        exp = _expected_image(host, hb)
        for g in host.plan.groups():
            n = w.shards * g.shard_bytes
            assert np.array_equal(got[g.base:g.base + n], exp[g.base:g.base + n]), (hb, g.dtype)
            # staging holds each host shard at its 16-byte aligned offset
            st = staging.cpu().numpy()
            views = host.shard_views(hb)
            gi = [x.dtype for x in host.plan.groups()].index(g.dtype)
            for r in range(w.shards):
                off = g.stage_base + r * g.shard_alloc_bytes
                assert np.array_equal(st[off:off + g.shard_bytes],
                                      views[gi * w.shards + r][:g.shard_bytes].numpy())
        assert_only_groups_written(got, host.plan.groups(), w.shards, 0xA5, (name, hb))
    with pytest.raises(dlo.DLOError):
        dlo.reassemble_staged(host.plan, host.shard_ptrs(0), staging, info.staging_bytes - 16,
                              dst, cs, gs)
    with pytest.raises(dlo.DLOError):
        dlo.reassemble(host.plan, host.shard_ptrs(0), dst, dlo.COPY_STAGED, cs)
    host.close()
