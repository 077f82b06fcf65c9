"""C-ABI checks that need no GPU: the library loads and exports every symbol
the header declares; the plan's layout and the host sharding agree with the
oracle byte for byte; bad arguments fail closed with a status."""
import ctypes

import numpy as np
import pytest

import oracle
from tests._util import build_lib
from layerwise_weight_offload_gb300 import dlo, workloads as W


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_lib()


def test_library_exports_every_header_symbol():
    names = dlo.header_symbols()
    assert len(names) >= 25
    L = dlo.lib()
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    # every declared function has a binding signature
    assert set(names) <= set(dlo._SIGS), set(names) - set(dlo._SIGS)
    assert "sm_103a" in dlo.version()


def _descs_random(rng, n_params):
    """Parameters of every dtype code; some are strided views (transposed or
    with gaps), given with their element strides."""
    descs = []
    for i in range(n_params):
        code = int(rng.integers(0, 8))
        ndim = int(rng.integers(1, 4))
        shape = tuple(int(v) for v in rng.integers(1, 9, size=ndim))
        kind = int(rng.integers(0, 3))
        if kind == 0 or ndim == 1:
            descs.append(("p%d" % i, shape, code))
        elif kind == 1:                  # a row-major [.., b, a] tensor seen as [.., a, b]
            a_, b_ = shape[-2], shape[-1]
            st = [int(np.prod(shape[j + 1:])) for j in range(ndim)]
            st[-2], st[-1] = 1, a_
            descs.append(("p%d" % i, shape, code, tuple(st)))
        else:                            # row-major with a padded leading stride
            rm = [int(np.prod(shape[j + 1:])) for j in range(ndim)]
            st = list(rm)
            st[0] = rm[0] + int(rng.integers(1, 5))
            descs.append(("p%d" % i, shape, code, tuple(st)))
    return descs


def _storage(desc):
    shape = desc[1]
    if len(desc) > 3:
        return oracle.storage_extent(shape, desc[3])
    return int(np.prod(shape))


@pytest.mark.parametrize("seed", range(40))
def test_plan_layout_and_shards_match_oracle(seed):
    rng = np.random.default_rng(seed)
    descs = _descs_random(rng, int(rng.integers(1, 7)))
    s = int(rng.integers(1, 9))
    plan = dlo.Plan(descs, s)
    info = plan.info()
    numels = [_storage(d) for d in descs]          # elements packed per parameter
    codes = [d[2] for d in descs]
    esizes = [dlo.ESIZE[c] for c in codes]
    raw = [rng.integers(0, 256, size=n * e, dtype=np.uint8) for n, e in zip(numels, esizes)]
    image, gdt, gbase, used = oracle.slot_image(raw, numels, codes, esizes, s, 256)
    assert info.slot_bytes == used
    assert info.n_groups == len(gdt)
    shards = []
    for gi, g in enumerate(plan.groups()):
        assert g.dtype == gdt[gi] and g.base == gbase[gi]
        assert g.shard_numel == oracle.shard_numel(g.numel, s)
        assert g.shard_alloc_bytes % 16 == 0 and g.shard_alloc_bytes >= g.shard_bytes
        shards += [np.full(g.shard_alloc_bytes, 0xEE, np.uint8) for _ in range(s)]
    plan.shard_host([r.ctypes.data for r in raw], [x.ctypes.data for x in shards])
    # each host shard equals the oracle's shard, then zeros to the 16-byte end
    for gi, g in enumerate(plan.groups()):
        flat = oracle.flatten_group(list(zip(raw, numels, codes)), g.dtype, g.esize)
        ref = oracle.shard(flat, g.numel, g.esize, s)
        for r in range(s):
            got = shards[gi * s + r]
            assert np.array_equal(got[:g.shard_bytes], ref[r])
            assert not got[g.shard_bytes:].any()
    # the parameter views: offsets inside the oracle's slot image
    for p in range(len(descs)):
        pi = plan.param(p)
        assert pi.storage_numel == numels[p]
        assert pi.numel == int(np.prod(descs[p][1]))
        if len(descs[p]) > 3:
            assert tuple(pi.stride[:len(descs[p][1])]) == tuple(descs[p][3])
        n = numels[p] * esizes[p]
        assert np.array_equal(image[pi.slot_offset:pi.slot_offset + n], raw[p])


@pytest.mark.parametrize("seed", range(10))
def test_staging_layout(seed):
    rng = np.random.default_rng(100 + seed)
    descs = _descs_random(rng, int(rng.integers(1, 7)))
    s = int(rng.integers(1, 9))
    plan = dlo.Plan(descs, s)
    info = plan.info()
    end = 0
    for g in plan.groups():
        assert g.stage_base % 256 == 0 and g.stage_base >= end
        assert g.shard_alloc_bytes % 16 == 0
        end = g.stage_base + s * g.shard_alloc_bytes
    assert info.staging_bytes == end


def test_staged_engine_arguments_fail_closed():
    L = dlo.lib()
    out = ctypes.c_void_p()
    d = dlo.EngineDesc()
    d.n_blocks = 2
    d.slot[0], d.slot[1] = 4096, 4096 * 3
    d.slot_bytes = 100
    d.compute_stream, d.copy_stream = 8, 16
    d.copy_mode = dlo.COPY_STAGED
    assert L.dlo_engine_create(ctypes.byref(d), ctypes.byref(out)) == dlo.ERR_INVALID  # no staging
    d.staging[0], d.staging[1] = 4096 * 8, 4096 * 9
    d.staging_bytes = 100
    assert L.dlo_engine_create(ctypes.byref(d), ctypes.byref(out)) == dlo.ERR_INVALID  # no gather
    d.gather_stream = 16
    assert L.dlo_engine_create(ctypes.byref(d), ctypes.byref(out)) == dlo.ERR_INVALID  # = copy
    d.gather_stream = 24
    d.staging[1] = 4096 * 9 + 16
    assert L.dlo_engine_create(ctypes.byref(d), ctypes.byref(out)) == dlo.ERR_INVALID  # misaligned
    d.copy_mode = 4
    assert L.dlo_engine_create(ctypes.byref(d), ctypes.byref(out)) == dlo.ERR_INVALID  # no mode 4
    assert L.dlo_reassemble_staged(None, None, None, 0, None, None, None) == dlo.ERR_INVALID


def test_role_contract_needs_dtype_and_layout():
    w = W.CONFIGS["tiny"]
    descs = W.block_param_descs(w)
    assert dlo.Plan(descs, 2).info().has_dit_roles == 1
    # a transposed fc1 weight, or an fp8 one, is moved but not a DiT role
    i = [d[0] for d in descs].index("mlp.fc1.weight")
    f, d = descs[i][1]
    t = list(descs)
    t[i] = (descs[i][0], (f, d), W.BF16, (1, f))
    assert dlo.Plan(t, 2).info().has_dit_roles == 0
    q = list(descs)
    q[i] = (descs[i][0], (f, d), dlo.FP8_E4M3)
    assert dlo.Plan(q, 2).info().has_dit_roles == 0


@pytest.mark.parametrize("name", ["tiny", "odd", "nano", "super", "sweep-d1664-t256-s8"])
def test_workload_plans(name):
    w = W.CONFIGS[name]
    plan = dlo.Plan(W.block_param_descs(w), w.shards)
    info = plan.info()
    assert info.has_dit_roles == 1
    bf = [g for g in plan.groups() if g.dtype == W.BF16][0]
    f32 = [g for g in plan.groups() if g.dtype == W.F32][0]
    assert bf.numel == 12 * w.hidden ** 2 and f32.numel == 8 * w.hidden
    assert bf.shard_numel == oracle.shard_numel(bf.numel, w.shards)
    assert f32.shard_numel == oracle.shard_numel(f32.numel, w.shards)
    for p in range(info.n_params):
        assert plan.param(p).slot_offset % 16 == 0


def test_bad_arguments_fail_closed():
    L = dlo.lib()
    out = ctypes.c_void_p()
    assert L.dlo_plan_create(None, 1, 1, ctypes.byref(out)) == dlo.ERR_INVALID
    assert "null" in dlo.last_error()
    arr = (dlo.ParamDesc * 1)()
    arr[0].name = b"x"
    arr[0].ndim = 1
    arr[0].shape[0] = 4
    arr[0].dtype = 8                                   # no such dtype code
    assert L.dlo_plan_create(arr, 1, 2, ctypes.byref(out)) == dlo.ERR_INVALID
    arr[0].dtype = 0
    arr[0].stride[0] = -1                              # negative stride
    assert L.dlo_plan_create(arr, 1, 2, ctypes.byref(out)) == dlo.ERR_INVALID
    arr[0].stride[0] = 0
    assert L.dlo_plan_create(arr, 1, 0, ctypes.byref(out)) == dlo.ERR_INVALID
    arr[0].shape[0] = 0
    assert L.dlo_plan_create(arr, 1, 1, ctypes.byref(out)) == dlo.ERR_INVALID
    with pytest.raises(dlo.DLOError):
        dlo.Plan([("a", (3,), 0)], 2).group(5)
    # engine: rejects equal streams, null slots, misalignment before any CUDA call
    d = dlo.EngineDesc()
    d.n_blocks = 2
    assert L.dlo_engine_create(ctypes.byref(d), ctypes.byref(out)) == dlo.ERR_INVALID
    d.slot[0], d.slot[1] = 4096, 4096 * 3
    d.slot_bytes = 100
    d.compute_stream = d.copy_stream = 8
    assert L.dlo_engine_create(ctypes.byref(d), ctypes.byref(out)) == dlo.ERR_INVALID
    d.copy_stream = 16
    d.slot[1] = 4096 * 3 + 8
    assert L.dlo_engine_create(ctypes.byref(d), ctypes.byref(out)) == dlo.ERR_INVALID
    # forward config checks
    assert dlo.forward_scratch_bytes(dlo.dit_cfg(1, 16, 96, 1, 256)) == 0     # hidden % 64
    assert dlo.forward_scratch_bytes(dlo.dit_cfg(1, 16, 256, 8, 1024)) == 0   # head dim 32
    assert dlo.forward_scratch_bytes(dlo.dit_cfg(1, 16, 256, 4, 1024)) > 0
    # engine calls on a null engine
    assert L.dlo_prefetch(None, 0, 0) == dlo.ERR_INVALID
    assert L.dlo_engine_destroy(None, 10) == dlo.OK


def test_scratch_bytes_cover_the_buffers():
    w = W.CONFIGS["odd"]
    cfg = dlo.dit_cfg(w.batch, w.tokens, w.hidden, w.heads, w.mlp)
    M, d, f = w.tokens, w.hidden, w.mlp
    assert dlo.forward_scratch_bytes(cfg) >= 2 * M * (d + 3 * d + d + f)


def test_forward_launch_count():
    # norms, attention (+ the merge of its KV slices), and the four linears
    # with a reduction each when some of their tiles are split into K slices
    for name in ("tiny", "odd", "nano", "super"):
        w = W.CONFIGS[name]
        n = dlo.forward_launches(dlo.dit_cfg(w.batch, w.tokens, w.hidden, w.heads, w.mlp))
        assert 7 <= n <= 12
    assert dlo.forward_launches(dlo.dit_cfg(1, 16, 96, 1, 256)) == 0       # invalid config


def test_gemm_pair_mode_and_query():
    # the mode takes -1, 0 or 1 and refuses anything else (no GPU needed);
    # the query answers 0 for empty or negative extents, and with no GPU the
    # pair kernel is never available, whatever the mode
    for mode in (dlo.GEMM_PAIR_OFF, dlo.GEMM_PAIR_ON, dlo.GEMM_PAIR_AUTO):
        dlo.set_gemm_pair_mode(mode)
    with pytest.raises(dlo.DLOError):
        dlo.set_gemm_pair_mode(2)
    with pytest.raises(dlo.DLOError):
        dlo.set_gemm_pair_mode(-2)
    assert not dlo.op_linear_on_pairs(0, 256, 256, dlo.EPI_BF16)
    assert not dlo.op_linear_on_pairs(256, -1, 256, dlo.EPI_BF16)
    import torch
    if not torch.cuda.is_available():
        dlo.set_gemm_pair_mode(dlo.GEMM_PAIR_ON)
        try:
            assert not dlo.op_linear_on_pairs(8192, 24576, 6144, dlo.EPI_GELU_BF16)
        finally:
            dlo.set_gemm_pair_mode(dlo.GEMM_PAIR_AUTO)
