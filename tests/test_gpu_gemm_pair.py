"""The CTA-pair GEMM kernel (one tcgen05 MMA over two SMs, 256 x 256 output
tiles) against the oracle's linear: every epilogue with and without a bias,
ragged M, N and K (including pairs whose second CTA's half of A or of W lies
wholly past the edge), more tiles than CTA pairs, a short last wave split in
K over the idle pairs; then whole block forwards
with every linear on CTA pairs (the QKV epilogue's transposed V included),
streamed equal to resident and both against the oracle's block."""
import numpy as np
import pytest
import torch

import oracle
from tests._util import build_lib, params_f32, assert_oracle_close
from layerwise_weight_offload_gb300 import dlo, workloads as W
from layerwise_weight_offload_gb300.stack import HostBlocks, StreamedStack, ResidentStack

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _pairs_for_every_linear():
    build_lib()
    dlo.set_gemm_pair_mode(dlo.GEMM_PAIR_ON)
    yield
    dlo.set_gemm_pair_mode(dlo.GEMM_PAIR_AUTO)


def _gen(seed):
    g = torch.Generator().manual_seed(seed)
    return lambda *shape, std=1.0: std * torch.randn(*shape, generator=g)


PAIR_SHAPES = [
    (256, 64, 256),      # one pair tile
    (512, 1024, 768),    # 2 x 3 tiles
    (300, 320, 264),     # ragged: the second CTA's rows of A (384..) and of W (384..) are all
                         # past the edge in the last row / column block
    (1, 64, 8),          # degenerate
    (129, 4096, 136),    # long K, ragged
    (4096, 512, 4352),   # 16 x 17 tiles: more than one wave of pairs, both accumulators cycle
]


@pytest.mark.parametrize("bias", [False, True])
@pytest.mark.parametrize("M,K,N", PAIR_SHAPES)
@pytest.mark.parametrize("epi", [dlo.EPI_BF16, dlo.EPI_GELU_BF16, dlo.EPI_RESID_F32])
def test_linear_pair(M, K, N, epi, bias):
    r = _gen(M * 31 + K * 3 + N + 7 * epi + bias)
    a = r(M, K).to(torch.bfloat16)
    w = r(N, K, std=0.05).to(torch.bfloat16)
    b = r(N, std=0.5).to(torch.bfloat16) if bias else None
    # unsplit on pairs: no workspace
    assert dlo.op_linear_workspace_bytes(M, N, K, epi) == 0
    ref = oracle.linear(a.float().numpy(), w.float().numpy())
    if bias:
        ref = ref + b.double().numpy()
    bd = b.cuda() if bias else None
    if epi == dlo.EPI_RESID_F32:
        x = r(M, N)
        gate = r(N, std=0.1)
        xd = x.cuda()
        dlo.op_linear(a.cuda(), M, K, w.cuda(), N, epi, xd, gate.cuda(), bias=bd)
        torch.cuda.synchronize()
        assert dlo.kernel_status() == 0
        got = xd.cpu().numpy()
        exp = x.numpy().astype(np.float64) + gate.numpy().astype(np.float64) * ref
        assert np.abs(got - exp).max() <= 1e-4 * max(1.0, np.abs(exp).max())
        assert_oracle_close(got - x.numpy(), exp - x.numpy(), "resid delta", 1e-3, 1e-4)
    else:
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        dlo.op_linear(a.cuda(), M, K, w.cuda(), N, epi, out, None, bias=bd)
        torch.cuda.synchronize()
        assert dlo.kernel_status() == 0
        got = out.float().cpu().numpy()
        if epi == dlo.EPI_GELU_BF16:
            ref = np.vectorize(oracle.gelu_tanh)(ref)
        tol = 2.0 ** -8 * np.abs(ref) + 1e-5 * np.sqrt(K) * np.abs(ref).max()
        assert np.all(np.abs(got - ref) <= tol), np.abs(got - ref).max()


@pytest.mark.parametrize("epi", [dlo.EPI_BF16, dlo.EPI_GELU_BF16, dlo.EPI_RESID_F32])
@pytest.mark.parametrize("shape", ["column", "grid"])
def test_linear_pair_tail_split(epi, shape):
    # a short last wave of pairs: its tiles run as K slices on the idle pairs
    # (fp32 partials of 256 x 256 blocks), summed in slice order by the tail
    # reduction; "grid": 3 column blocks, the tail's last tile being the
    # ragged last row block of the ragged last column block.  Checked on the
    # rows of the last 6 row blocks (every tail tile) and a sample of the others.
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    K = 2048
    if shape == "column":
        M, N = 256 * (pairs + 5) - 37, 256
    else:
        t = next(t for t in range(1, pairs) if (pairs + t) % 3 == 0)
        M, N = 256 * ((pairs + t) // 3) - 50, 760
    nws = dlo.op_linear_workspace_bytes(M, N, K, epi)
    assert nws > 0 and nws % (256 * 256 * 4) == 0
    g = torch.Generator().manual_seed(M + N + epi)
    a = torch.randn(M, K, generator=g).to(torch.bfloat16)
    w = (0.05 * torch.randn(N, K, generator=g)).to(torch.bfloat16)
    ws = torch.full((nws // 4,), float("nan"), device="cuda")
    rng = np.random.default_rng(M)
    sel = np.unique(np.concatenate([np.arange(max(0, M - 6 * 256), M), rng.integers(0, M, 256)]))
    ref = oracle.linear(a[sel].float().numpy(), w.float().numpy())
    if epi == dlo.EPI_RESID_F32:
        x = torch.randn(M, N, generator=g)
        gate = 0.1 * torch.randn(N, generator=g)
        xd = x.cuda()
        dlo.op_linear(a.cuda(), M, K, w.cuda(), N, epi, xd, gate.cuda(), None, ws, nws)
        torch.cuda.synchronize()
        assert dlo.kernel_status() == 0
        got = xd.cpu().numpy()[sel]
        exp = x.numpy()[sel].astype(np.float64) + gate.numpy().astype(np.float64) * ref
        assert np.abs(got - exp).max() <= 1e-4 * max(1.0, np.abs(exp).max())
    else:
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        dlo.op_linear(a.cuda(), M, K, w.cuda(), N, epi, out, None, None, ws, nws)
        torch.cuda.synchronize()
        assert dlo.kernel_status() == 0
        full = out.float().cpu().numpy()
        assert not np.isnan(full).any()
        got = full[sel]
        if epi == dlo.EPI_GELU_BF16:
            ref = np.vectorize(oracle.gelu_tanh)(ref)
        tol = 2.0 ** -8 * np.abs(ref) + 1e-5 * np.sqrt(K) * np.abs(ref).max()
        assert np.all(np.abs(got - ref) <= tol), np.abs(got - ref).max()


def test_auto_policy_on_the_workload_shapes():
    # by shape: pairs for every linear of the Super and Nano blocks, none at
    # the odd workload's sizes (fewer pair tiles than pairs)
    dlo.set_gemm_pair_mode(dlo.GEMM_PAIR_AUTO)
    for T, d, f, want in [(8192, 6144, 24576, True), (4096, 3840, 15360, True),
                          (1024, 1024, 4096, False)]:
        for N, K, epi in [(3 * d, d, dlo.EPI_BF16), (d, d, dlo.EPI_RESID_F32),
                          (f, d, dlo.EPI_GELU_BF16), (d, f, dlo.EPI_RESID_F32)]:
            assert dlo.op_linear_on_pairs(T, N, K, epi) == want, (T, N, K)


def test_mode_switch_changes_the_plan():
    # a shape that splits in K on single CTAs runs unsplit on pairs
    M, K, N = 77, 4096, 1024
    assert dlo.op_linear_workspace_bytes(M, N, K, dlo.EPI_RESID_F32) == 0
    dlo.set_gemm_pair_mode(dlo.GEMM_PAIR_OFF)
    assert dlo.op_linear_workspace_bytes(M, N, K, dlo.EPI_RESID_F32) > 0
    with pytest.raises(dlo.DLOError):
        dlo.set_gemm_pair_mode(2)


@pytest.mark.parametrize("cfg", [
    dict(n_blocks=3, hidden=320, heads=5, mlp=1280, tokens=200, shards=3),
    dict(n_blocks=2, hidden=384, heads=3, mlp=1536, tokens=77, shards=5, batch=2),
    dict(n_blocks=2, hidden=512, heads=4, mlp=2048, tokens=1000, shards=2, variant="full"),
])
def test_block_forward_on_pairs_streamed_vs_resident_vs_oracle(cfg):
    w = W.custom("pairs", steps=2, **cfg)
    host = HostBlocks(w, seed=21, keep_params=True)
    x0 = W.gen_x(w, seed=21)
    dcfg = dlo.dit_cfg(w.batch, w.tokens, w.hidden, w.heads, w.mlp, w.eps, **W.cfg_flags(w))
    # two norms, attention (+ the merge of its KV slices), four unsplit
    # linears, the q/k norm and rotary kernel of the checkpoint-shaped block
    extra = 1 if w.variant == "full" else 0
    assert dlo.forward_launches(dcfg) in (7 + extra, 8 + extra)
    rs = ResidentStack(host)
    x = x0.clone().cuda()
    per_block = []
    for _ in range(w.steps):
        rs.stream.wait_stream(torch.cuda.current_stream())
        for i in range(w.n_blocks):
            xin = x.clone()
            rs.block(i, x)
            torch.cuda.current_stream().wait_stream(rs.stream)
            per_block.append((i, xin, x.clone()))
    torch.cuda.synchronize()
    st = StreamedStack(host, copy_mode=dlo.COPY_AUTO)
    xs = x0.clone().cuda()
    for _ in range(w.steps):
        st.compute.wait_stream(torch.cuda.current_stream())
        st.step(xs)
        torch.cuda.current_stream().wait_stream(st.compute)
    torch.cuda.synchronize()
    st.close()
    assert torch.equal(xs, x)
    assert dlo.kernel_status() == 0
    for i, xin, xout in per_block:
        p = params_f32(host.params[i % w.distinct])
        xin_np = xin.cpu().numpy()
        ref = oracle.block_forward(xin_np, p, w.batch, w.tokens, w.hidden, w.heads, w.mlp, w.eps,
                                   rope_base=W.oracle_rope_base(w))
        got = xout.cpu().numpy()
        assert_oracle_close(got, ref, "block %d output" % i)
        assert_oracle_close(got - xin_np, ref - xin_np, "block %d update" % i, 2e-2, 1e-2)
    host.close()
