"""Each kernel of the block forward against the oracle's step, on the same
seeded inputs: RMSNorm+adaLN, the tcgen05 linear with its three epilogues
(ragged M, N and K included), and attention (head dims 64 and 128, ragged
token counts, two batch items)."""
import numpy as np
import pytest
import torch

import oracle
from tests._util import build_lib, assert_oracle_close
from layerwise_weight_offload_gb300 import dlo

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_lib()


def _gen(seed):
    g = torch.Generator().manual_seed(seed)
    return lambda *shape, std=1.0: std * torch.randn(*shape, generator=g)


def _status_clean():
    torch.cuda.synchronize()
    assert dlo.kernel_status() == 0


@pytest.mark.parametrize("rows,d", [(1, 64), (7, 256), (200, 1024), (33, 3840), (5, 6656),
                                    (3, 8192), (2, 8196), (4, 100)])
def test_rmsnorm_mod(rows, d):
    r = _gen(rows * 7 + d)
    x = r(rows, d)
    g = 1.0 + r(d, std=0.1)
    shift, scale = r(d, std=0.1), r(d, std=0.1)
    xd, gd, sd, cd = (t.cuda() for t in (x, g, shift, scale))
    h = torch.empty(rows, d, dtype=torch.bfloat16, device="cuda")
    dlo.op_rmsnorm_mod(xd, rows, d, gd, sd, cd, 1e-6, h)
    _status_clean()
    ref = oracle.rmsnorm_mod(x.numpy(), g.numpy(), shift.numpy(), scale.numpy(), 1e-6)
    got = h.float().cpu().numpy()
    # bf16 output: each element within one bf16 rounding of the exact value
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)


LIN_SHAPES = [
    (128, 64, 256),      # one tile
    (256, 1024, 3072),   # several tiles in M, N and K
    (200, 320, 264),     # ragged M, N (vs 256) and K (vs 64)
    (1, 64, 8),          # degenerate
    (1000, 1024, 1024),
    (77, 4096, 1024),    # long K: splits 8 ways when a workspace is given
    (1024, 4096, 1024),  # the odd workload's fc2 shape
]


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("M,K,N", LIN_SHAPES)
@pytest.mark.parametrize("epi", [dlo.EPI_BF16, dlo.EPI_GELU_BF16, dlo.EPI_RESID_F32])
def test_linear(M, K, N, epi, split):
    r = _gen(M * 131 + K * 7 + N + epi)
    a = r(M, K).to(torch.bfloat16)
    w = r(N, K, std=0.05).to(torch.bfloat16)
    ad, wd = a.cuda(), w.cuda()
    nws = dlo.op_linear_workspace_bytes(M, N, K, epi) if split else 0
    if split and nws == 0:
        pytest.skip("this shape does not split")
    ws = torch.full((max(nws, 16) // 4,), float("nan"), device="cuda") if split else None
    ref = oracle.linear(a.float().numpy(), w.float().numpy())
    if epi == dlo.EPI_RESID_F32:
        x = r(M, N)
        gate = r(N, std=0.1)
        xd, gd = x.cuda(), gate.cuda()
        dlo.op_linear(ad, M, K, wd, N, epi, xd, gd, None, ws, nws)
        _status_clean()
        got = xd.cpu().numpy()
        exp = x.numpy().astype(np.float64) + gate.numpy().astype(np.float64) * ref
        # fp32 accumulation against fp64: |err| << 1e-4 for these magnitudes
        assert np.abs(got - exp).max() <= 1e-4 * max(1.0, np.abs(exp).max())
        delta_got = got - x.numpy()
        assert_oracle_close(delta_got, exp - x.numpy(), "resid delta", 1e-3, 1e-4)
    else:
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        dlo.op_linear(ad, M, K, wd, N, epi, out, None, None, ws, nws)
        _status_clean()
        got = out.float().cpu().numpy()
        if epi == dlo.EPI_GELU_BF16:
            ref = np.vectorize(oracle.gelu_tanh)(ref)
        tol = 2.0 ** -8 * np.abs(ref) + 1e-5 * np.sqrt(K) * np.abs(ref).max()
        assert np.all(np.abs(got - ref) <= tol), np.abs(got - ref).max()


@pytest.mark.parametrize("B,T,d,H", [(1, 7, 256, 4), (2, 300, 512, 4), (1, 1000, 1024, 16)])
@pytest.mark.parametrize("norm,rope", [(True, True), (True, False), (False, True)])
def test_qk_norm_rope(B, T, d, H, norm, rope):
    r = _gen(B * T + d + 2 * norm + rope)
    hd = d // H
    qkv = (r(B * T, 3 * d)).to(torch.bfloat16)
    gq, gk = (1.0 + r(hd, std=0.1)), (1.0 + r(hd, std=0.1))
    dev = qkv.cuda()
    dlo.op_qk_norm_rope(dev, B, T, d, H, gq.cuda() if norm else None,
                        gk.cuda() if norm else None, 1e-6, 10000.0 if rope else 0.0)
    _status_clean()
    ref = qkv.double().numpy()
    if norm:
        ref = oracle.qk_norm(ref, d, H, gq.numpy(), gk.numpy(), 1e-6)
    if rope:
        ref = oracle.rope(ref, B, T, d, H, 10000.0)
    got = dev.double().cpu().numpy()
    # v untouched bit for bit; q and k within a bf16 rounding plus the fp32
    # angle (position * frequency rounded to fp32: up to T * 2^-24 rad)
    assert np.array_equal(got[:, 2 * d:], qkv.double().numpy()[:, 2 * d:])
    err = np.abs(got[:, :2 * d] - ref[:, :2 * d])
    scale = np.abs(ref[:, :2 * d]).max()
    assert np.all(err <= 2.0 ** -8 * np.abs(ref[:, :2 * d]) + (T * 2.0 ** -23 + 1e-5) * scale), \
        err.max()


@pytest.mark.parametrize("epi", [dlo.EPI_BF16, dlo.EPI_GELU_BF16, dlo.EPI_RESID_F32])
@pytest.mark.parametrize("M,K,N,split", [(200, 320, 264, False), (77, 4096, 1024, True),
                                         (1000, 1024, 1024, False)])
def test_linear_bias(M, K, N, epi, split):
    r = _gen(M + K + N + epi)
    a = r(M, K).to(torch.bfloat16)
    w = r(N, K, std=0.05).to(torch.bfloat16)
    bias = r(N, std=0.5).to(torch.bfloat16)
    nws = dlo.op_linear_workspace_bytes(M, N, K, epi) if split else 0
    if split and nws == 0:
        pytest.skip("this shape does not split")
    ws = torch.full((max(nws, 16) // 4,), float("nan"), device="cuda") if split else None
    ref = oracle.linear(a.float().numpy(), w.float().numpy()) + bias.double().numpy()
    if epi == dlo.EPI_RESID_F32:
        x = r(M, N)
        gate = r(N, std=0.1)
        xd = x.cuda()
        dlo.op_linear(a.cuda(), M, K, w.cuda(), N, epi, xd, gate.cuda(), None, ws, nws,
                      bias=bias.cuda())
        _status_clean()
        exp = x.numpy().astype(np.float64) + gate.numpy().astype(np.float64) * ref
        assert np.abs(xd.cpu().numpy() - exp).max() <= 1e-4 * max(1.0, np.abs(exp).max())
    else:
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        dlo.op_linear(a.cuda(), M, K, w.cuda(), N, epi, out, None, None, ws, nws,
                      bias=bias.cuda())
        _status_clean()
        got = out.float().cpu().numpy()
        if epi == dlo.EPI_GELU_BF16:
            ref = np.vectorize(oracle.gelu_tanh)(ref)
        tol = 2.0 ** -8 * np.abs(ref) + 1e-5 * np.sqrt(K) * np.abs(ref).max()
        assert np.all(np.abs(got - ref) <= tol), np.abs(got - ref).max()


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.fixture
def one_cta_gemm():
    # the single-CTA kernel and its K splits for every linear (a shape with
    # enough tiles would otherwise run on CTA pairs)
    dlo.set_gemm_pair_mode(dlo.GEMM_PAIR_OFF)
    yield
    dlo.set_gemm_pair_mode(dlo.GEMM_PAIR_AUTO)


@pytest.mark.parametrize("epi", [dlo.EPI_BF16, dlo.EPI_GELU_BF16, dlo.EPI_RESID_F32])
@pytest.mark.parametrize("shape", ["column", "grid"])
def test_linear_tail_split(epi, shape, one_cta_gemm):
    # a short last wave: only its tiles are split in K, the rest finish in
    # the kernel; "grid": 3 column blocks, the tail tile being the ragged
    # last row block of the ragged last column block.  Checked on the rows of
    # the last 6 row blocks (every tail tile) and a sample of the others.
    sms = _sms()
    K = 2048
    if shape == "column":
        tail = 5
        M, N = 128 * (sms + tail) - 37, 256
    else:
        tail = next(t for t in range(1, sms) if (sms + t) % 3 == 0)
        M, N = 128 * ((sms + tail) // 3) - 50, 760
    ts = min(sms // tail, K // 64 // 4, 8)
    nws = dlo.op_linear_workspace_bytes(M, N, K, epi)
    assert nws == tail * ts * 128 * 256 * 4
    r = _gen(M + N + epi)
    a = r(M, K).to(torch.bfloat16)
    w = r(N, K, std=0.05).to(torch.bfloat16)
    ad, wd = a.cuda(), w.cuda()
    ws = torch.full((nws // 4,), float("nan"), device="cuda")
    rng = np.random.default_rng(M)
    sel = np.unique(np.concatenate([np.arange(max(0, M - 6 * 128), M),
                                    rng.integers(0, M, 256)]))
    ref = oracle.linear(a[sel].float().numpy(), w.float().numpy())
    if epi == dlo.EPI_RESID_F32:
        x = r(M, N)
        gate = r(N, std=0.1)
        xd = x.cuda()
        dlo.op_linear(ad, M, K, wd, N, epi, xd, gate.cuda(), None, ws, nws)
        _status_clean()
        got = xd.cpu().numpy()[sel]
        exp = x.numpy()[sel].astype(np.float64) + gate.numpy().astype(np.float64) * ref
        assert np.abs(got - exp).max() <= 1e-4 * max(1.0, np.abs(exp).max())
    else:
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        dlo.op_linear(ad, M, K, wd, N, epi, out, None, None, ws, nws)
        _status_clean()
        full = out.float().cpu().numpy()
        assert not np.isnan(full).any()
        got = full[sel]
        if epi == dlo.EPI_GELU_BF16:
            ref = np.vectorize(oracle.gelu_tanh)(ref)
        tol = 2.0 ** -8 * np.abs(ref) + 1e-5 * np.sqrt(K) * np.abs(ref).max()
        assert np.all(np.abs(got - ref) <= tol), np.abs(got - ref).max()


def _attention(qkv, B, T, d, H, o):
    n = dlo.op_attention_scratch_bytes(B, T, d)
    scratch = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")   # NaN-filled
    dlo.op_attention(qkv, B, T, d, H, o, scratch, n)


ATT_SHAPES = [
    (1, 64, 256, 4),     # hd 64, one KV tile
    (1, 200, 256, 4),    # ragged tokens
    (2, 130, 512, 4),    # hd 128, two batch items, ragged
    (1, 1, 128, 1),      # single token: output = v
    (1, 1024, 1024, 16),
    (1, 333, 384, 3),
    (1, 2500, 256, 2),   # many KV tiles: rescaling path, hd 128
    (3, 129, 128, 2),    # three batch items, one key past a tile
    # grids of at least one CTA per SM take two query tiles per CTA
    (2, 1100, 2048, 16),  # hd 128, ragged last pair, second batch item; on 152 SMs the
                          # last wave (8 pairs) runs as KV slices merged by a second kernel
    (1, 2000, 1216, 19),  # hd 64, last CTA's second tile partly past the end
    (1, 2100, 1280, 20),  # hd 64, ragged: 180 pairs, the last 28 as 5 KV slices each
    (1, 1536, 2048, 16),  # one query tile per CTA: 192 tiles, the last 40 as 3 KV slices
]


@pytest.mark.parametrize("B,T,d,H", ATT_SHAPES)
def test_attention(B, T, d, H):
    r = _gen(B * 1000 + T + d + H)
    qkv = r(B * T, 3 * d).to(torch.bfloat16)
    o = torch.full((B * T, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    _attention(qkv.cuda(), B, T, d, H, o)
    _status_clean()
    ref = oracle.attention(qkv.float().numpy(), B, T, d, H)
    got = o.float().cpu().numpy()
    assert_oracle_close(got, ref, "attention", 1e-2, 4e-3)
    if T == 1:
        assert np.array_equal(got, qkv[:, 2 * d:].float().numpy())


def test_attention_scale_is_checked_by_two_tokens():
    # two tokens, one head of 64: output is a sigmoid-weighted mix of v0, v1
    d = 64
    qkv = torch.zeros(2, 3 * d)
    qkv[:, :d] = torch.randn(2, d, generator=torch.Generator().manual_seed(0))
    qkv[:, d:2 * d] = torch.randn(2, d, generator=torch.Generator().manual_seed(1))
    qkv[:, 2 * d:] = torch.randn(2, d, generator=torch.Generator().manual_seed(2))
    qkv = qkv.to(torch.bfloat16)
    o = torch.empty(2, d, dtype=torch.bfloat16, device="cuda")
    _attention(qkv.cuda(), 1, 2, d, 1, o)
    _status_clean()
    ref = oracle.attention(qkv.float().numpy(), 1, 2, d, 1)
    assert_oracle_close(o.float().cpu().numpy(), ref, "two tokens", 1e-2, 4e-3)


def test_rejects_unsupported_shapes():
    a = torch.zeros(4, 12, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dlo.DLOError):
        dlo.op_linear(a, 4, 12, a, 4, dlo.EPI_BF16, a)            # K, N not multiples of 8
    q = torch.zeros(4, 96 * 3, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dlo.DLOError):
        _attention(q, 1, 4, 96, 3, q)                              # head dim 32


@pytest.mark.parametrize("d,H", [(256, 4), (256, 2), (3072, 24)])
def test_attention_scores_growing_across_tiles(d, H):
    # scores rise with the key index, so later KV tiles have a much larger
    # row maximum than the first one: exercises the rescale-and-redo path
    T = 2048
    hd = d // H
    qkv = torch.zeros(T, 3 * d)
    qkv[:, :d] = 1.0
    ramp = torch.arange(T, dtype=torch.float32) / T
    qkv[:, d:2 * d] = (ramp * 40.0 / hd ** 0.5)[:, None] * 8.0
    qkv[:, 2 * d:] = torch.randn(T, d, generator=torch.Generator().manual_seed(5))
    qkv = qkv.to(torch.bfloat16)
    o = torch.full((T, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    _attention(qkv.cuda(), 1, T, d, H, o)
    _status_clean()
    ref = oracle.attention(qkv.float().numpy(), 1, T, d, H)
    assert_oracle_close(o.float().cpu().numpy(), ref, "growing scores", 1e-2, 4e-3)
