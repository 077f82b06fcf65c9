"""Pins of the CPU oracle to facts that do not come from the oracle itself:
numbers the pages print, closed forms, invariants, special cases that reduce
to a textbook result, and library routines on small shapes.  No GPU."""
import ctypes
import itertools
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return [list(map(int, l.split())) for l in fh if l.strip() and not l.startswith("#")]


# ---------------------------------------------------------------- sharding

def test_shard_size_matches_pages_printed_sizes():
    # block 368 MB -> DP2 shard 184 MB; Super 124 GB over DP4 -> 31 GB/rank
    for total, dp, shard in _rows("overlap_analysis.txt"):
        assert oracle.shard_numel(total, dp) == shard


def test_shard_size_is_smallest_equal_split():
    # Equal-size shards (all_gather_into_tensor needs them) with the least
    # padding: s*S >= N and (S-1)*s < N.
    for n in range(0, 200):
        for s in range(1, 9):
            S = oracle.shard_numel(n, s)
            assert S * s >= n
            assert n == 0 or (S - 1) * s < n


@pytest.mark.parametrize("esize", [1, 2, 4])
def test_shard_reassemble_brute_force(esize):
    rng = np.random.default_rng(1)
    for n in range(1, 65):
        for s in range(1, 9):
            flat = rng.integers(1, 256, size=n * esize, dtype=np.uint8)  # no zero bytes
            shards = oracle.shard(flat, n, esize, s)
            S = oracle.shard_numel(n, s)
            assert all(len(x) == S * esize for x in shards)
            gathered = oracle.reassemble(shards, S, esize)
            # rank-order concatenation reproduces the flat buffer ...
            assert np.array_equal(gathered[: n * esize], flat)
            # ... and everything past it is zero padding
            assert not gathered[n * esize:].any()
            # shard r is exactly the r-th window of the concatenation
            for r, x in enumerate(shards):
                assert np.array_equal(x, gathered[r * S * esize:(r + 1) * S * esize])


def test_shard_of_nonmultiple_pads_last_shard_only():
    # 10 elements over 3 shards -> 4,4,4 with two zeros at the end of shard 2
    flat = np.arange(1, 11, dtype=np.uint8)
    sh = oracle.shard(flat, 10, 1, 3)
    assert [list(x) for x in sh] == [[1, 2, 3, 4], [5, 6, 7, 8], [9, 10, 0, 0]]


def test_flatten_groups_by_dtype_in_registration_order():
    # params of two dtype codes interleaved; each group keeps registration order
    a = np.array([1, 2], np.uint16).view(np.uint8)
    b = np.array([3.0], np.float32).view(np.uint8)
    c = np.array([4, 5, 6], np.uint16).view(np.uint8)
    params = [(b, 1, 1), (a, 2, 0), (c, 3, 0)]
    g0 = oracle.flatten_group(params, 0, 2).view(np.uint16)
    g1 = oracle.flatten_group(params, 1, 4).view(np.float32)
    assert list(g0) == [1, 2, 4, 5, 6]
    assert list(g1) == [3.0]


# closed forms of the shard lengths of the workloads: S_g = ceil(N_g / s)
# with N_bf16 = 12 d^2 (d = hidden, f = 4d) and N_f32 = 8 d.
@pytest.mark.parametrize("d,s,S_bf16,S_f32", [
    (256, 2, 393_216, 1_024),
    (1024, 3, 4_194_304, 2_731),
    (3840, 4, 44_236_800, 7_680),
    (6144, 2, 226_492_416, 24_576),
])
def test_workload_shard_lengths(d, s, S_bf16, S_f32):
    assert oracle.shard_numel(12 * d * d, s) == S_bf16
    assert oracle.shard_numel(8 * d, s) == S_f32


def test_odd_workload_shards_are_misaligned_to_16_bytes():
    # 3 shards of 2731 f32: 10924 bytes, 12 mod 16 -> shard 1 and 2 land at
    # non-16-byte-aligned offsets of the gathered buffer.
    S = oracle.shard_numel(8 * 1024, 3)
    assert S * 3 - 8 * 1024 == 1
    assert (S * 4) % 16 == 12


def test_slot_layout_bases_and_sizes():
    from layerwise_weight_offload_gb300 import workloads as W
    w = W.CONFIGS["odd"]
    descs = W.block_param_descs(w)
    numels = [int(np.prod(sh)) for _, sh, _ in descs]
    dtypes = [c for _, _, c in descs]
    esizes = [W.ESIZE[c] for c in dtypes]
    gdt, gbase, used = oracle.slot_layout(numels, dtypes, esizes, w.shards, 256)
    # groups in order of first appearance: f32 (norm1.weight comes first), bf16
    assert gdt == [W.F32, W.BF16]
    assert gbase[0] == 0
    f32_bytes = 3 * 2731 * 4
    assert gbase[1] == (f32_bytes + 255) // 256 * 256
    assert used == gbase[1] + 3 * 4_194_304 * 2
    assert all(b % 256 == 0 for b in gbase)


def test_slot_image_round_trip_small():
    rng = np.random.default_rng(7)
    numels = [5, 7, 3, 11]
    dtypes = [1, 0, 1, 0]
    esizes = [4, 2, 4, 2]
    raw = [rng.integers(1, 256, size=n * e, dtype=np.uint8) for n, e in zip(numels, esizes)]
    for s in range(1, 6):
        image, gdt, gbase, used = oracle.slot_image(raw, numels, dtypes, esizes, s, 16)
        # group 1 (code 1, f32) holds params 0 and 2 back to back
        f32 = np.concatenate([raw[0], raw[2]])
        assert np.array_equal(image[gbase[0]:gbase[0] + len(f32)], f32)
        bf = np.concatenate([raw[1], raw[3]])
        assert np.array_equal(image[gbase[1]:gbase[1] + len(bf)], bf)


# ---------------------------------------------------------------- schedule

def test_schedule_matches_hand_derived_golden():
    got = oracle.schedule(3, 2)[:, :6].tolist()
    assert got == _rows("schedule_n3_steps2.txt")


@pytest.mark.parametrize("n", range(1, 10))
@pytest.mark.parametrize("steps", range(1, 5))
def test_schedule_closed_form_and_invariants(n, steps):
    ev = oracle.schedule(n, steps)
    for row in ev:
        k, blk, rs, pb, ps, waits, viol = row.tolist()
        assert blk == k % n
        assert rs == k % 2                 # i%2 plus correction == global parity
        assert ps == 1 - rs                # only two slots, never the one read
        assert pb == (blk + 1) % n         # circular tail -> head prefetch
        assert waits == (k - 1 if k > 0 else -1)
        assert viol == 0


@pytest.mark.parametrize("n", [3, 5, 7, 9])
def test_odd_count_collides_without_correction(n):
    # The pages: without _prefetched_slot tracking, the circular tail->head
    # prefetch collides with the head's read slot for odd block counts.
    ev = oracle.schedule(n, 2, use_correction=False)
    assert (ev[:n, 6] == 0).all()          # first pass: i%2 alone is right
    assert (ev[n:, 6] != 0).any()          # second pass: collision


@pytest.mark.parametrize("n", [2, 4, 8])
def test_even_count_needs_no_correction(n):
    a = oracle.schedule(n, 3, use_correction=False)
    b = oracle.schedule(n, 3, use_correction=True)
    assert np.array_equal(a, b)
    assert (a[:, 6] == 0).all()


def test_at_most_two_blocks_resident():
    for n in range(1, 10):
        ev = oracle.schedule(n, 3)
        holds = {0: 0, 1: None}
        for row in ev:
            _, blk, rs, pb, ps, _, _ = row.tolist()
            assert holds[rs] == blk
            holds[ps] = pb
            assert len([v for v in holds.values() if v is not None]) <= 2


# ---------------------------------------------------------------- block math

def test_gelu_array_is_the_scalar_gelu_element_by_element():
    z = np.random.default_rng(40).standard_normal((7, 13)) * 4
    got = oracle.gelu_tanh_array(z)
    assert got.shape == z.shape
    assert all(got.flat[i] == oracle.gelu_tanh(float(z.flat[i])) for i in range(z.size))


def test_gelu_tanh_close_to_erf_gelu_and_odd_identity():
    for z in np.linspace(-8, 8, 1601):
        exact = 0.5 * z * (1 + math.erf(z / math.sqrt(2)))
        g = oracle.gelu_tanh(z)
        assert abs(g - exact) < 5e-4           # published accuracy of the tanh form
        # tanh is odd, so gelu(z) - gelu(-z) = z exactly (up to rounding)
        assert abs(g - oracle.gelu_tanh(-z) - z) < 1e-12 * max(1, abs(z))
    assert oracle.gelu_tanh(0.0) == 0.0


def test_rmsnorm_closed_forms():
    d = 7
    one = np.ones(d, np.float32)
    zero = np.zeros(d, np.float32)
    x = np.full((1, d), 3.0)
    h = oracle.rmsnorm_mod(x, one, zero, zero, eps=1e-6)
    assert np.allclose(h, 3.0 / math.sqrt(9.0 + 1e-6), rtol=0, atol=1e-15)
    # scale = -1 or gain = 0 leaves only the shift
    shift = np.arange(d, dtype=np.float32)
    rng = np.random.default_rng(0)
    xr = rng.standard_normal((4, d))
    assert np.array_equal(oracle.rmsnorm_mod(xr, one, shift, -one), np.tile(shift, (4, 1)))
    assert np.array_equal(oracle.rmsnorm_mod(xr, zero, shift, zero), np.tile(shift, (4, 1)))
    # eps = 0: invariant to scaling the row; unit mean square
    h1 = oracle.rmsnorm_mod(xr, one, zero, zero, eps=0.0)
    h2 = oracle.rmsnorm_mod(5.0 * xr, one, zero, zero, eps=0.0)
    assert np.allclose(h1, h2, atol=1e-13)
    assert np.allclose((h1 ** 2).mean(axis=1), 1.0, atol=1e-13)
    # scale doubles the normalised row: (1 + 1)
    h3 = oracle.rmsnorm_mod(xr, one, zero, one, eps=0.0)
    assert np.allclose(h3, 2 * h1, atol=1e-13)


@pytest.mark.parametrize("rows,k,n", [(1, 1, 1), (3, 5, 7), (17, 33, 9), (64, 48, 80)])
def test_linear_against_numpy_matmul(rows, k, n):
    rng = np.random.default_rng(rows * 100 + n)
    a = rng.standard_normal((rows, k))
    w = rng.standard_normal((n, k)).astype(np.float32)
    y = oracle.linear(a, w, threads=3)
    assert np.allclose(y, a @ w.astype(np.float64).T, rtol=1e-12, atol=1e-12)


def _qkv(rng, b, t, d):
    return rng.standard_normal((b * t, 3 * d))


def test_attention_zero_queries_average_values():
    rng = np.random.default_rng(3)
    b, t, d, h = 2, 9, 8, 2
    qkv = _qkv(rng, b, t, d)
    qkv[:, :d] = 0.0
    o = oracle.attention(qkv, b, t, d, h)
    v = qkv[:, 2 * d:].reshape(b, t, d)
    assert np.allclose(o.reshape(b, t, d), v.mean(axis=1, keepdims=True).repeat(t, 1), atol=1e-14)


def test_attention_single_token_returns_value():
    rng = np.random.default_rng(4)
    qkv = _qkv(rng, 3, 1, 16)
    o = oracle.attention(qkv, 3, 1, 16, 4)
    assert np.allclose(o, qkv[:, 32:], atol=0)


def test_attention_two_tokens_sigmoid_closed_form():
    # one head of dim 4 -> scale 1/2; softmax over two scores = sigmoid(s0-s1)
    d = 4
    qkv = np.zeros((2, 3 * d))
    qkv[0, :d] = [1, 0, 0, 0]
    qkv[1, :d] = [0, 2, 0, 0]
    qkv[0, d:2 * d] = [3, 1, 0, 0]         # k0
    qkv[1, d:2 * d] = [-1, 2, 0, 0]        # k1
    qkv[0, 2 * d:] = [1, 2, 3, 4]          # v0
    qkv[1, 2 * d:] = [-4, 0, 1, 2]         # v1
    o = oracle.attention(qkv, 1, 2, d, 1)
    for t, (s0, s1) in enumerate([(3 * 0.5, -1 * 0.5), (2 * 0.5, 4 * 0.5)]):
        p0 = 1.0 / (1.0 + math.exp(-(s0 - s1)))
        expect = p0 * qkv[0, 2 * d:] + (1 - p0) * qkv[1, 2 * d:]
        assert np.allclose(o[t], expect, atol=1e-14)


def test_attention_permutations_and_head_independence():
    rng = np.random.default_rng(5)
    b, t, d, h = 1, 12, 16, 4
    qkv = _qkv(rng, b, t, d)
    o = oracle.attention(qkv, b, t, d, h)
    perm = rng.permutation(t)
    # permuting tokens permutes the output rows (no positions, non-causal)
    op = oracle.attention(qkv[perm], b, t, d, h)
    assert np.allclose(op, o[perm], atol=1e-13)
    # changing head 1's q, k and v leaves the other heads' columns unchanged
    hd = d // h
    q2 = qkv.copy()
    for base in (0, d, 2 * d):
        q2[:, base + hd:base + 2 * hd] = rng.standard_normal((t, hd))
    o2 = oracle.attention(q2, b, t, d, h)
    keep = [c for c in range(d) if not hd <= c < 2 * hd]
    assert np.allclose(o2[:, keep], o[:, keep], atol=0)
    assert not np.allclose(o2[:, hd:2 * hd], o[:, hd:2 * hd])


def test_attention_batch_items_are_independent():
    rng = np.random.default_rng(6)
    t, d = 5, 8
    qkv = _qkv(rng, 2, t, d)
    o = oracle.attention(qkv, 2, t, d, 2)
    o0 = oracle.attention(qkv[:t], 1, t, d, 2)
    assert np.allclose(o[:t], o0, atol=0)


def _params(rng, d, f):
    p = {}
    for name in oracle.PARAM_ORDER:
        if name.startswith("norm"):
            p[name] = np.ones(d, np.float32)
        elif name.startswith("ada"):
            p[name] = (0.1 * rng.standard_normal(d)).astype(np.float32)
    p["attn.qkv.weight"] = (0.02 * rng.standard_normal((3 * d, d))).astype(np.float32)
    p["attn.out.weight"] = (0.02 * rng.standard_normal((d, d))).astype(np.float32)
    p["mlp.fc1.weight"] = (0.02 * rng.standard_normal((f, d))).astype(np.float32)
    p["mlp.fc2.weight"] = (0.02 * rng.standard_normal((d, f))).astype(np.float32)
    return p


def test_block_zero_gates_is_identity():
    rng = np.random.default_rng(8)
    d, f, t = 16, 64, 6
    p = _params(rng, d, f)
    p["ada1.gate"][:] = 0
    p["ada2.gate"][:] = 0
    x = rng.standard_normal((t, d)).astype(np.float32)
    y = oracle.block_forward(x, p, 1, t, d, 4, f)
    assert np.array_equal(y, x.astype(np.float64))


def _perm_matrix(perm):
    m = np.zeros((len(perm), len(perm)), np.float32)
    m[np.arange(len(perm)), perm] = 1.0
    return m


def test_block_attention_branch_closed_form():
    # Wq = Wk = 0 -> uniform attention; Wv, Wo permutations; MLP gated off.
    rng = np.random.default_rng(9)
    d, f, t, heads = 12, 48, 5, 3
    p = _params(rng, d, f)
    pv, po = rng.permutation(d), rng.permutation(d)
    w = np.zeros((3 * d, d), np.float32)
    w[2 * d:] = _perm_matrix(pv)
    p["attn.qkv.weight"] = w
    p["attn.out.weight"] = _perm_matrix(po)
    p["ada2.gate"][:] = 0
    x = rng.standard_normal((t, d)).astype(np.float32)
    y = oracle.block_forward(x, p, 1, t, d, heads, f)
    h = oracle.rmsnorm_mod(x.astype(np.float64), p["norm1.weight"], p["ada1.shift"], p["ada1.scale"])
    v = h[:, pv]                                # y = h W^T with W a permutation
    o = np.tile(v.mean(axis=0), (t, 1))         # uniform attention
    expect = x + p["ada1.gate"] * o[:, po]
    assert np.allclose(y, expect, atol=1e-13)


def test_block_mlp_branch_closed_form():
    # attention gated off; W1's first d rows a permutation, rest zero;
    # W2's first d columns a permutation, rest zero.
    rng = np.random.default_rng(10)
    d, f, t = 8, 32, 4
    p = _params(rng, d, f)
    p["ada1.gate"][:] = 0
    p1, p2 = rng.permutation(d), rng.permutation(d)
    w1 = np.zeros((f, d), np.float32)
    w1[:d] = _perm_matrix(p1)
    w2 = np.zeros((d, f), np.float32)
    w2[:, :d] = _perm_matrix(p2)
    p["mlp.fc1.weight"], p["mlp.fc2.weight"] = w1, w2
    x = (3 * rng.standard_normal((t, d))).astype(np.float32)
    y = oracle.block_forward(x, p, 1, t, d, 2, f)
    h2 = oracle.rmsnorm_mod(x.astype(np.float64), p["norm2.weight"], p["ada2.shift"], p["ada2.scale"])
    u = np.vectorize(oracle.gelu_tanh)(h2[:, p1])
    expect = x + p["ada2.gate"] * u[:, p2]
    assert np.allclose(y, expect, atol=1e-13)


def _np_rmsnorm_mod(x, g, shift, scale, eps=1e-6):
    """RMSNorm with adaLN modulation written out in numpy."""
    x = np.asarray(x, dtype=np.float64)
    inv = 1.0 / np.sqrt((x * x).mean(axis=1, keepdims=True) + eps)
    f = lambda a: np.asarray(a, dtype=np.float64)
    return x * inv * f(g) * (1.0 + f(scale)) + f(shift)


def _np_gelu_tanh(z):
    return 0.5 * z * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (z + 0.044715 * z ** 3)))


def _both_branch_weights(rng, p, d, f):
    """Wq = Wk = 0 (uniform attention), Wv, Wo, W1's first d rows and W2's
    first d columns permutations, every other weight zero."""
    pv, po, p1, p2 = (rng.permutation(d) for _ in range(4))
    w = np.zeros((3 * d, d), np.float32)
    w[2 * d:] = _perm_matrix(pv)
    w1 = np.zeros((f, d), np.float32)
    w1[:d] = _perm_matrix(p1)
    w2 = np.zeros((d, f), np.float32)
    w2[:, :d] = _perm_matrix(p2)
    p["attn.qkv.weight"], p["attn.out.weight"] = w, _perm_matrix(po)
    p["mlp.fc1.weight"], p["mlp.fc2.weight"] = w1, w2
    return pv, po, p1, p2


def test_block_both_branches_closed_form_mlp_reads_the_updated_residual():
    # Both branches on at once.  Attention is uniform per batch item (q = k =
    # 0), so o is the item's mean of v = h[:, pv]; the MLP's RMSNorm must read
    # the residual AFTER the attention update, x1 = x + gate1 * o Wo^T.  The
    # expected value is written out in numpy; a block whose MLP normalised
    # the block input (parallel branches) differs from it by far more than
    # the tolerance, which the second assertion checks.
    rng = np.random.default_rng(30)
    d, f, t, heads, batch = 8, 32, 5, 2, 2
    p = _params(rng, d, f)
    p["ada1.gate"] = (0.5 + rng.random(d)).astype(np.float32)
    p["ada2.gate"] = (0.5 + rng.random(d)).astype(np.float32)
    pv, po, p1, p2 = _both_branch_weights(rng, p, d, f)
    x = (2 * rng.standard_normal((batch * t, d))).astype(np.float32)
    y = oracle.block_forward(x, p, batch, t, d, heads, f)
    xd = x.astype(np.float64)
    h = _np_rmsnorm_mod(xd, p["norm1.weight"], p["ada1.shift"], p["ada1.scale"])
    v = h[:, pv]
    o = np.concatenate([np.tile(v[i * t:(i + 1) * t].mean(axis=0), (t, 1))
                        for i in range(batch)])
    x1 = xd + p["ada1.gate"].astype(np.float64) * o[:, po]
    h2 = _np_rmsnorm_mod(x1, p["norm2.weight"], p["ada2.shift"], p["ada2.scale"])
    expect = x1 + p["ada2.gate"].astype(np.float64) * _np_gelu_tanh(h2[:, p1])[:, p2]
    assert np.allclose(y, expect, atol=1e-12, rtol=0)
    h2_par = _np_rmsnorm_mod(xd, p["norm2.weight"], p["ada2.shift"], p["ada2.scale"])
    parallel = x1 + p["ada2.gate"].astype(np.float64) * _np_gelu_tanh(h2_par[:, p1])[:, p2]
    assert np.abs(parallel - expect).max() > 1e-3


def test_full_block_both_branches_closed_form_with_biases():
    # The checkpoint-shaped block with both branches on: q = k = 0 (zero
    # weights and zero q/k biases, so the q/k norm and RoPE leave zeros and
    # attention is uniform), v = h[:, pv] + bv, out = o Wo^T + bo, and the
    # MLP with its biases on the updated residual x1; written out in numpy.
    rng = np.random.default_rng(31)
    d, f, t, heads = 8, 32, 6, 2
    p = _params(rng, d, f)
    p.update(_extras(rng, d, f, d // heads))
    p["attn.qkv.bias"][:2 * d] = 0
    p["ada1.gate"] = (0.5 + rng.random(d)).astype(np.float32)
    p["ada2.gate"] = (0.5 + rng.random(d)).astype(np.float32)
    pv, po, p1, p2 = _both_branch_weights(rng, p, d, f)
    x = (2 * rng.standard_normal((t, d))).astype(np.float32)
    y = oracle.block_forward(x, p, 1, t, d, heads, f, rope_base=10000.0)
    b = {k: p[k].astype(np.float64) for k in
         ("attn.qkv.bias", "attn.out.bias", "mlp.fc1.bias", "mlp.fc2.bias")}
    xd = x.astype(np.float64)
    h = _np_rmsnorm_mod(xd, p["norm1.weight"], p["ada1.shift"], p["ada1.scale"])
    v = h[:, pv] + b["attn.qkv.bias"][2 * d:]
    o = np.tile(v.mean(axis=0), (t, 1))
    x1 = xd + p["ada1.gate"].astype(np.float64) * (o[:, po] + b["attn.out.bias"])
    h2 = _np_rmsnorm_mod(x1, p["norm2.weight"], p["ada2.shift"], p["ada2.scale"])
    u = np.zeros((t, f))
    u[:, :d] = h2[:, p1]
    u = _np_gelu_tanh(u + b["mlp.fc1.bias"])
    expect = x1 + p["ada2.gate"].astype(np.float64) * (u[:, :d][:, p2] + b["mlp.fc2.bias"])
    assert np.allclose(y, expect, atol=1e-12, rtol=0)


def test_block_token_permutation_equivariance_and_batch():
    rng = np.random.default_rng(11)
    d, f, t = 16, 64, 7
    p = _params(rng, d, f)
    x = rng.standard_normal((2 * t, d)).astype(np.float32)
    y = oracle.block_forward(x, p, 2, t, d, 4, f)
    perm = rng.permutation(t)
    xp = x.copy()
    xp[:t] = x[:t][perm]
    yp = oracle.block_forward(xp, p, 2, t, d, 4, f)
    assert np.allclose(yp[:t], y[:t][perm], atol=1e-12)
    assert np.allclose(yp[t:], y[t:], atol=0)


def test_block_rows_equals_full_block_on_listed_rows():
    # the sampled-rows form must reproduce the full forward's rows exactly
    rng = np.random.default_rng(12)
    d, f, t = 16, 64, 9
    p = _params(rng, d, f)
    x = rng.standard_normal((2 * t, d)).astype(np.float32)
    full = oracle.block_forward(x, p, 2, t, d, 4, f, threads=3)
    rows = [0, 5, 8, 9, 17]
    part = oracle.block_forward_rows(x, p, rows, 2, t, d, 4, f, threads=3)
    assert np.array_equal(part, full[rows])


# ---- strided views packed in physical order ([D5] "Request and loading
# constraints") ------------------------------------------------------------

def _random_view(rng):
    ndim = int(rng.integers(1, 5))
    shape = [int(v) for v in rng.integers(1, 6, size=ndim)]
    strides = [int(v) for v in rng.integers(0, 40, size=ndim)]
    return shape, strides


@pytest.mark.parametrize("seed", range(30))
def test_storage_extent_matches_numpy_byte_bounds(seed):
    # independent pin: numpy's own bounds of an as_strided view over a buffer
    rng = np.random.default_rng(seed)
    shape, strides = _random_view(rng)
    base = np.zeros(4096, dtype=np.uint8)
    view = np.lib.stride_tricks.as_strided(base, shape=shape, strides=strides)
    lo, hi = np.lib.array_utils.byte_bounds(view)
    assert oracle.storage_extent(shape, strides) == hi - lo


def test_storage_extent_of_contiguous_and_transposed():
    assert oracle.storage_extent([7, 5], [5, 1]) == 35
    assert oracle.storage_extent([5, 7], [1, 5]) == 35           # its transpose
    assert oracle.storage_extent([3, 4, 2], [8, 2, 1]) == 24
    assert oracle.storage_extent([6], [3]) == 16                  # every third
    assert oracle.storage_extent([4, 3], [0, 1]) == 3             # broadcast rows


@pytest.mark.parametrize("esize", [1, 2, 4])
def test_transposed_view_survives_physical_order_packing(esize):
    # pack the storage of a transposed view, shard and reassemble it, then the
    # same strides over the gathered bytes give the view back
    rng = np.random.default_rng(esize)
    a = rng.integers(0, 256, size=(9, 13 * esize), dtype=np.uint8)    # [m, n] rows
    m, n = 9, 13
    t_shape, t_strides = (n, m), (1, n)                                 # elements
    ext = oracle.storage_extent(t_shape, t_strides)
    assert ext == m * n
    flat = oracle.flatten_group([(a.reshape(-1), ext, 5)], 5, esize)
    for s in (1, 2, 3, 5):
        shards = oracle.shard(flat, ext, esize, s)
        gathered = oracle.reassemble(shards, oracle.shard_numel(ext, s), esize)
        back = np.lib.stride_tricks.as_strided(
            gathered, shape=(n, m, esize),
            strides=(t_strides[0] * esize, t_strides[1] * esize, 1))
        want = a.reshape(m, n, esize).transpose(1, 0, 2)
        assert np.array_equal(back, want)


# ---- the checkpoint-shaped block: biases, per-head q/k RMSNorm, rotary
# embedding (readings stated in the oracle; RoPE after Su et al., RoFormer) --

def test_rope_two_dims_is_a_rotation_by_the_position():
    # hd = 2: one pair, frequency base^0 = 1, so the token at position p is
    # rotated by p radians, q and k alike; v is untouched
    t = 5
    qkv = np.zeros((t, 6))
    qkv[:, 0], qkv[:, 2], qkv[:, 3], qkv[:, 4] = 1.0, 2.0, -1.0, 7.0
    r = oracle.rope(qkv, 1, t, 2, 1, 10000.0)
    p = np.arange(t)
    assert np.allclose(r[:, 0], np.cos(p), atol=1e-15) and np.allclose(r[:, 1], np.sin(p), atol=1e-15)
    # k = (2, -1): (2 cos + sin, 2 sin - cos)
    assert np.allclose(r[:, 2], 2 * np.cos(p) + np.sin(p), atol=1e-14)
    assert np.allclose(r[:, 3], 2 * np.sin(p) - np.cos(p), atol=1e-14)
    assert np.array_equal(r[:, 4:], qkv[:, 4:])


def test_rope_frequencies_and_positions_per_batch_item():
    # hd = 4: pair i rotates by p * base^(-2i/4); positions restart at 0 in
    # every batch item (its first token is unrotated)
    base, t = 10000.0, 4
    qkv = np.zeros((2 * t, 12))
    qkv[:, 0:4] = [1.0, 0.0, 1.0, 0.0]
    r = oracle.rope(qkv, 2, t, 4, 1, base)
    for row in range(2 * t):
        p = row % t
        for i in range(2):
            ang = p * base ** (-2.0 * i / 4)
            assert abs(r[row, 2 * i] - math.cos(ang)) < 1e-14
            assert abs(r[row, 2 * i + 1] - math.sin(ang)) < 1e-14
    assert np.array_equal(r[t], qkv[t])


def test_rope_preserves_pair_norms_and_depends_on_relative_position():
    rng = np.random.default_rng(21)
    t, d, heads = 9, 16, 2
    hd = d // heads
    qkv = rng.standard_normal((t, 3 * d))
    r = oracle.rope(qkv, 1, t, d, heads, 10000.0)
    pair = lambda a: a[:, :2 * d].reshape(t, -1, 2)
    assert np.allclose(np.linalg.norm(pair(r), axis=2), np.linalg.norm(pair(qkv), axis=2),
                       atol=1e-12)
    # the same q and k at every position: rotated q_m . k_n depends on n - m only
    same = np.tile(rng.standard_normal((1, 3 * d)), (t, 1))
    rs = oracle.rope(same, 1, t, d, heads, 10000.0)
    dot = lambda m, n, j: rs[m, j * hd:(j + 1) * hd] @ rs[n, d + j * hd:d + (j + 1) * hd]
    for j in range(heads):
        for m, n in [(3, 5), (1, 7), (6, 2)]:
            assert abs(dot(m, n, j) - dot(0, n - m, j) if n >= m else
                       dot(m, n, j) - dot(m - n, 0, j)) < 1e-12


def test_qk_norm_per_head_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(22)
    t, d, heads = 5, 24, 3
    hd = d // heads
    qkv = rng.standard_normal((t, 3 * d))
    qkv[:, :hd] *= 50.0                            # heads normalised separately
    ones = np.ones(hd, np.float32)
    r = oracle.qk_norm(qkv, d, heads, ones, ones, eps=0.0)
    for part in range(2):
        for j in range(heads):
            v = r[:, part * d + j * hd:part * d + (j + 1) * hd]
            assert np.allclose((v ** 2).mean(axis=1), 1.0, atol=1e-13)
    assert np.array_equal(r[:, 2 * d:], qkv[:, 2 * d:])
    r2 = oracle.qk_norm(3.5 * qkv, d, heads, ones, ones, eps=0.0)
    assert np.allclose(r2[:, :2 * d], r[:, :2 * d], atol=1e-13)
    g = (1 + rng.standard_normal(hd)).astype(np.float32)
    gk = (1 + rng.standard_normal(hd)).astype(np.float32)
    rg = oracle.qk_norm(qkv, d, heads, g, gk, eps=0.0)
    for j in range(heads):
        assert np.allclose(rg[:, j * hd:(j + 1) * hd], r[:, j * hd:(j + 1) * hd] * g, atol=1e-13)
        assert np.allclose(rg[:, d + j * hd:d + (j + 1) * hd],
                           r[:, d + j * hd:d + (j + 1) * hd] * gk, atol=1e-13)


def _extras(rng, d, f, hd):
    return {"attn.qkv.bias": (0.02 * rng.standard_normal(3 * d)).astype(np.float32),
            "attn.out.bias": (0.02 * rng.standard_normal(d)).astype(np.float32),
            "mlp.fc1.bias": (0.02 * rng.standard_normal(f)).astype(np.float32),
            "mlp.fc2.bias": (0.02 * rng.standard_normal(d)).astype(np.float32),
            "attn.q_norm.weight": (1 + 0.1 * rng.standard_normal(hd)).astype(np.float32),
            "attn.k_norm.weight": (1 + 0.1 * rng.standard_normal(hd)).astype(np.float32)}


def test_full_block_with_zero_weights_adds_the_gated_biases():
    # every weight zero: attention mixes equal values (v = bv for every
    # token), so o = bv and the out-projection gives bo; the MLP gives b2:
    # x_out = x + gate1 * bo + gate2 * b2 exactly, with q/k norm and RoPE on
    rng = np.random.default_rng(23)
    d, f, t, heads = 16, 64, 6, 2
    p = _params(rng, d, f)
    for k in ("attn.qkv.weight", "attn.out.weight", "mlp.fc1.weight", "mlp.fc2.weight"):
        p[k][:] = 0
    p.update(_extras(rng, d, f, d // heads))
    x = rng.standard_normal((2 * t, d)).astype(np.float32)
    y = oracle.block_forward(x, p, 2, t, d, heads, f, rope_base=10000.0)
    g1, g2 = p["ada1.gate"].astype(np.float64), p["ada2.gate"].astype(np.float64)
    x1 = x.astype(np.float64) + g1 * p["attn.out.bias"].astype(np.float64)
    expect = x1 + g2 * p["mlp.fc2.bias"].astype(np.float64)
    assert np.allclose(y, expect, atol=1e-15)


def test_full_block_attention_branch_closed_form_with_norm_and_rope():
    # Wq = Wk = 0 with q/k biases: after the q/k norm and RoPE the scores are
    # computed from the rotated bias vectors; against that attention written
    # out here in numpy, with v a permutation of h and Wo a permutation
    rng = np.random.default_rng(24)
    d, f, t, heads = 8, 32, 5, 2
    hd = d // heads
    p = _params(rng, d, f)
    p.update(_extras(rng, d, f, hd))
    pv, po = rng.permutation(d), rng.permutation(d)
    w = np.zeros((3 * d, d), np.float32)
    w[2 * d:] = _perm_matrix(pv)
    p["attn.qkv.weight"] = w
    p["attn.out.weight"] = _perm_matrix(po)
    p["ada2.gate"][:] = 0
    x = rng.standard_normal((t, d)).astype(np.float32)
    y = oracle.block_forward(x, p, 1, t, d, heads, f, rope_base=100.0)
    h = oracle.rmsnorm_mod(x.astype(np.float64), p["norm1.weight"], p["ada1.shift"], p["ada1.scale"])
    b = p["attn.qkv.bias"].astype(np.float64)
    o = np.zeros((t, d))
    for j in range(heads):
        def prep(vec, g, pos):
            v = vec / np.sqrt((vec ** 2).mean() + 1e-6) * g.astype(np.float64)
            out = v.copy()
            for i in range(hd // 2):
                ang = pos * 100.0 ** (-2.0 * i / hd)
                out[2 * i] = v[2 * i] * math.cos(ang) - v[2 * i + 1] * math.sin(ang)
                out[2 * i + 1] = v[2 * i] * math.sin(ang) + v[2 * i + 1] * math.cos(ang)
            return out
        qb, kb = b[j * hd:(j + 1) * hd], b[d + j * hd:d + (j + 1) * hd]
        vv = h[:, pv][:, j * hd:(j + 1) * hd] + b[2 * d + j * hd:2 * d + (j + 1) * hd]
        for tq in range(t):
            q = prep(qb, p["attn.q_norm.weight"], tq)
            s = np.array([q @ prep(kb, p["attn.k_norm.weight"], u) for u in range(t)]) / math.sqrt(hd)
            wgt = np.exp(s - s.max())
            o[tq, j * hd:(j + 1) * hd] = (wgt[:, None] * vv).sum(axis=0) / wgt.sum()
    expect = x + p["ada1.gate"] * (o[:, po] + p["attn.out.bias"])
    assert np.allclose(y, expect, atol=1e-12)


def test_full_block_without_extras_equals_plain_block():
    rng = np.random.default_rng(25)
    d, f, t = 16, 64, 5
    p = _params(rng, d, f)
    x = rng.standard_normal((t, d)).astype(np.float32)
    # the extended entry point itself, every extra absent (null pointers)
    arrs = [np.ascontiguousarray(p[n], dtype=np.float32) for n in oracle.PARAM_ORDER]
    ptrs = (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    out = np.zeros((t, d), dtype=np.float64)
    oracle.lib().oracle_block_forward_ex(x.ctypes.data, 1, t, d, 4, f, 1e-6, ptrs, None, None,
                                         None, None, None, None, 0.0, out.ctypes.data, 2)
    assert np.array_equal(out, oracle.block_forward(x, p, 1, t, d, 4, f))


_ALL_EXTRAS = ("attn.qkv.bias", "attn.out.bias", "mlp.fc1.bias", "mlp.fc2.bias",
               "attn.q_norm.weight", "attn.k_norm.weight")


@pytest.mark.parametrize("keep,rope", [
    (_ALL_EXTRAS, 10000.0), (_ALL_EXTRAS, 0.0),
    (("attn.qkv.bias", "mlp.fc2.bias"), 10000.0), (("attn.qkv.bias", "mlp.fc2.bias"), 0.0),
    (("attn.q_norm.weight", "attn.k_norm.weight"), 10000.0),
    (("attn.q_norm.weight", "attn.k_norm.weight"), 0.0),
    ((), 10000.0),
])
def test_full_block_rows_equals_full_block_on_listed_rows(keep, rope):
    # the checkpoint-shaped block's sampled-rows form reproduces the full
    # forward's rows exactly, with any subset of the additions; two batch
    # items, so the rotation's positions restart (rows 9 and 17 are tokens 0
    # and 8 of the second item)
    rng = np.random.default_rng(29)
    d, f, t, heads = 16, 64, 9, 4
    p = _params(rng, d, f)
    p.update({k: v for k, v in _extras(rng, d, f, d // heads).items() if k in keep})
    x = rng.standard_normal((2 * t, d)).astype(np.float32)
    full = oracle.block_forward(x, p, 2, t, d, heads, f, threads=3, rope_base=rope)
    rows = [0, 5, 8, 9, 17]
    part = oracle.block_forward_rows(x, p, rows, 2, t, d, heads, f, threads=3, rope_base=rope)
    assert np.array_equal(part, full[rows])
    # the additions matter at these values: the plain block differs
    plain = {k: v for k, v in p.items() if k not in keep}
    assert not np.allclose(oracle.block_forward(x, plain, 2, t, d, heads, f), full, atol=1e-6)
    assert np.array_equal(part, oracle.block_forward_rows(x, p, rows, 2, t, d, heads, f,
                                                          threads=1, rope_base=rope))
