"""Helpers shared by the tests (no method arithmetic here)."""
import numpy as np
import torch


def build_lib():
    from layerwise_weight_offload_gb300 import build
    return build.build()


def bf16_to_f32(t):
    """Exact widening of a bf16 tensor to float32 numpy."""
    return t.detach().float().cpu().numpy()


def params_f32(params):
    return {k: bf16_to_f32(v) for k, v in params.items()}


def raw_bytes(t):
    t = t.detach().contiguous().cpu()
    return t.view(torch.uint8).numpy().reshape(-1)


def assert_oracle_close(gpu, ref, what="", max_rel=2e-2, mean_rel=5e-3):
    """The acceptance bar: max|gpu-ref| <= max_rel * max|ref| and
    mean|gpu-ref| / mean|ref| <= mean_rel."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.isfinite(gpu).all(), what + ": non-finite GPU values"
    err = np.abs(gpu - ref)
    mx = float(err.max()) if err.size else 0.0
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    mean_err = float(err.mean()) if err.size else 0.0
    mean_ref = float(np.abs(ref).mean()) if ref.size else 0.0
    assert mx <= max_rel * scale + 1e-30, "%s: max err %.3e > %.1e * %.3e" % (what, mx, max_rel, scale)
    assert mean_err <= mean_rel * mean_ref + 1e-30, \
        "%s: mean err %.3e > %.1e * %.3e" % (what, mean_err, mean_rel, mean_ref)
    return mx / max(scale, 1e-30), mean_err / max(mean_ref, 1e-30)


def assert_only_groups_written(got, groups, shards, fill, where=""):
    """Canary check of a slot: every byte outside the groups' gathered ranges
    (the gaps up to each 256-aligned group base, and past the last group)
    still holds the fill pattern."""
    got = np.asarray(got)
    mask = np.zeros(got.size, dtype=bool)
    for g in groups:
        mask[g.base:g.base + shards * g.shard_bytes] = True
    bad = np.nonzero((~mask) & (got != fill))[0]
    assert bad.size == 0, "%s: %d bytes outside the groups written, first at %d" % (
        where, bad.size, int(bad[0]))
