"""CPU oracle for the DLO block stream — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``dlo_oracle.cpp`` (a plain
fp64 C++ statement of the method) through ctypes and shares no code with the
CUDA library.  See ``dlo_oracle.cpp`` for the cited passages and readings.
"""
import ctypes
import os

import numpy as np

from .build_oracle import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build()
        L = ctypes.CDLL(path)
        i32, i64, vp, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
        L.oracle_shard_numel.restype = i64
        L.oracle_shard_numel.argtypes = [i64, i32]
        L.oracle_storage_extent.restype = i64
        L.oracle_storage_extent.argtypes = [i32, vp, vp]
        L.oracle_flatten_group.restype = i64
        L.oracle_flatten_group.argtypes = [vp, vp, vp, i32, i32, i32, vp]
        L.oracle_shard.restype = None
        L.oracle_shard.argtypes = [vp, i64, i32, i32, vp]
        L.oracle_reassemble.restype = None
        L.oracle_reassemble.argtypes = [vp, i64, i32, i32, vp]
        L.oracle_slot_layout.restype = i64
        L.oracle_slot_layout.argtypes = [vp, vp, vp, i32, i32, i64, vp, vp, vp]
        L.oracle_schedule.restype = i32
        L.oracle_schedule.argtypes = [i32, i32, i32, vp]
        L.oracle_gelu_tanh.restype = dbl
        L.oracle_gelu_tanh.argtypes = [dbl]
        L.oracle_gelu_tanh_array.restype = None
        L.oracle_gelu_tanh_array.argtypes = [vp, i64, vp]
        L.oracle_rmsnorm_mod.restype = None
        L.oracle_rmsnorm_mod.argtypes = [vp, i64, i64, vp, vp, vp, dbl, vp]
        L.oracle_linear.restype = None
        L.oracle_linear.argtypes = [vp, i64, i64, vp, i64, vp, i32]
        L.oracle_attention.restype = None
        L.oracle_attention.argtypes = [vp, i64, i64, i64, i64, vp, i32]
        L.oracle_block_forward.restype = None
        L.oracle_block_forward.argtypes = [vp, i64, i64, i64, i64, i64, dbl, vp, vp, i32]
        L.oracle_qk_norm.restype = None
        L.oracle_qk_norm.argtypes = [vp, i64, i64, i64, vp, vp, dbl]
        L.oracle_rope.restype = None
        L.oracle_rope.argtypes = [vp, i64, i64, i64, i64, dbl]
        L.oracle_block_forward_ex.restype = None
        L.oracle_block_forward_ex.argtypes = [vp, i64, i64, i64, i64, i64, dbl, vp, vp, vp, vp,
                                              vp, vp, vp, dbl, vp, i32]
        L.oracle_block_forward_rows.restype = None
        L.oracle_block_forward_rows.argtypes = [vp, i64, i64, i64, i64, i64, dbl, vp, vp, i64,
                                                vp, i32]
        L.oracle_block_forward_ex_rows.restype = None
        L.oracle_block_forward_ex_rows.argtypes = [vp, i64, i64, i64, i64, i64, dbl, vp, vp, vp,
                                                   vp, vp, vp, vp, dbl, vp, i64, vp, i32]
        _lib = L
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _ptr_array(arrs):
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def default_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---- sharding ------------------------------------------------------------

def shard_numel(total_numel, dp_size):
    return int(lib().oracle_shard_numel(total_numel, dp_size))


def storage_extent(shape, strides):
    """Elements packed for a view of these extents and element strides."""
    sh = np.asarray(shape, dtype=np.int64)
    st = np.asarray(strides, dtype=np.int64)
    return int(lib().oracle_storage_extent(len(sh), _ptr(sh), _ptr(st)))


def flatten_group(params, dtype_code, esize):
    """params: list of (uint8 ndarray of raw bytes, numel, dtype_code)."""
    sel = [p for p in params if p[2] == dtype_code]
    total = sum(p[1] for p in sel)
    out = np.zeros(total * esize, dtype=np.uint8)
    srcs = [np.ascontiguousarray(p[0]) for p in params]
    numels = np.array([p[1] for p in params], dtype=np.int64)
    dtypes = np.array([p[2] for p in params], dtype=np.int32)
    n = lib().oracle_flatten_group(_ptr_array(srcs), _ptr(numels), _ptr(dtypes),
                                   len(params), dtype_code, esize, _ptr(out))
    assert n == total
    return out


def shard(flat_bytes, numel, esize, dp_size):
    S = shard_numel(numel, dp_size)
    flat = np.ascontiguousarray(flat_bytes, dtype=np.uint8)
    outs = [np.full(S * esize, 0xCD, dtype=np.uint8) for _ in range(dp_size)]
    lib().oracle_shard(_ptr(flat), numel, esize, dp_size, _ptr_array(outs))
    return outs


def reassemble(shards, shard_numel_, esize):
    out = np.full(len(shards) * shard_numel_ * esize, 0xCD, dtype=np.uint8)
    srcs = [np.ascontiguousarray(s, dtype=np.uint8) for s in shards]
    lib().oracle_reassemble(_ptr_array(srcs), shard_numel_, esize, len(shards), _ptr(out))
    return out


def slot_layout(numels, dtypes, esizes, dp_size, align=256):
    n = len(numels)
    nu = np.asarray(numels, dtype=np.int64)
    dt = np.asarray(dtypes, dtype=np.int32)
    es = np.asarray(esizes, dtype=np.int32)
    gd = np.zeros(max(n, 1), dtype=np.int32)
    gb = np.zeros(max(n, 1), dtype=np.int64)
    ng = np.zeros(1, dtype=np.int32)
    used = lib().oracle_slot_layout(_ptr(nu), _ptr(dt), _ptr(es), n, dp_size, align,
                                    _ptr(gd), _ptr(gb), _ptr(ng))
    k = int(ng[0])
    return [int(x) for x in gd[:k]], [int(x) for x in gb[:k]], int(used)


def slot_image(param_bytes, numels, dtypes, esizes, dp_size, align=256):
    """Expected bytes of a slot holding one block: for every dtype group, the
    flat group sharded and reassembled in rank order at the group's base."""
    gdt, gbase, used = slot_layout(numels, dtypes, esizes, dp_size, align)
    image = np.zeros(used, dtype=np.uint8)
    params = list(zip(param_bytes, numels, dtypes))
    for g, (code, base) in enumerate(zip(gdt, gbase)):
        es = [e for e, d in zip(esizes, dtypes) if d == code][0]
        flat = flatten_group(params, code, es)
        n = len(flat) // es
        sh = shard(flat, n, es, dp_size)
        gathered = reassemble(sh, shard_numel(n, dp_size), es)
        image[base:base + len(gathered)] = gathered
    return image, gdt, gbase, used


# ---- schedule ------------------------------------------------------------

SCHED_FIELDS = ("k", "block", "read_slot", "prefetch_block", "prefetch_slot",
                "waits_on_free_of_k", "violations")


def schedule(n_blocks, n_steps, use_correction=True):
    out = np.zeros(7 * max(1, n_blocks * n_steps), dtype=np.int32)
    n = lib().oracle_schedule(n_blocks, n_steps, 1 if use_correction else 0, _ptr(out))
    assert n == n_blocks * n_steps
    return out[: 7 * n].reshape(n, 7)


# ---- block forward ---------------------------------------------------------

def gelu_tanh(z):
    return float(lib().oracle_gelu_tanh(float(z)))


def gelu_tanh_array(z):
    """gelu_tanh applied element by element (float64 copy)."""
    z = np.ascontiguousarray(z, dtype=np.float64)
    out = np.empty_like(z)
    lib().oracle_gelu_tanh_array(_ptr(z), z.size, _ptr(out))
    return out


def rmsnorm_mod(x, g, shift, scale, eps=1e-6):
    x = np.ascontiguousarray(x, dtype=np.float64)
    rows, d = x.shape
    h = np.zeros_like(x)
    f32 = lambda a: np.ascontiguousarray(a, dtype=np.float32)
    g, shift, scale = f32(g), f32(shift), f32(scale)
    lib().oracle_rmsnorm_mod(_ptr(x), rows, d, _ptr(g), _ptr(shift), _ptr(scale), eps, _ptr(h))
    return h


def linear(a, w, threads=None):
    a = np.ascontiguousarray(a, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, k = a.shape
    n, k2 = w.shape
    assert k == k2
    y = np.zeros((rows, n), dtype=np.float64)
    lib().oracle_linear(_ptr(a), rows, k, _ptr(w), n, _ptr(y), threads or default_threads())
    return y


def attention(qkv, batch, tokens, d, heads, threads=None):
    qkv = np.ascontiguousarray(qkv, dtype=np.float64)
    assert qkv.shape == (batch * tokens, 3 * d)
    o = np.zeros((batch * tokens, d), dtype=np.float64)
    lib().oracle_attention(_ptr(qkv), batch, tokens, d, heads, _ptr(o), threads or default_threads())
    return o


PARAM_ORDER = ("norm1.weight", "ada1.shift", "ada1.scale", "ada1.gate",
               "attn.qkv.weight", "attn.out.weight",
               "norm2.weight", "ada2.shift", "ada2.scale", "ada2.gate",
               "mlp.fc1.weight", "mlp.fc2.weight")


# the checkpoint-shaped block's optional parameters, in the C call's order
EXTRA_ORDER = ("attn.qkv.bias", "attn.out.bias", "mlp.fc1.bias", "mlp.fc2.bias",
               "attn.q_norm.weight", "attn.k_norm.weight")


def qk_norm(qkv, d, heads, gq, gk, eps=1e-6):
    """Per-head RMSNorm of the q and k columns of qkv [rows, 3d] (a copy)."""
    q = np.array(qkv, dtype=np.float64, order="C", copy=True)
    gq = np.ascontiguousarray(gq, dtype=np.float32)
    gk = np.ascontiguousarray(gk, dtype=np.float32)
    lib().oracle_qk_norm(_ptr(q), q.shape[0], d, heads, _ptr(gq), _ptr(gk), eps)
    return q


def rope(qkv, batch, tokens, d, heads, base=10000.0):
    """Rotary embedding of the q and k columns of qkv [batch*tokens, 3d] (a copy)."""
    q = np.array(qkv, dtype=np.float64, order="C", copy=True)
    lib().oracle_rope(_ptr(q), batch, tokens, d, heads, base)
    return q


def block_forward(x, params, batch, tokens, d, heads, f, eps=1e-6, threads=None,
                  rope_base=0.0):
    """x: float32 [batch*tokens, d]; params: dict name -> float32 ndarray.
    Parameters named in EXTRA_ORDER are applied when present (the
    checkpoint-shaped block); rope_base > 0 applies rotary embedding."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(batch * tokens, d)
    arrs = [np.ascontiguousarray(params[n], dtype=np.float32) for n in PARAM_ORDER]
    out = np.zeros((batch * tokens, d), dtype=np.float64)
    extras = [np.ascontiguousarray(params[n], dtype=np.float32) if n in params else None
              for n in EXTRA_ORDER]
    if any(e is not None for e in extras) or rope_base > 0:
        ptrs = [e.ctypes.data if e is not None else None for e in extras]
        lib().oracle_block_forward_ex(_ptr(x), batch, tokens, d, heads, f, eps,
                                      _ptr_array(arrs), *ptrs, float(rope_base), _ptr(out),
                                      threads or default_threads())
        return out
    lib().oracle_block_forward(_ptr(x), batch, tokens, d, heads, f, eps,
                               _ptr_array(arrs), _ptr(out), threads or default_threads())
    return out


def block_forward_rows(x, params, rows, batch, tokens, d, heads, f, eps=1e-6, threads=None,
                       rope_base=0.0):
    """Block output for the listed query rows only (K and V from all tokens);
    the checkpoint-shaped additions as in block_forward."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(batch * tokens, d)
    arrs = [np.ascontiguousarray(params[n], dtype=np.float32) for n in PARAM_ORDER]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.zeros((len(rows), d), dtype=np.float64)
    extras = [np.ascontiguousarray(params[n], dtype=np.float32) if n in params else None
              for n in EXTRA_ORDER]
    if any(e is not None for e in extras) or rope_base > 0:
        ptrs = [e.ctypes.data if e is not None else None for e in extras]
        lib().oracle_block_forward_ex_rows(_ptr(x), batch, tokens, d, heads, f, eps,
                                           _ptr_array(arrs), *ptrs, float(rope_base), _ptr(rows),
                                           len(rows), _ptr(out), threads or default_threads())
        return out
    lib().oracle_block_forward_rows(_ptr(x), batch, tokens, d, heads, f, eps, _ptr_array(arrs),
                                    _ptr(rows), len(rows), _ptr(out),
                                    threads or default_threads())
    return out
