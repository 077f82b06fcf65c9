"""ctypes binding of ``libdlo.so`` (include/dlo.h): argument marshalling only.

Every function keeps the C name without the ``dlo_`` prefix, takes plain
integers (device or host addresses, e.g. ``tensor.data_ptr()``) or objects
with ``data_ptr()``, and raises :class:`DLOError` when the C call returns a
non-zero status.  All computation happens in the library's CUDA kernels; if
the library cannot be loaded this module raises at import of the library,
there is no fallback.
"""
import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libdlo.so")

OK, ERR_INVALID, ERR_CUDA, ERR_TIMEOUT, ERR_STATE, ERR_NOMEM, ERR_PARTIAL = range(7)
BF16, F32, F16, FP8_E4M3, FP8_E5M2, I8, U8, E8M0 = 0, 1, 2, 3, 4, 5, 6, 7
ESIZE = {BF16: 2, F32: 4, F16: 2, FP8_E4M3: 1, FP8_E5M2: 1, I8: 1, U8: 1, E8M0: 1}
COPY_AUTO, COPY_DMA, COPY_KERNEL, COPY_STAGED = 0, 1, 2, 3
EPI_BF16, EPI_GELU_BF16, EPI_RESID_F32 = 0, 1, 2
COPY_MODE_NAMES = {COPY_AUTO: "auto", COPY_DMA: "dma", COPY_KERNEL: "kernel",
                   COPY_STAGED: "staged"}


class DLOError(RuntimeError):
    def __init__(self, status, where, message):
        super().__init__("%s failed with status %d: %s" % (where, status, message))
        self.status = status


c_i32, c_i64, c_vp, c_sz, c_f32 = (ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p,
                                   ctypes.c_size_t, ctypes.c_float)


class ParamDesc(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("ndim", c_i32), ("shape", c_i64 * 4),
                ("dtype", c_i32), ("stride", c_i64 * 4)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("n_params", c_i32), ("n_groups", c_i32), ("n_shards", c_i32),
                ("has_dit_roles", c_i32), ("slot_bytes", c_i64), ("group_align", c_i64),
                ("staging_bytes", c_i64)]


class GroupInfo(ctypes.Structure):
    _fields_ = [("dtype", c_i32), ("esize", c_i32), ("numel", c_i64), ("shard_numel", c_i64),
                ("shard_bytes", c_i64), ("shard_alloc_bytes", c_i64), ("base", c_i64),
                ("stage_base", c_i64)]


class ParamInfo(ctypes.Structure):
    _fields_ = [("group", c_i32), ("dtype", c_i32), ("numel", c_i64), ("group_offset", c_i64),
                ("slot_offset", c_i64), ("storage_numel", c_i64), ("stride", c_i64 * 4)]


class DitCfg(ctypes.Structure):
    _fields_ = [("batch", c_i32), ("tokens", c_i32), ("hidden", c_i32), ("heads", c_i32),
                ("mlp", c_i32), ("eps", c_f32), ("flags", c_i32)]


class EngineDesc(ctypes.Structure):
    _fields_ = [("n_blocks", c_i32), ("slot", c_vp * 2), ("slot_bytes", c_i64),
                ("compute_stream", c_vp), ("copy_stream", c_vp), ("copy_mode", c_i32),
                ("copy_ctas", c_i32), ("timing", c_i32), ("dma_streams", c_i32),
                ("staging", c_vp * 2), ("staging_bytes", c_i64), ("gather_stream", c_vp),
                ("host_staging", c_vp * 2), ("host_staging_bytes", c_i64),
                ("pack_threads", c_i32), ("two_copy_streams", c_i32),
                ("log_capacity", c_i32), ("poison", c_i32), ("checks", c_i32)]


class SchedEvent(ctypes.Structure):
    _fields_ = [("k", c_i32), ("block", c_i32), ("read_slot", c_i32), ("prefetch_block", c_i32),
                ("prefetch_slot", c_i32), ("waits_on_free_of_k", c_i32), ("copy_mode", c_i32)]


class CopyRecord(ctypes.Structure):
    _fields_ = [("seq", c_i64), ("block", c_i32), ("slot", c_i32), ("copy_ms", c_f32),
                ("bytes", c_i64)]


class EngineStats(ctypes.Structure):
    _fields_ = [("chosen_mode", c_i32), ("n_forwards", c_i32), ("n_prefetches", c_i32),
                ("n_kernel_prefetches", c_i32), ("race_dma_us", ctypes.c_double),
                ("race_kernel_us", ctypes.c_double), ("n_direct_prefetches", c_i32),
                ("n_packed_prefetches", c_i32), ("pack_ms", ctypes.c_double),
                ("n_copy_kernel_launches", c_i32), ("log_dropped", c_i64),
                ("timed_dropped", c_i64), ("checked_pieces", c_i64)]


class CopyPiece(ctypes.Structure):
    _fields_ = [("group", c_i32), ("shard", c_i32), ("dst_offset", c_i64),
                ("src_offset", c_i64), ("bytes", c_i64)]


PIECES_SLOT_FROM_SHARDS, PIECES_STAGING_FROM_SHARDS, PIECES_SLOT_FROM_STAGING = 0, 1, 2


_P = ctypes.POINTER
_SIGS = {
    "dlo_plan_create": (c_i32, [_P(ParamDesc), c_i32, c_i32, _P(c_vp)]),
    "dlo_plan_query": (c_i32, [c_vp, _P(PlanInfo)]),
    "dlo_plan_group": (c_i32, [c_vp, c_i32, _P(GroupInfo)]),
    "dlo_plan_param": (c_i32, [c_vp, c_i32, _P(ParamInfo)]),
    "dlo_shard_host": (c_i32, [c_vp, _P(c_vp), _P(c_vp)]),
    "dlo_check_pieces": (c_i32, [c_vp, c_i32, _P(CopyPiece), c_i32, c_i64, _P(c_i32)]),
    "dlo_plan_destroy": (None, [c_vp]),
    "dlo_reassemble": (c_i32, [c_vp, _P(c_vp), c_vp, c_i32, c_vp]),
    "dlo_reassemble_staged": (c_i32, [c_vp, _P(c_vp), c_vp, c_i64, c_vp, c_vp, c_vp]),
    "dlo_forward_scratch_bytes": (c_sz, [_P(DitCfg)]),
    "dlo_forward_launches": (c_i32, [_P(DitCfg)]),
    "dlo_forward": (c_i32, [_P(DitCfg), c_vp, c_vp, c_vp, c_vp, c_sz, c_vp]),
    "dlo_forward_noalloc": (c_i32, [_P(DitCfg), c_vp, c_vp, c_vp, c_vp]),
    "dlo_op_rmsnorm_mod": (c_i32, [c_vp, c_i64, c_i64, c_vp, c_vp, c_vp, c_f32, c_vp, c_vp]),
    "dlo_op_linear_workspace_bytes": (c_sz, [c_i64, c_i64, c_i64, c_i32]),
    "dlo_op_linear": (c_i32, [c_vp, c_i64, c_i64, c_vp, c_i64, c_i32, c_vp, c_vp, c_vp, c_vp,
                              c_sz, c_vp]),
    "dlo_op_qk_norm_rope": (c_i32, [c_vp, c_i64, c_i64, c_i64, c_i64, c_vp, c_vp, c_f32, c_f32,
                                    c_vp]),
    "dlo_set_gemm_pair_mode": (c_i32, [c_i32]),
    "dlo_op_linear_on_pairs": (c_i32, [c_i64, c_i64, c_i64, c_i32]),
    "dlo_op_attention_scratch_bytes": (c_sz, [c_i64, c_i64, c_i64]),
    "dlo_op_attention": (c_i32, [c_vp, c_i64, c_i64, c_i64, c_i64, c_vp, c_vp, c_sz, c_vp]),
    "dlo_engine_create": (c_i32, [_P(EngineDesc), _P(c_vp)]),
    "dlo_register_block": (c_i32, [c_vp, c_i32, c_vp, _P(c_vp)]),
    "dlo_register_block_source": (c_i32, [c_vp, c_i32, c_vp, _P(c_vp)]),
    "dlo_host_register_ranges": (c_i32, [_P(c_vp), _P(c_i64), c_i32, c_i32, c_i64, _P(c_i64)]),
    "dlo_host_unregister_ranges": (c_i32, [_P(c_vp), _P(c_i64), c_i32]),
    "dlo_debug_fake_host_register": (c_i32, [c_i32, c_i32, c_i32]),
    "dlo_debug_fake_host_register_log": (c_i32, [_P(c_i32), c_i32, _P(c_i32)]),
    "dlo_prefetch": (c_i32, [c_vp, c_i32, c_i32]),
    "dlo_wait": (c_i32, [c_vp, c_i32]),
    "dlo_wait_host": (c_i32, [c_vp, c_i32, c_i32]),
    "dlo_param_view": (c_i32, [c_vp, c_i32, c_i32, _P(c_vp)]),
    "dlo_pre_forward": (c_i32, [c_vp, c_i32, _P(c_i32)]),
    "dlo_post_forward": (c_i32, [c_vp, c_i32]),
    "dlo_block_forward": (c_i32, [c_vp, c_i32, _P(DitCfg), c_vp, c_vp, c_sz]),
    "dlo_schedule_log": (c_i32, [c_vp, _P(SchedEvent), c_i32, _P(c_i32)]),
    "dlo_engine_query": (c_i32, [c_vp, _P(EngineStats)]),
    "dlo_engine_copy_times": (c_i32, [c_vp, _P(c_f32), _P(c_i64), c_i32, _P(c_i32)]),
    "dlo_engine_copy_spans": (c_i32, [c_vp, _P(c_f32), _P(c_f32), c_i32, _P(c_i32)]),
    "dlo_engine_copy_log": (c_i32, [c_vp, c_i64, _P(CopyRecord), c_i32, _P(c_i32), _P(c_i64)]),
    "dlo_replace_block_shards": (c_i32, [c_vp, c_i32, _P(c_vp), c_i32]),
    "dlo_engine_destroy": (c_i32, [c_vp, c_i32]),
    "dlo_kernel_status": (c_i32, [_P(c_i32)]),
    "dlo_set_launch_overlap": (c_i32, [c_i32]),
    "dlo_debug_wait_probe": (c_i32, [c_i32, c_i64, c_i64, _P(c_i64), _P(c_i32)]),
    "dlo_last_error": (ctypes.c_char_p, []),
    "dlo_version": (ctypes.c_char_p, []),
}

_lib = None


def lib():
    """Loads libdlo.so (built by ``layerwise_weight_offload_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError("libdlo.so is not built (run __graft_entry__.build() or "
                              "python -m layerwise_weight_offload_gb300.build); "
                              "there is no fallback path")
        L = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def header_symbols(path=None):
    """Names of the functions include/dlo.h declares."""
    path = path or os.path.join(os.path.dirname(_PKG), "include", "dlo.h")
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dlo_[a-z_0-9]+)\s*\(", text)))


def _check(status, where):
    if status != OK:
        msg = lib().dlo_last_error()
        raise DLOError(status, where, msg.decode() if msg else "")


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError("cannot take the address of %r" % type(x))


def _ptrs(xs):
    return (c_vp * len(xs))(*[_ptr(x) for x in xs])


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def last_error():
    return lib().dlo_last_error().decode()


def version():
    return lib().dlo_version().decode()


# ---- plan ------------------------------------------------------------------

class Plan:
    def __init__(self, descs, n_shards):
        """descs: sequence of (name, shape, dtype code) or (name, shape, dtype
        code, element strides) in registration order; no strides (or all 0)
        means row-major contiguous."""
        self._names = [d[0].encode() for d in descs]
        arr = (ParamDesc * len(descs))()
        for i, d in enumerate(descs):
            name, shape, code = d[:3]
            strides = d[3] if len(d) > 3 else None
            arr[i].name = self._names[i]
            arr[i].ndim = len(shape)
            for j, v in enumerate(shape):
                arr[i].shape[j] = int(v)
            if strides is not None:
                for j, v in enumerate(strides):
                    arr[i].stride[j] = int(v)
            arr[i].dtype = int(code)
        h = c_vp()
        _check(lib().dlo_plan_create(arr, len(descs), int(n_shards), ctypes.byref(h)),
               "dlo_plan_create")
        self.handle = h.value
        self.n_shards = int(n_shards)

    def info(self):
        out = PlanInfo()
        _check(lib().dlo_plan_query(self.handle, ctypes.byref(out)), "dlo_plan_query")
        return out

    def group(self, g):
        out = GroupInfo()
        _check(lib().dlo_plan_group(self.handle, g, ctypes.byref(out)), "dlo_plan_group")
        return out

    def param(self, p):
        out = ParamInfo()
        _check(lib().dlo_plan_param(self.handle, p, ctypes.byref(out)), "dlo_plan_param")
        return out

    def groups(self):
        return [self.group(g) for g in range(self.info().n_groups)]

    def shard_host(self, param_srcs, shard_dsts):
        _check(lib().dlo_shard_host(self.handle, _ptrs(param_srcs), _ptrs(shard_dsts)),
               "dlo_shard_host")

    def destroy(self):
        if self.handle:
            lib().dlo_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def plan_create(descs, n_shards):
    return Plan(descs, n_shards)


def check_pieces(plan, phase, pieces, target_bytes):
    """Checks one prefetch's copies, given as (group, shard, dst_offset,
    src_offset, bytes) tuples, against the plan.  Returns None if they pass;
    otherwise (index of the first failing piece or -1, message)."""
    arr = (CopyPiece * max(1, len(pieces)))()
    for i, q in enumerate(pieces):
        arr[i] = CopyPiece(*[int(v) for v in q])
    bad = c_i32(-2)
    st = lib().dlo_check_pieces(plan.handle, int(phase), arr, len(pieces), int(target_bytes),
                                ctypes.byref(bad))
    if st == OK:
        assert bad.value == -1
        return None
    if st != ERR_STATE:
        _check(st, "dlo_check_pieces")
    return bad.value, last_error()


def reassemble(plan, shard_ptrs, dst, mode=COPY_DMA, stream=None):
    _check(lib().dlo_reassemble(plan.handle, _ptrs(shard_ptrs), _ptr(dst), int(mode),
                                _stream(stream)), "dlo_reassemble")


def reassemble_staged(plan, shard_ptrs, staging, staging_bytes, dst, copy_stream=None,
                      gather_stream=None):
    _check(lib().dlo_reassemble_staged(plan.handle, _ptrs(shard_ptrs), _ptr(staging),
                                       int(staging_bytes), _ptr(dst), _stream(copy_stream),
                                       _stream(gather_stream)), "dlo_reassemble_staged")


# ---- block forward -----------------------------------------------------------

FWD_GRAPH, FWD_ROPE, FWD_QK_NORM = 1, 2, 4
ROPE_BASE = 10000.0


def dit_cfg(batch, tokens, hidden, heads, mlp, eps=1e-6, graph=True, rope=False, qk_norm=False):
    flags = (FWD_GRAPH if graph else 0) | (FWD_ROPE if rope else 0) | \
        (FWD_QK_NORM if qk_norm else 0)
    return DitCfg(int(batch), int(tokens), int(hidden), int(heads), int(mlp), float(eps), flags)


def forward_launches(cfg):
    return int(lib().dlo_forward_launches(ctypes.byref(cfg)))


def forward_scratch_bytes(cfg):
    return int(lib().dlo_forward_scratch_bytes(ctypes.byref(cfg)))


def forward(cfg, plan, block_base, x, scratch, scratch_bytes, stream=None):
    _check(lib().dlo_forward(ctypes.byref(cfg), plan.handle, _ptr(block_base), _ptr(x),
                             _ptr(scratch), int(scratch_bytes), _stream(stream)), "dlo_forward")


def forward_noalloc(cfg, plan, block_base, x, stream=None):
    """dlo_forward with the library's static scratch (allocates nothing)."""
    _check(lib().dlo_forward_noalloc(ctypes.byref(cfg), plan.handle, _ptr(block_base), _ptr(x),
                                     _stream(stream)), "dlo_forward_noalloc")


def op_rmsnorm_mod(x, rows, d, g, shift, scale, eps, h, stream=None):
    _check(lib().dlo_op_rmsnorm_mod(_ptr(x), rows, d, _ptr(g), _ptr(shift), _ptr(scale),
                                    float(eps), _ptr(h), _stream(stream)), "dlo_op_rmsnorm_mod")


def op_linear_workspace_bytes(M, N, K, epilogue):
    return int(lib().dlo_op_linear_workspace_bytes(M, N, K, int(epilogue)))


def op_linear(a, M, K, w, N, epilogue, out, gate=None, stream=None, workspace=None,
              workspace_bytes=0, bias=None):
    _check(lib().dlo_op_linear(_ptr(a), M, K, _ptr(w), N, int(epilogue), _ptr(out), _ptr(gate),
                               _ptr(bias), _ptr(workspace), int(workspace_bytes),
                               _stream(stream)),
           "dlo_op_linear")


GEMM_PAIR_AUTO, GEMM_PAIR_OFF, GEMM_PAIR_ON = -1, 0, 1


def set_gemm_pair_mode(mode):
    """Which GEMM kernel runs the linears: GEMM_PAIR_AUTO (by shape),
    GEMM_PAIR_OFF (single CTAs) or GEMM_PAIR_ON (CTA pairs for all)."""
    _check(lib().dlo_set_gemm_pair_mode(int(mode)), "dlo_set_gemm_pair_mode")


def op_linear_on_pairs(M, N, K, epilogue):
    """True if a linear of this shape runs on CTA pairs (gemm_pair_kernel)."""
    return bool(lib().dlo_op_linear_on_pairs(M, N, K, int(epilogue)))


def op_qk_norm_rope(qkv, batch, tokens, d, heads, gq=None, gk=None, eps=1e-6, rope_base=0.0,
                    stream=None):
    _check(lib().dlo_op_qk_norm_rope(_ptr(qkv), batch, tokens, d, heads, _ptr(gq), _ptr(gk),
                                     float(eps), float(rope_base), _stream(stream)),
           "dlo_op_qk_norm_rope")


def op_attention_scratch_bytes(batch, tokens, d):
    return int(lib().dlo_op_attention_scratch_bytes(batch, tokens, d))


def op_attention(qkv, batch, tokens, d, heads, o, scratch, scratch_bytes, stream=None):
    _check(lib().dlo_op_attention(_ptr(qkv), batch, tokens, d, heads, _ptr(o), _ptr(scratch),
                                  int(scratch_bytes), _stream(stream)), "dlo_op_attention")


def host_register_ranges(ptrs, sizes, read_only=False, limit_bytes=0):
    """Page-locks the ranges, all or nothing; returns the registered bytes."""
    n = len(ptrs)
    arr = (c_i64 * max(n, 1))(*[int(s) for s in sizes])
    out = c_i64(0)
    _check(lib().dlo_host_register_ranges(_ptrs(ptrs), arr, n, 1 if read_only else 0,
                                          int(limit_bytes), ctypes.byref(out)),
           "dlo_host_register_ranges")
    return out.value


def host_unregister_ranges(ptrs, sizes):
    n = len(ptrs)
    arr = (c_i64 * max(n, 1))(*[int(s) for s in sizes])
    _check(lib().dlo_host_unregister_ranges(_ptrs(ptrs), arr, n), "dlo_host_unregister_ranges")


def debug_fake_host_register(enable, fail_register_at=-1, fail_unregister_at=-1):
    _check(lib().dlo_debug_fake_host_register(int(enable), int(fail_register_at),
                                              int(fail_unregister_at)),
           "dlo_debug_fake_host_register")


def debug_fake_host_register_log():
    buf = (c_i32 * 256)()
    n = c_i32(0)
    _check(lib().dlo_debug_fake_host_register_log(buf, 256, ctypes.byref(n)),
           "dlo_debug_fake_host_register_log")
    return list(buf[:min(n.value, 256)])


def set_launch_overlap(mode):
    """True/1: always, False/0: never, -1: by block size (the default)."""
    m = -1 if mode == -1 else (1 if mode else 0)
    _check(lib().dlo_set_launch_overlap(m), "dlo_set_launch_overlap")


def kernel_status():
    v = c_i32()
    _check(lib().dlo_kernel_status(ctypes.byref(v)), "dlo_kernel_status")
    return v.value


def debug_wait_probe(spin, limit_ns, abort_ns=0):
    """Runs the library's bounded device wait against a phase nobody
    completes; returns (status, elapsed_ns, code) without raising."""
    el, code = c_i64(), c_i32()
    st = lib().dlo_debug_wait_probe(1 if spin else 0, int(limit_ns), int(abort_ns),
                                    ctypes.byref(el), ctypes.byref(code))
    return st, el.value, code.value


# ---- engine ------------------------------------------------------------------

class Engine:
    def __init__(self, n_blocks, slot0, slot1, slot_bytes, compute_stream, copy_stream,
                 copy_mode=COPY_AUTO, copy_ctas=0, timing=False, dma_streams=0,
                 staging=None, staging_bytes=0, gather_stream=None, host_staging=None,
                 host_staging_bytes=0, pack_threads=0, two_copy_streams=False,
                 log_capacity=0, poison=False, checks=False):
        """staging: two device buffers (and gather_stream) for COPY_STAGED;
        host_staging: two page-locked host buffers for rank-local source
        blocks whose parameters are pageable."""
        d = EngineDesc()
        d.n_blocks = int(n_blocks)
        d.slot[0] = _ptr(slot0)
        d.slot[1] = _ptr(slot1)
        d.slot_bytes = int(slot_bytes)
        d.compute_stream = _stream(compute_stream)
        d.copy_stream = _stream(copy_stream)
        d.copy_mode = int(copy_mode)
        d.copy_ctas = int(copy_ctas)
        d.timing = 1 if timing else 0
        d.dma_streams = int(dma_streams)
        if staging is not None:
            d.staging[0] = _ptr(staging[0])
            d.staging[1] = _ptr(staging[1])
        d.staging_bytes = int(staging_bytes)
        d.gather_stream = _stream(gather_stream)
        if host_staging is not None:
            d.host_staging[0] = _ptr(host_staging[0])
            d.host_staging[1] = _ptr(host_staging[1])
        d.host_staging_bytes = int(host_staging_bytes)
        d.pack_threads = int(pack_threads)
        d.two_copy_streams = 1 if two_copy_streams else 0
        d.log_capacity = int(log_capacity)
        d.poison = 1 if poison else 0
        d.checks = 1 if checks else 0
        h = c_vp()
        _check(lib().dlo_engine_create(ctypes.byref(d), ctypes.byref(h)), "dlo_engine_create")
        self.handle = h.value
        self.n_blocks = int(n_blocks)

    def register_block(self, block, plan, shard_ptrs):
        _check(lib().dlo_register_block(self.handle, block, plan.handle, _ptrs(shard_ptrs)),
               "dlo_register_block")

    def register_block_source(self, block, plan, param_srcs):
        _check(lib().dlo_register_block_source(self.handle, block, plan.handle,
                                               _ptrs(param_srcs)), "dlo_register_block_source")

    def replace_block_shards(self, block, shard_ptrs, timeout_ms=60000):
        _check(lib().dlo_replace_block_shards(self.handle, block, _ptrs(shard_ptrs),
                                              int(timeout_ms)), "dlo_replace_block_shards")

    def copy_log(self, since, cap=4096):
        """Completed timed prefetches with seq >= since: ([(seq, block, slot,
        ms, bytes)], next_since), without waiting on the GPU."""
        buf = (CopyRecord * cap)()
        n, nxt = c_i32(), c_i64()
        _check(lib().dlo_engine_copy_log(self.handle, int(since), buf, cap, ctypes.byref(n),
                                         ctypes.byref(nxt)), "dlo_engine_copy_log")
        return ([(r.seq, r.block, r.slot, r.copy_ms, r.bytes) for r in buf[:n.value]],
                nxt.value)

    def prefetch(self, block, slot):
        _check(lib().dlo_prefetch(self.handle, block, slot), "dlo_prefetch")

    def wait(self, block):
        _check(lib().dlo_wait(self.handle, block), "dlo_wait")

    def wait_host(self, block, timeout_ms):
        _check(lib().dlo_wait_host(self.handle, block, int(timeout_ms)), "dlo_wait_host")

    def param_view(self, block, param):
        out = c_vp()
        _check(lib().dlo_param_view(self.handle, block, param, ctypes.byref(out)),
               "dlo_param_view")
        return out.value

    def pre_forward(self, block):
        s = c_i32()
        _check(lib().dlo_pre_forward(self.handle, block, ctypes.byref(s)), "dlo_pre_forward")
        return s.value

    def post_forward(self, block):
        _check(lib().dlo_post_forward(self.handle, block), "dlo_post_forward")

    def block_forward(self, block, cfg, x, scratch, scratch_bytes):
        _check(lib().dlo_block_forward(self.handle, block, ctypes.byref(cfg), _ptr(x),
                                       _ptr(scratch), int(scratch_bytes)), "dlo_block_forward")

    def schedule_log(self):
        n = c_i32()
        _check(lib().dlo_schedule_log(self.handle, None, 0, ctypes.byref(n)), "dlo_schedule_log")
        buf = (SchedEvent * max(1, n.value))()
        _check(lib().dlo_schedule_log(self.handle, buf, n.value, ctypes.byref(n)),
               "dlo_schedule_log")
        return [(e.k, e.block, e.read_slot, e.prefetch_block, e.prefetch_slot,
                 e.waits_on_free_of_k, e.copy_mode) for e in buf[:n.value]]

    def query(self):
        s = EngineStats()
        _check(lib().dlo_engine_query(self.handle, ctypes.byref(s)), "dlo_engine_query")
        return s

    def copy_times(self):
        n = c_i32()
        _check(lib().dlo_engine_copy_times(self.handle, None, None, 0, ctypes.byref(n)),
               "dlo_engine_copy_times")
        ms = (c_f32 * max(1, n.value))()
        by = (c_i64 * max(1, n.value))()
        _check(lib().dlo_engine_copy_times(self.handle, ms, by, n.value, ctypes.byref(n)),
               "dlo_engine_copy_times")
        return list(ms[:n.value]), list(by[:n.value])

    def copy_spans(self):
        """[(start_ms, end_ms)] of every timed prefetch, on one clock."""
        n = c_i32()
        _check(lib().dlo_engine_copy_spans(self.handle, None, None, 0, ctypes.byref(n)),
               "dlo_engine_copy_spans")
        s = (c_f32 * max(1, n.value))()
        t = (c_f32 * max(1, n.value))()
        _check(lib().dlo_engine_copy_spans(self.handle, s, t, n.value, ctypes.byref(n)),
               "dlo_engine_copy_spans")
        return list(zip(s[:n.value], t[:n.value]))

    def destroy(self, timeout_ms=60000):
        if self.handle:
            _check(lib().dlo_engine_destroy(self.handle, int(timeout_ms)), "dlo_engine_destroy")
            self.handle = None


def engine_create(*args, **kw):
    return Engine(*args, **kw)
