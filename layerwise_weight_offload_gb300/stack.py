"""Assembles block stacks from the C ABI: pinned host shards, a streamed
two-slot engine, and an all-resident reference over the same kernels.

PyTorch provides device memory, pinned host memory and streams only; every
step of the method runs in the library (``dlo``).
"""
import ctypes
import mmap

import torch

from . import dlo
from . import workloads as W


def _round_up(v, a):
    return (v + a - 1) // a * a


_MADV_COLLAPSE = 25


def _collapse(ptr, nbytes):
    """Asks the kernel to back [ptr, ptr+nbytes) with huge pages now
    (MADV_COLLAPSE, Linux 6.1+); ignored where unsupported."""
    try:
        libc = ctypes.CDLL(None, use_errno=True)
        libc.madvise.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
        libc.madvise(ctypes.c_void_p(ptr), ctypes.c_size_t(nbytes), _MADV_COLLAPSE)
    except (OSError, AttributeError):
        pass


class PinnedBuffer:
    """Page-locked, device-mapped host bytes of an exact size, backed by
    transparent huge pages.

    The bytes come from an anonymous mapping aligned to 512 MiB and marked
    MADV_HUGEPAGE, touched once, then registered with the CUDA driver
    (cudaHostRegister, portable | mapped).  On the GB300 (NVLink-C2C, 64 KiB
    base pages) the GPU's sustained host->device rate from pinned memory
    built of small pages falls far below the link rate once the footprint
    is several GB (address translations no longer fit the GPU's caches);
    from huge-page memory it stays at the link rate.  Unlike a caching
    pinned allocator, the size is not rounded to a power of two."""

    ALIGN = 512 << 20

    def __init__(self, nbytes):
        self.nbytes = int(nbytes)
        size = self.nbytes + self.ALIGN
        self._map = mmap.mmap(-1, size, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
        try:
            self._map.madvise(mmap.MADV_HUGEPAGE)
        except (AttributeError, OSError, ValueError):
            pass
        self._cbuf = (ctypes.c_uint8 * size).from_buffer(self._map)
        base = ctypes.addressof(self._cbuf)
        self.ptr = _round_up(base, self.ALIGN)
        self.offset = self.ptr - base
        ctypes.memset(self.ptr, 0, self.nbytes)       # first touch: huge pages
        _collapse(self.ptr, self.nbytes)
        self._t = torch.frombuffer(self._map, dtype=torch.uint8)
        rt = torch.cuda.cudart()
        err = rt.cudaHostRegister(self.ptr, self.nbytes, 1 | 2)   # portable | mapped
        code = err.value if hasattr(err, "value") else int(err)
        if code != 0:
            raise RuntimeError("cudaHostRegister of %d bytes failed (%d)" % (self.nbytes, code))
        self.registered = True

    def view(self, offset, nbytes):
        return self._t[self.offset + offset:self.offset + offset + nbytes]

    def huge_fraction(self):
        """Fraction of the buffer's resident bytes backed by huge pages
        (from /proc/self/smaps), or None where that is not readable."""
        try:
            with open("/proc/self/smaps") as fh:
                lines = fh.read().splitlines()
        except OSError:
            return None
        lo, hi = self.ptr, self.ptr + self.nbytes
        rss = huge = 0
        inside = False
        for line in lines:
            head = line.split(" ", 1)[0]
            if "-" in head and ":" not in head:
                a, b = (int(v, 16) for v in head.split("-"))
                inside = a < hi and b > lo
            elif inside and line.startswith("Rss:"):
                rss += int(line.split()[1])
            elif inside and line.startswith("AnonHugePages:"):
                huge += int(line.split()[1])
        return huge / rss if rss else None

    def close(self):
        if self.registered:
            torch.cuda.cudart().cudaHostUnregister(self.ptr)
            self.registered = False
        if self._map is not None:
            self._t = None
            self._cbuf = None
            try:
                self._map.close()
            except BufferError:
                pass            # a view still exports the buffer; freed with it
            self._map = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class HostBlocks:
    """The pinned shards of `w.distinct` host blocks: per block, for every
    dtype group g and shard r, shard_alloc_bytes at a 256-byte aligned offset
    of one registered buffer."""

    def __init__(self, w: W.Workload, seed=0, gen_device="cpu", keep_params=False):
        self.w = w
        self.descs = W.block_param_descs(w)
        self.plan = dlo.Plan(self.descs, w.shards)
        self.groups = self.plan.groups()
        s = w.shards
        self.offsets = []
        off = 0
        for g in self.groups:
            for _ in range(s):
                self.offsets.append(off)
                off += _round_up(g.shard_alloc_bytes, 256)
        self.block_bytes = off
        self.buf = PinnedBuffer(self.block_bytes * w.distinct)
        self.params = [] if keep_params else None
        for hb in range(w.distinct):
            p = W.gen_block(w, hb, seed, device=gen_device)
            p = {k: v.cpu().contiguous() for k, v in p.items()}
            srcs = [p[name].data_ptr() for name, _, _ in self.descs]
            self.plan.shard_host(srcs, self.shard_ptrs(hb))
            if keep_params:
                self.params.append(p)
            del p

    def pretouch(self, stream=None):
        """Reads every host block once from the GPU (a copy-kernel pass, then
        a DMA pass, into a scratch slot) so that first-access costs of the
        pinned pages are paid at setup rather than in the first forwards."""
        dst = torch.empty(self.plan.info().slot_bytes, dtype=torch.uint8, device="cuda")
        s = stream or torch.cuda.Stream()
        for mode in (dlo.COPY_KERNEL, dlo.COPY_DMA):
            for hb in range(self.w.distinct):
                dlo.reassemble(self.plan, self.shard_ptrs(hb), dst, mode, s)
        s.synchronize()
        del dst

    def shard_ptrs(self, hb):
        base = self.buf.ptr + hb * self.block_bytes
        return [base + o for o in self.offsets]

    def shard_views(self, hb):
        """uint8 tensors over the shards of host block hb, [g * s + r]."""
        out = []
        for i, o in enumerate(self.offsets):
            g = self.groups[i // self.w.shards]
            out.append(self.buf.view(hb * self.block_bytes + o, g.shard_alloc_bytes))
        return out

    def close(self):
        self.buf.close()


class StreamedStack:
    """Two slots and the hook schedule: the path the pages describe."""

    def __init__(self, host: HostBlocks, copy_mode=dlo.COPY_AUTO, copy_ctas=0, timing=False,
                 device="cuda"):
        w = host.w
        self.w, self.host, self.plan = w, host, host.plan
        self.slot_bytes = _round_up(self.plan.info().slot_bytes, 256)
        self.slots = [torch.empty(self.slot_bytes, dtype=torch.uint8, device=device)
                      for _ in range(2)]
        self.compute = torch.cuda.Stream(device=device)
        self.copy = torch.cuda.Stream(device=device)
        self.engine = dlo.Engine(w.n_blocks, self.slots[0], self.slots[1], self.slot_bytes,
                                 self.compute, self.copy, copy_mode, copy_ctas, timing)
        for i in range(w.n_blocks):
            self.engine.register_block(i, self.plan, host.shard_ptrs(i % w.distinct))
        self.cfg = dlo.dit_cfg(w.batch, w.tokens, w.hidden, w.heads, w.mlp, w.eps)
        self.scratch_bytes = dlo.forward_scratch_bytes(self.cfg)
        self.scratch = torch.empty(self.scratch_bytes, dtype=torch.uint8, device=device)
        self.primed = False

    def prime(self):
        """Setup prefetch: block 0 into slot 0."""
        self.engine.prefetch(0, 0)
        self.primed = True

    def step(self, x):
        """One denoising step (every block once) on the compute stream; x is
        the fp32 residual [batch*tokens, hidden], updated in place."""
        if not self.primed:
            self.prime()
        for i in range(self.w.n_blocks):
            self.engine.block_forward(i, self.cfg, x, self.scratch, self.scratch_bytes)

    def close(self):
        if self.engine is not None:
            self.engine.destroy()
            self.engine = None


class ResidentStack:
    """Every distinct block reassembled once into its own device buffer (the
    same slot layout), then the same forward kernels: the reference run the
    streamed path must match bit for bit."""

    def __init__(self, host: HostBlocks, device="cuda", stream=None):
        w = host.w
        self.w, self.host, self.plan = w, host, host.plan
        self.slot_bytes = _round_up(self.plan.info().slot_bytes, 256)
        self.stream = stream or torch.cuda.Stream(device=device)
        self.bufs = []
        for hb in range(w.distinct):
            b = torch.empty(self.slot_bytes, dtype=torch.uint8, device=device)
            dlo.reassemble(self.plan, host.shard_ptrs(hb), b, dlo.COPY_DMA, self.stream)
            self.bufs.append(b)
        self.stream.synchronize()
        self.cfg = dlo.dit_cfg(w.batch, w.tokens, w.hidden, w.heads, w.mlp, w.eps)
        self.scratch_bytes = dlo.forward_scratch_bytes(self.cfg)
        self.scratch = torch.empty(self.scratch_bytes, dtype=torch.uint8, device=device)

    def block(self, i, x):
        dlo.forward(self.cfg, self.plan, self.bufs[i % self.w.distinct], x, self.scratch,
                    self.scratch_bytes, self.stream)

    def step(self, x):
        for i in range(self.w.n_blocks):
            self.block(i, x)
