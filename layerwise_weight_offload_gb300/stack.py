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
_HUGE = 512 << 20        # PMD size of a 64 KiB-page kernel; also a multiple of 2 MiB


def _collapse(ptr, nbytes):
    """Asks the kernel to back [ptr, ptr+nbytes) with huge pages now
    (MADV_COLLAPSE, Linux 6.1+).  True if it reports success."""
    try:
        libc = ctypes.CDLL(None, use_errno=True)
        libc.madvise.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
        return libc.madvise(ctypes.c_void_p(ptr), ctypes.c_size_t(nbytes), _MADV_COLLAPSE) == 0
    except (OSError, AttributeError):
        return False


class PinnedBuffer:
    """Page-locked, device-mapped host bytes backed by transparent huge
    pages, with an allocator that only hands out huge-page ranges.

    The mapping is anonymous, aligned to 512 MiB and marked MADV_HUGEPAGE.
    Ranges of 512 MiB are prepared as the allocator reaches them: touched,
    then collapsed (MADV_COLLAPSE); a range the kernel could not back with a
    huge page is skipped.  The prepared prefix is then registered with the
    CUDA driver (cudaHostRegister, portable | mapped).

    Why: on the GB300 (NVLink-C2C, 64 KiB base pages) the GPU's sustained
    host->device rate from pinned memory made of small pages falls far
    below the link rate once the footprint is several GB (17-150 GB/s
    measured, against 211 GB/s from huge-page memory), and a block that
    lands even partly in small pages takes 10-40x longer to stream.

    With defer=False (default) `nbytes` are placed and registered at once
    and `ptr` points at them; with defer=True the caller place()s its pieces
    and then calls register()."""

    SMALL = 256 << 20     # below this the footprint is too small to matter

    def __init__(self, nbytes, spare=0.25, tries=3, defer=False):
        self.nbytes = int(nbytes)
        self.small = self.nbytes < self.SMALL
        n_ranges = max(1, -(-self.nbytes // _HUGE))
        self.capacity = (_round_up(self.nbytes, 1 << 16) if self.small
                         else (n_ranges + int(n_ranges * spare) + 2) * _HUGE)
        self.tries = tries
        self._map = mmap.mmap(-1, self.capacity + _HUGE,
                              flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
        if not self.small:
            try:
                self._map.madvise(mmap.MADV_HUGEPAGE)
            except (AttributeError, OSError, ValueError):
                pass
        self._cbuf = (ctypes.c_uint8 * (self.capacity + _HUGE)).from_buffer(self._map)
        base = ctypes.addressof(self._cbuf)
        self.ptr = _round_up(base, _HUGE)
        self.offset = self.ptr - base
        self.good = []                  # per prepared 512 MiB range
        self.rate = []                  # per range: surveyed H2D GB/s, or None
        self.fast = []                  # per range: None (not surveyed) or bool
        self.segments = []              # registered [first, end) range spans
        self._cursor = 0
        self._t = None
        self.registered = False
        self.registered_bytes = 0
        if not defer:
            self.base_offset = self.place([self.nbytes], 256 if self.small else _HUGE)[0]
            self.register()
            self.ptr += self.base_offset
            self.offset += self.base_offset

    def _prepare(self, upto):
        if self.small:
            if not self.good:
                ctypes.memset(self.ptr, 0, self.capacity)
                self.good = [False]
            return
        while len(self.good) < upto:
            r = len(self.good)
            if (r + 1) * _HUGE > self.capacity:
                raise MemoryError("PinnedBuffer: capacity exhausted")
            ctypes.memset(self.ptr + r * _HUGE, 0, _HUGE)      # first touch
            ok = False
            for _ in range(self.tries):
                if _collapse(self.ptr + r * _HUGE, _HUGE):
                    ok = True
                    break
            self.good.append(ok)
            self.rate.append(None)
            self.fast.append(None)

    def place(self, sizes, align=256):
        """Offsets (from .ptr) for pieces of the given sizes, in order.
        Pieces go into runs of huge-page ranges first (a piece never covers
        a range the kernel could not back with a huge page); pieces that
        find no such run once the spare room is used up take the remaining
        space, small pages included."""
        if self.registered:
            raise RuntimeError("PinnedBuffer: place after register")
        if self.small:
            self._prepare(1)
            offs = []
            for n in sizes:
                pos = _round_up(self._cursor, align)
                if pos + int(n) > self.capacity:
                    raise MemoryError("PinnedBuffer: %d bytes do not fit" % int(n))
                offs.append(pos)
                self._cursor = pos + int(n)
            return offs
        offs = [None] * len(sizes)
        cursor = self._cursor
        for i, n in enumerate(sizes):
            n = int(n)
            pos = _round_up(cursor, align)
            while True:
                first, last = pos // _HUGE, (pos + n - 1) // _HUGE
                if (last + 1) * _HUGE > self.capacity:
                    break
                self._prepare(last + 1)
                bad = [r for r in range(first, last + 1) if not self.good[r]]
                if not bad:
                    offs[i] = pos
                    cursor = pos + n
                    break
                pos = (bad[-1] + 1) * _HUGE
        self._cursor = max(cursor, self._cursor)
        # leftovers: first fit into the space no piece uses
        for i, n in enumerate(sizes):
            if offs[i] is not None:
                continue
            used = sorted((o, o + int(sizes[j])) for j, o in enumerate(offs) if o is not None)
            pos, n = 0, int(n)
            for a, b in used + [(self.capacity, self.capacity)]:
                pos = _round_up(pos, align)
                if pos + n <= a:
                    break
                pos = max(pos, b)
            if pos + n > self.capacity:
                raise MemoryError("PinnedBuffer: %d bytes do not fit" % n)
            self._prepare((pos + n - 1) // _HUGE + 1)
            offs[i] = pos
            self._cursor = max(self._cursor, pos + n)
        return offs

    def register(self):
        """Registers the prepared ranges not registered yet (all of them on the
        first call) with the CUDA driver as one segment."""
        rt = torch.cuda.cudart()
        if self.small:
            start, nbytes = 0, self.capacity
        else:
            first = self.segments[-1][1] if self.segments else 0
            start, nbytes = first * _HUGE, (len(self.good) - first) * _HUGE
            if nbytes <= 0:
                return
        err = rt.cudaHostRegister(self.ptr + start, nbytes, 1 | 2)   # portable | mapped
        code = err.value if hasattr(err, "value") else int(err)
        if code != 0:
            raise RuntimeError("cudaHostRegister of %d bytes failed (%d)" % (nbytes, code))
        if not self.small:
            self.segments.append((start // _HUGE, len(self.good)))
        self._reg_ptrs = getattr(self, "_reg_ptrs", []) + [self.ptr + start]
        self.registered = True
        self.registered_bytes += nbytes
        if self._t is None:
            self._t = torch.frombuffer(self._map, dtype=torch.uint8)

    def survey(self, min_frac=0.6, device="cuda"):
        """Times a 512 MiB host->device copy of every registered huge-page
        range not surveyed yet, on the second of two passes over all of them
        (so every range is timed after the others' copies, as in a streaming
        loop, and after its own first-access costs), and marks as slow the
        ranges below min_frac of the median rate.

        Why: on some GB300 hosts a part of the huge-page ranges streams to the
        GPU at a few GB/s in steady state while the rest reaches the link
        rate (211 GB/s), though all are physically contiguous and in the same
        memory zone; a block placed there stalls every step it is read in."""
        todo = [r for seg in self.segments for r in range(*seg)
                if self.good[r] and self.fast[r] is None]
        if not todo:
            return
        dst = torch.empty(_HUGE, dtype=torch.uint8, device=device)
        s = torch.cuda.Stream(device=device)
        for rep in range(2):
            evs = []
            with torch.cuda.stream(s):
                for r in todo:
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(s)
                    dst.copy_(self.view(r * _HUGE, _HUGE), non_blocking=True)
                    e1.record(s)
                    evs.append((r, e0, e1))
            s.synchronize()
        for r, e0, e1 in evs:
            self.rate[r] = _HUGE / (e0.elapsed_time(e1) * 1e6)
        rates = sorted(x for x in self.rate if x is not None)
        ref = rates[len(rates) // 2]
        for r in todo:
            self.fast[r] = self.rate[r] >= min_frac * ref
        del dst

    def place_surveyed(self, sizes, align=256, min_frac=0.6):
        """Offsets (from .ptr) for pieces of the given sizes, placed only in
        runs of huge-page ranges that streamed at the link rate in a survey
        (see survey()) and never across a registration segment.  Ranges are
        prepared, registered and surveyed in rounds until the fast ones hold
        every piece; if the reservation runs out first, the remaining pieces
        go to any registered space.  Registers as it goes (no register()
        afterwards)."""
        if self.small:
            offs = self.place(sizes, align)
            self.register()
            return offs
        sizes = [int(n) for n in sizes]
        need = sum(_round_up(n, align) for n in sizes)
        want = -(-need // _HUGE) + len(sizes) // 16 + 2
        n_ranges = self.capacity // _HUGE
        while True:
            usable = sum(1 for r, f in enumerate(self.fast) if f and self.good[r])
            short = want - usable
            if short > 0 and len(self.good) < n_ranges:
                self._prepare(min(n_ranges, len(self.good) + short))
                self.register()
                self.survey(min_frac)
                continue
            offs = self._fit(sizes, align)
            if offs is not None or len(self.good) >= n_ranges:
                break
            want += max(2, want // 8)
        if offs is None:
            offs = self._fit(sizes, align, any_range=True)
        if offs is None:
            raise MemoryError("PinnedBuffer: the pieces do not fit")
        return offs

    def _fit(self, sizes, align, any_range=False):
        """First-fit of the pieces into runs of usable ranges inside one
        registration segment each; None if some piece finds no room."""
        def usable(r):
            return any_range or (self.good[r] and self.fast[r])
        offs = []
        taken = []                          # (start, end) byte spans handed out
        for n in sizes:
            found = None
            for a, b in self.segments:
                pos = a * _HUGE
                while pos + n <= b * _HUGE:
                    pos = _round_up(pos, align)
                    first, last = pos // _HUGE, (pos + n - 1) // _HUGE
                    if last >= b:
                        break
                    bad = [r for r in range(first, last + 1) if not usable(r)]
                    if bad:
                        pos = (bad[-1] + 1) * _HUGE
                        continue
                    clash = [e for s, e in taken if s < pos + n and e > pos]
                    if clash:
                        pos = max(clash)
                        continue
                    found = pos
                    break
                if found is not None:
                    break
            if found is None:
                return None
            offs.append(found)
            taken.append((found, found + n))
        return offs

    def view(self, offset, nbytes):
        return self._t[self.offset + offset:self.offset + offset + nbytes]

    def survey_summary(self):
        """Counts and rates of the surveyed ranges (None if none were)."""
        rates = [x for x in self.rate if x is not None]
        if not rates:
            return None
        rates.sort()
        return {"ranges": len(rates), "slow": sum(1 for f in self.fast if f is False),
                "median_gbs": rates[len(rates) // 2], "min_gbs": rates[0]}

    def good_fraction(self):
        """Fraction of the prepared 512 MiB ranges backed by a huge page
        (None for a small buffer, which uses base pages)."""
        if self.small or not self.good:
            return None
        return sum(self.good) / len(self.good)

    def huge_fraction(self):
        """Fraction of the mapping's resident bytes backed by huge pages
        (from /proc/self/smaps), or None where that is not readable."""
        try:
            with open("/proc/self/smaps") as fh:
                lines = fh.read().splitlines()
        except OSError:
            return None
        lo, hi = self.ptr, self.ptr + self.capacity
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
            for p in getattr(self, "_reg_ptrs", []):
                torch.cuda.cudart().cudaHostUnregister(p)
            self._reg_ptrs = []
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
    """The pinned shards of `w.distinct` host blocks.  For every host block
    and dtype group g, the group's shards sit at a constant stride (the
    shard bytes rounded up to 256) inside one huge-page-backed piece, so a
    prefetch can move each group as one 2-D DMA."""

    def __init__(self, w: W.Workload, seed=0, gen_device="cpu", keep_params=False, params=None):
        self.w = w
        self.descs = W.block_param_descs(w)
        self.plan = dlo.Plan(self.descs, w.shards)
        self.groups = self.plan.groups()
        s = w.shards
        self.strides = [_round_up(g.shard_alloc_bytes, 256) for g in self.groups]
        piece = [s * st for st in self.strides]
        self.buf = PinnedBuffer(w.distinct * sum(_round_up(p, 256) for p in piece), spare=0.5,
                                defer=True)
        where = self.buf.place_surveyed([piece[g] for _ in range(w.distinct)
                                         for g in range(len(self.groups))])
        self.offsets = []                  # [hb][g * s + r] offsets from buf.ptr
        for hb in range(w.distinct):
            offs = []
            for g, st in enumerate(self.strides):
                o = where[hb * len(self.groups) + g]
                offs += [o + r * st for r in range(s)]
            self.offsets.append(offs)
        self.params = [] if keep_params else None
        for hb in range(w.distinct):
            if params is not None:
                p = params[hb]
            else:
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
        return [self.buf.ptr + o for o in self.offsets[hb]]

    def shard_views(self, hb):
        """uint8 tensors over the shards of host block hb, [g * s + r]."""
        out = []
        for i, o in enumerate(self.offsets[hb]):
            g = self.groups[i // self.w.shards]
            out.append(self.buf.view(o, g.shard_alloc_bytes))
        return out

    def close(self):
        self.buf.close()


class StreamedStack:
    """Two slots and the hook schedule: the path the pages describe."""

    def __init__(self, host: HostBlocks, copy_mode=dlo.COPY_AUTO, copy_ctas=0, timing=False,
                 device="cuda", two_copy_streams=False, log_capacity=0):
        w = host.w
        self.w, self.host, self.plan = w, host, host.plan
        self.slot_bytes = _round_up(self.plan.info().slot_bytes, 256)
        self.slots = [torch.empty(self.slot_bytes, dtype=torch.uint8, device=device)
                      for _ in range(2)]
        self.compute = torch.cuda.Stream(device=device)
        self.copy = torch.cuda.Stream(device=device)
        self.staging, self.gather, staging_bytes = None, None, 0
        if copy_mode == dlo.COPY_STAGED:
            # the two-phase form: H2D into device staging, then a
            # device-to-device gather on a third stream
            staging_bytes = _round_up(self.plan.info().staging_bytes, 256)
            self.staging = [torch.empty(staging_bytes, dtype=torch.uint8, device=device)
                            for _ in range(2)]
            self.gather = torch.cuda.Stream(device=device)
        self.engine = dlo.Engine(w.n_blocks, self.slots[0], self.slots[1], self.slot_bytes,
                                 self.compute, self.copy, copy_mode, copy_ctas, timing,
                                 staging=self.staging, staging_bytes=staging_bytes,
                                 gather_stream=self.gather, two_copy_streams=two_copy_streams,
                                 log_capacity=log_capacity)
        for i in range(w.n_blocks):
            self.engine.register_block(i, self.plan, host.shard_ptrs(i % w.distinct))
        self.cfg = dlo.dit_cfg(w.batch, w.tokens, w.hidden, w.heads, w.mlp, w.eps,
                               **W.cfg_flags(w))
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


class SourceStack:
    """The rank-local path ([D5] "Rank-local path without DLO AllGather"):
    one shard, blocks registered by the host addresses of their parameters
    (host.params, ordinary pageable tensors).  transport "pageable": CPU
    threads pack each block into one of two pinned host staging slots before
    its DMA; "registered": the parameters' memory is page-locked (all or
    nothing) and copied straight into the slots."""

    def __init__(self, host: HostBlocks, transport="pageable", pack_threads=0, timing=False,
                 device="cuda"):
        w = host.w
        if w.shards != 1 or host.params is None:
            raise ValueError("SourceStack needs a one-shard HostBlocks with keep_params=True")
        self.w, self.host, self.plan, self.transport = w, host, host.plan, transport
        self.slot_bytes = _round_up(self.plan.info().slot_bytes, 256)
        self.slots = [torch.empty(self.slot_bytes, dtype=torch.uint8, device=device)
                      for _ in range(2)]
        self.compute = torch.cuda.Stream(device=device)
        self.copy = torch.cuda.Stream(device=device)
        self.srcs = [[host.params[hb][name].data_ptr() for name, _, _ in host.descs]
                     for hb in range(w.distinct)]
        self.reg = None
        self.hs = None
        staging = None
        if transport == "registered":
            ptrs, sizes = [], []
            for hb in range(w.distinct):
                for name, _, _ in host.descs:
                    t = host.params[hb][name]
                    ptrs.append(t.data_ptr())
                    sizes.append(t.numel() * t.element_size())
            dlo.host_register_ranges(ptrs, sizes)
            self.reg = (ptrs, sizes)
        else:
            self.hs = PinnedBuffer(2 * self.slot_bytes, defer=True)
            offs = self.hs.place_surveyed([self.slot_bytes, self.slot_bytes])
            staging = [self.hs.ptr + o for o in offs]
        self.engine = dlo.Engine(w.n_blocks, self.slots[0], self.slots[1], self.slot_bytes,
                                 self.compute, self.copy, dlo.COPY_DMA, 0, timing,
                                 host_staging=staging,
                                 host_staging_bytes=self.slot_bytes if staging else 0,
                                 pack_threads=pack_threads)
        for i in range(w.n_blocks):
            self.engine.register_block_source(i, self.plan, self.srcs[i % w.distinct])
        self.cfg = dlo.dit_cfg(w.batch, w.tokens, w.hidden, w.heads, w.mlp, w.eps,
                               **W.cfg_flags(w))
        self.scratch_bytes = dlo.forward_scratch_bytes(self.cfg)
        self.scratch = torch.empty(self.scratch_bytes, dtype=torch.uint8, device=device)
        self.primed = False

    def prime(self):
        self.engine.prefetch(0, 0)
        self.primed = True

    def step(self, x):
        if not self.primed:
            self.prime()
        for i in range(self.w.n_blocks):
            self.engine.block_forward(i, self.cfg, x, self.scratch, self.scratch_bytes)

    def close(self):
        if self.engine is not None:
            self.engine.destroy()
            self.engine = None
        if self.reg is not None:
            dlo.host_unregister_ranges(*self.reg)
            self.reg = None
        if self.hs is not None:
            self.hs.close()
            self.hs = None


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
        self.cfg = dlo.dit_cfg(w.batch, w.tokens, w.hidden, w.heads, w.mlp, w.eps,
                               **W.cfg_flags(w))
        self.scratch_bytes = dlo.forward_scratch_bytes(self.cfg)
        self.scratch = torch.empty(self.scratch_bytes, dtype=torch.uint8, device=device)

    def block(self, i, x):
        dlo.forward(self.cfg, self.plan, self.bufs[i % self.w.distinct], x, self.scratch,
                    self.scratch_bytes, self.stream)

    def step(self, x):
        for i in range(self.w.n_blocks):
            self.block(i, x)
