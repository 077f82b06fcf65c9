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

    def __init__(self, nbytes, spare=0.25, tries=3, defer=False, extra_ranges=0, huge=None):
        """extra_ranges: 512 MiB ranges reserved beyond the spare room for
        relocate() (address space only until used).  huge: True to use
        huge-page ranges whatever the size (None: only from SMALL up)."""
        self.nbytes = int(nbytes)
        self.small = self.nbytes < self.SMALL if huge is None else not huge
        n_ranges = max(1, -(-self.nbytes // _HUGE))
        self.capacity = (_round_up(self.nbytes, 1 << 16) if self.small
                         else (n_ranges + int(n_ranges * spare) + 2 + extra_ranges) * _HUGE)
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

    def relocate(self, pieces, min_gbs, align=256, device="cuda"):
        """Moves pieces [(offset, nbytes)] (from .ptr) into fresh huge-page
        ranges after the prepared ones, back to back at `align`: each new
        range's first touch is the data itself (copied from the old place,
        which stays intact), then collapse, registration and one timed
        host->device copy of the new span after a warm-up copy.  Returns the
        new offsets if that copy reached min_gbs, else None (the new ranges
        are then marked slow and left unused).  The old ranges are marked
        slow either way.  Needs room in the reservation (spare); None if
        there is none.

        Why: on some GB300 hosts ranges that passed the placement survey
        stream at 3-30 GB/s once the weights are written into them, on every
        later pass, idle or under compute; a block there stalls the stream
        each time it is read."""
        if self.small:
            return None
        offs, pos = [], 0
        for _, n in pieces:
            pos = _round_up(pos, align)
            offs.append(pos)
            pos += int(n)
        k = -(-pos // _HUGE)
        r0 = len(self.good)
        if (r0 + k) * _HUGE > self.capacity:
            return None
        base = r0 * _HUGE
        for (old, n), o in zip(pieces, offs):
            ctypes.memmove(self.ptr + base + o, self.ptr + old, int(n))
        if pos < k * _HUGE:
            ctypes.memset(self.ptr + base + pos, 0, k * _HUGE - pos)
        for r in range(k):
            ok = any(_collapse(self.ptr + base + r * _HUGE, _HUGE) for _ in range(self.tries))
            self.good.append(ok)
            self.rate.append(None)
            self.fast.append(None)
        self.register()
        for old, n in pieces:
            for r in range(old // _HUGE, (old + int(n) - 1) // _HUGE + 1):
                self.fast[r] = False
        dst = torch.empty(pos, dtype=torch.uint8, device=device)
        st = torch.cuda.Stream(device=device)
        ms = None
        with torch.cuda.stream(st):
            for _ in range(2):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(st)
                dst.copy_(self.view(base, pos), non_blocking=True)
                b.record(st)
                b.synchronize()
                ms = a.elapsed_time(b)
        del dst
        gbs = pos / (ms * 1e6)
        good = gbs >= min_gbs and all(self.good[r0:r0 + k])
        for r in range(r0, r0 + k):
            self.rate[r] = gbs
            self.fast[r] = good
        return [base + o for o in offs] if good else None

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


class PinnedIO:
    """Page-locked host buffers for what a step moves besides the weights,
    its input copied in and its result read back, placed like the weight
    shards: in huge-page ranges that streamed at the link rate in a survey
    (PinnedBuffer.place_surveyed), then verify() times every buffer's
    host->device and device->host copy and moves a slow buffer to fresh
    ranges (PinnedBuffer.relocate).  Take views with tensor() after
    verify(): a move changes the buffer's address.

    Why: the host ranges that stall weight copies stall these as well, and
    buffers of a few hundred MB from torch's pinned allocator sit in base
    pages: on one GB300 host a 201 MB input copied at 7.5 GB/s (27 ms, the
    link rate gives 1 ms), and every step waited for it."""

    def __init__(self, nbytes, count, device="cuda"):
        self.nbytes, self.count, self.device = int(nbytes), int(count), device
        per = _round_up(self.nbytes, 256)
        k = -(-per // _HUGE)                  # 512 MiB ranges one moved buffer takes
        # room for two moves of every buffer (address space until used)
        self.buf = PinnedBuffer(per * self.count, defer=True, huge=True,
                                extra_ranges=2 * self.count * k + 1)
        self.offs = self.buf.place_surveyed([self.nbytes] * self.count)
        self.relocated, self.failed, self.rates_gbs = [], [], None

    def tensor(self, i, shape, dtype):
        """Buffer i as a tensor of `shape` and `dtype` (nbytes in all)."""
        t = self.buf.view(self.offs[i], self.nbytes).view(dtype)
        return t.view(shape)

    def rates(self, passes=2):
        """(host->device, device->host) GB/s of each buffer, timed on the
        last of `passes` round trips (the contents are kept)."""
        dev = torch.empty(self.nbytes, dtype=torch.uint8, device=self.device)
        s = torch.cuda.Stream(device=self.device)
        out = []
        for o in self.offs:
            h = self.buf.view(o, self.nbytes)
            for _ in range(passes):
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                with torch.cuda.stream(s):
                    ev[0].record(s)
                    dev.copy_(h, non_blocking=True)
                    ev[1].record(s)
                    h.copy_(dev, non_blocking=True)
                    ev[2].record(s)
                s.synchronize()
            out.append((self.nbytes / (ev[0].elapsed_time(ev[1]) * 1e6),
                        self.nbytes / (ev[1].elapsed_time(ev[2]) * 1e6)))
        del dev
        return out

    def verify(self, min_gbs, rounds=2):
        """Moves every buffer whose copy in either direction is below
        min_gbs to fresh huge-page ranges (its contents move with it), up to
        `rounds` times; returns the last measured rates."""
        for _ in range(rounds):
            rates = self.rates()
            slow = [i for i, (a, b) in enumerate(rates) if min(a, b) < min_gbs]
            if not slow:
                break
            for i in slow:
                new = self.buf.relocate([(self.offs[i], self.nbytes)], min_gbs,
                                        device=self.device)
                if new is None:
                    self.failed.append(i)
                else:
                    self.offs[i] = new[0]
                    self.relocated.append(i)
        else:
            rates = self.rates()
        self.rates_gbs = rates
        return rates

    def close(self):
        self.buf.close()


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
        hb_bytes = sum(_round_up(p, 256) for p in piece)
        # room to relocate up to 8 host blocks (HostBlocks.relocate_block)
        self.buf = PinnedBuffer(w.distinct * hb_bytes, spare=0.5, defer=True,
                                extra_ranges=min(w.distinct, 8) * (-(-hb_bytes // _HUGE)) + 1)
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

    def block_copy_ms(self, passes=2, mode=None, stream=None):
        """Per host block, the time of the last of `passes` reassemblies
        into a scratch slot (DMA by default), as a prefetch moves it."""
        mode = dlo.COPY_DMA if mode is None else mode
        dst = torch.empty(self.plan.info().slot_bytes, dtype=torch.uint8, device="cuda")
        s = stream or torch.cuda.Stream()
        ms = {}
        for _ in range(passes):
            evs = []
            for hb in range(self.w.distinct):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(s)
                dlo.reassemble(self.plan, self.shard_ptrs(hb), dst, mode, s)
                b.record(s)
                evs.append((hb, a, b))
            s.synchronize()
            for hb, a, b in evs:
                ms[hb] = a.elapsed_time(b)
        del dst
        return ms

    def relocate_block(self, hb, min_gbs):
        """Moves host block hb's shards to fresh host ranges (one piece per
        dtype group, the group's shards at their constant stride); True if
        the new place streams at min_gbs (else hb stays where it was)."""
        s = self.w.shards
        pieces = [(self.offsets[hb][g * s], s * st) for g, st in enumerate(self.strides)]
        new = self.buf.relocate(pieces, min_gbs)
        if new is None:
            return False
        offs = []
        for g, st in enumerate(self.strides):
            offs += [new[g] + r * st for r in range(s)]
        self.offsets[hb] = offs
        return True

    def verify(self, factor=1.5, rounds=3):
        """After the shards are written: times every host block's copy (the
        second of two passes) and relocates the blocks slower than `factor`
        x the median by more than 1 ms, up to `rounds` times.  Returns a
        report.  The placement survey times the ranges before the weights
        are written into them; on some hosts ranges turn slow after that."""
        report = {"rounds": 0, "slow_found": [], "relocated": [], "failed": [],
                  "median_ms": None}
        for _ in range(rounds):
            ms = self.block_copy_ms()
            med = sorted(ms.values())[len(ms) // 2]
            report["median_ms"] = report["median_ms"] or med
            slow = [hb for hb, v in ms.items() if v > factor * med and v - med > 1.0]
            report["rounds"] += 1
            if not slow:
                break
            bytes_hb = sum(g.shard_bytes * self.w.shards for g in self.groups)
            for hb in slow:
                report["slow_found"].append((hb, round(ms[hb], 3)))
                ok = self.relocate_block(hb, bytes_hb / (med * 1e6) / factor)
                (report["relocated"] if ok else report["failed"]).append(hb)
        return report

    def close(self):
        self.buf.close()


class IOHealer:
    """Watches the copies of a step's input and result buffers (PinnedIO)
    while a pass runs.  Host ranges can turn slow after PinnedIO.verify,
    during the pass: a buffer whose copy took over `factor` times the link
    time for its bytes (and at least `min_ms`) is named for a move, at most
    `max_moves` times per buffer.  PinnedBuffer.relocate keeps the old place
    intact, so the copies already queued from or into it stay valid and only
    the copies queued after the move use the new place."""

    def __init__(self, io, link_gbs, factor=4.0, min_ms=2.0, max_moves=2):
        self.io = io
        self.slow_ms = max(min_ms, factor * io.nbytes / (link_gbs * 1e6))
        self.max_moves = max_moves
        self.moved = [0] * io.count
        self.log = []

    def observe(self, times):
        """times: [(buffer index, copy ms)] of one completed step; returns
        the buffers to move, in order (slow, each named once, and moved
        fewer than max_moves times so far)."""
        out = []
        for i, ms in times:
            if ms > self.slow_ms and self.moved[i] < self.max_moves and i not in out:
                out.append(i)
        return out

    def move(self, step, i, ms, min_gbs):
        """Moves buffer i to fresh huge-page ranges (contents kept); True if
        the new place streams at min_gbs.  Logged as (step, buffer, copy ms,
        new place fast)."""
        self.moved[i] += 1
        new = self.io.buf.relocate([(self.io.offs[i], self.io.nbytes)], min_gbs,
                                   device=self.io.device)
        self.log.append([step, i, round(ms, 2), new is not None])
        if new is None:
            return False
        self.io.offs[i] = new[0]
        return True


class CopyHealer:
    """Names the host blocks whose prefetches have turned slow, from the
    engine's copy log: a copy is slow when its rate is below the median rate
    of the recent copies divided by `factor` and it took at least
    `min_extra_ms` longer than a copy at that rate would; a host block is
    named once `strikes` of its copies since it last moved were slow, or at
    once after a copy below the median rate divided by `severe` (each copy
    from a slow place stalls the stream, and a second one costs as much as
    the move).  A block that keeps turning slow is named at most `max_moves`
    times."""

    def __init__(self, distinct, factor=2.0, min_extra_ms=1.0, strikes=2, window=512,
                 max_moves=3, severe=4.0):
        self.distinct = distinct
        self.factor, self.min_extra_ms, self.strikes = factor, min_extra_ms, strikes
        self.severe = severe
        self.window, self.max_moves = window, max_moves
        self.rates = []
        self.count = {}
        self.moves = {}

    def observe(self, records):
        """records: (seq, block, slot, ms, bytes) of completed prefetches;
        returns the host blocks to move now."""
        for _, _, _, ms, nbytes in records:
            if ms > 0:
                self.rates.append(nbytes / ms)
        self.rates = self.rates[-self.window:]
        if len(self.rates) < 8:
            return []
        med = sorted(self.rates)[len(self.rates) // 2]
        out = []
        for _, block, _, ms, nbytes in records:
            hb = block % self.distinct
            expect = nbytes / med
            if ms * med < nbytes * self.factor or ms - expect < self.min_extra_ms:
                continue
            hit = self.strikes if ms * med >= nbytes * self.severe else 1
            self.count[hb] = self.count.get(hb, 0) + hit
            if (self.count[hb] >= self.strikes and self.moves.get(hb, 0) < self.max_moves
                    and hb not in out):
                out.append(hb)
        return out

    def moved(self, hb):
        self.count[hb] = 0
        self.moves[hb] = self.moves.get(hb, 0) + 1


class StreamedStack:
    """Two slots and the hook schedule: the path the pages describe."""

    def __init__(self, host: HostBlocks, copy_mode=dlo.COPY_AUTO, copy_ctas=0, timing=False,
                 device="cuda", two_copy_streams=False, log_capacity=0, heal=False,
                 poison=False, checks=False):
        """heal: watch every prefetch's copy time (the engine times each
        one) and, between steps, move host blocks whose copies have turned
        slow to fresh host ranges (CopyHealer, HostBlocks.relocate_block,
        dlo_replace_block_shards).  poison, checks: the engine's debugging
        options (slots overwritten after each forward; every copy's offsets
        checked against the plan before it is issued)."""
        w = host.w
        timing = timing or heal
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
                                 log_capacity=log_capacity, poison=poison, checks=checks)
        for i in range(w.n_blocks):
            self.engine.register_block(i, self.plan, host.shard_ptrs(i % w.distinct))
        self.cfg = dlo.dit_cfg(w.batch, w.tokens, w.hidden, w.heads, w.mlp, w.eps,
                               **W.cfg_flags(w))
        self.scratch_bytes = dlo.forward_scratch_bytes(self.cfg)
        self.scratch = torch.empty(self.scratch_bytes, dtype=torch.uint8, device=device)
        self.primed = False
        self.healer = CopyHealer(w.distinct) if heal else None
        self.heal_since = 0
        self.heal_log = []              # (forwards so far, host block, moved?)

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
        if self.healer is not None:
            self.heal()

    def heal(self, max_moves=4):
        """Reads the completed prefetches since the last call (no wait on
        the GPU) and moves up to max_moves host blocks the healer names."""
        recs, self.heal_since = self.engine.copy_log(self.heal_since)
        todo = self.healer.observe(recs)[:max_moves]
        if not todo:
            return
        bytes_hb = sum(g.shard_bytes * self.w.shards for g in self.host.groups)
        med = sorted(self.healer.rates)[len(self.healer.rates) // 2]
        for hb in todo:
            ok = self.host.relocate_block(hb, med / 1e6 / self.healer.factor)
            if ok:
                for i in range(hb, self.w.n_blocks, self.w.distinct):
                    self.engine.replace_block_shards(i, self.host.shard_ptrs(hb))
            self.healer.moved(hb)
            self.heal_log.append((self.engine.query().n_forwards, hb, ok))

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
    nothing) and copied straight into the slots.

    pages (registered only): "huge" first copies the parameters into an
    anonymous mapping backed by transparent huge pages (what a checkpoint on
    a huge-page-backed file system maps), "base" registers the tensors'
    own memory (base pages).  The GPU streams page-locked memory of 64 KiB
    pages at a fraction of the link rate once the footprint is several GB
    (PinnedBuffer), so only the huge-page form keeps up at scale."""

    def __init__(self, host: HostBlocks, transport="pageable", pack_threads=0, timing=False,
                 device="cuda", pages="huge"):
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
        self.arena = None
        self.base_host = None
        staging = None
        if transport == "registered":
            ptrs, sizes = [], []
            for hb in range(w.distinct):
                for name, _, _ in host.descs:
                    t = host.params[hb][name]
                    ptrs.append(t.data_ptr())
                    sizes.append(t.numel() * t.element_size())
            if pages == "huge":
                # huge-page-backed copies of the parameters, registered below
                # (the arena itself is never registered by PinnedBuffer)
                self.arena = PinnedBuffer(sum(_round_up(n, 256) for n in sizes), spare=0.1,
                                          defer=True)
                offs = self.arena.place(sizes, 256)
                moved = []
                for p, n, o in zip(ptrs, sizes, offs):
                    ctypes.memmove(self.arena.ptr + o, p, n)
                    moved.append(self.arena.ptr + o)
                ptrs = moved
                k = len(host.descs)
                self.srcs = [ptrs[hb * k:(hb + 1) * k] for hb in range(w.distinct)]
                dlo.host_register_ranges(ptrs, sizes)
                self.reg = (ptrs, sizes)
            else:
                # the tensors' own memory, registered once for all the stacks
                # over this HostBlocks (a second registration of a range fails)
                n = getattr(host, "_base_reg_users", 0)
                if n == 0:
                    dlo.host_register_ranges(ptrs, sizes)
                    host._base_reg = (ptrs, sizes)
                host._base_reg_users = n + 1
                self.base_host = host
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
        if self.base_host is not None:
            self.base_host._base_reg_users -= 1
            if self.base_host._base_reg_users == 0:
                dlo.host_unregister_ranges(*self.base_host._base_reg)
            self.base_host = None
        if self.arena is not None:
            self.arena.close()
            self.arena = None
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
