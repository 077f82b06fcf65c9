"""Assembles block stacks from the C ABI: pinned host shards, a streamed
two-slot engine, and an all-resident reference over the same kernels.

PyTorch provides device memory, pinned host memory and streams only; every
step of the method runs in the library (``dlo``).
"""
import torch

from . import dlo
from . import workloads as W


def _round_up(v, a):
    return (v + a - 1) // a * a


class PinnedBuffer:
    """Page-locked, device-mapped host bytes of an exact size.

    Allocated as ordinary host memory and registered with the CUDA driver
    (cudaHostRegister, portable | mapped), so the size is not rounded the way
    a caching pinned allocator rounds it."""

    def __init__(self, nbytes):
        self.nbytes = int(nbytes)
        self._t = torch.empty(self.nbytes + 4096, dtype=torch.uint8)
        base = self._t.data_ptr()
        self.ptr = _round_up(base, 4096)
        self.offset = self.ptr - base
        rt = torch.cuda.cudart()
        err = rt.cudaHostRegister(self.ptr, self.nbytes, 1 | 2)   # portable | mapped
        code = err.value if hasattr(err, "value") else int(err)
        if code != 0:
            raise RuntimeError("cudaHostRegister of %d bytes failed (%d)" % (self.nbytes, code))
        self.registered = True

    def view(self, offset, nbytes):
        return self._t[self.offset + offset:self.offset + offset + nbytes]

    def close(self):
        if self.registered:
            torch.cuda.cudart().cudaHostUnregister(self.ptr)
            self.registered = False

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
