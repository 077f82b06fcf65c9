"""Synthetic workloads of the per-block weight stream: shapes and seeded inputs.

This module holds no arithmetic of the method.  It names the block shapes the
stream is exercised on and draws their inputs from seeded generators, so that
the CUDA path and the CPU oracle can be fed identical tensors.

Block parameters, in registration order (the order in which a DiT block
module would register them; flattening by dtype keeps this order):

    norm1.weight [d] f32, ada1.shift/scale/gate [d] f32,
    attn.qkv.weight [3d, d] bf16, attn.out.weight [d, d] bf16,
    norm2.weight [d] f32, ada2.shift/scale/gate [d] f32,
    mlp.fc1.weight [f, d] bf16, mlp.fc2.weight [d, f] bf16

Values: linear weights ~ N(0, 0.02) rounded to bf16 (round to nearest even),
RMSNorm gains = 1, adaLN shift/scale/gate ~ N(0, 0.1) in f32, activations
x ~ N(0, 1) in f32.  Every tensor has its own torch.Generator seeded from
(seed, block, parameter index), so any block can be regenerated alone.

The checkpoint-shaped variant ("full") adds what real DiT checkpoints carry:
bf16 biases ~ N(0, 0.02) after each linear weight, and fp32 per-head q/k
RMSNorm gains ~ 1 + N(0, 0.1) [hd] after the QKV bias; its forward also
applies rotary position embedding to q and k.
"""
from dataclasses import dataclass, replace

import torch

BF16, F32 = 0, 1          # dtype codes of the C ABI
FP8_E4M3, I8, E8M0 = 3, 5, 7
ESIZE = {BF16: 2, F32: 4}
TORCH_DTYPE = {BF16: torch.bfloat16, F32: torch.float32}


@dataclass(frozen=True)
class Workload:
    name: str
    n_blocks: int         # block forwards per denoising step
    hidden: int           # d
    heads: int            # H (head dim = d / H)
    mlp: int              # f
    tokens: int           # T
    shards: int           # s: data-parallel shards per dtype group
    steps: int            # denoising steps
    distinct: int         # distinct host blocks; block i uses host block i % distinct
    batch: int = 1
    eps: float = 1e-6
    variant: str = "dit"  # "full": biases, q/k RMSNorm and RoPE (checkpoint-shaped)

    @property
    def head_dim(self):
        return self.hidden // self.heads

    def bf16_numel(self):
        d, f = self.hidden, self.mlp
        return 3 * d * d + d * d + f * d + d * f

    def f32_numel(self):
        return 8 * self.hidden

    def flops_per_block(self):
        """Dense-contraction FLOPs of one block forward (elementwise work and
        softmax exponentials are not counted): the four linears plus QK^T and
        PV."""
        d, f, T, B = self.hidden, self.mlp, self.tokens, self.batch
        lin = 2 * B * T * (3 * d * d + d * d + f * d + d * f)
        att = 4 * B * T * T * d
        return lin + att


def _sweep():
    out = {}
    for d in (1664, 3328, 6656):
        for T in (256, 4096, 16384):
            for s in (1, 2, 4, 8):
                name = "sweep-d%d-t%d-s%d" % (d, T, s)
                out[name] = Workload(name, 16, d, d // 128, 4 * d, T, s, 1, 16)
    return out


CONFIGS = {
    "tiny": Workload("tiny", 8, 256, 4, 1024, 256, 2, 1, 8),
    "odd": Workload("odd", 9, 1024, 16, 4096, 1024, 3, 3, 9),
    "nano": Workload("nano", 72, 3840, 30, 15360, 4096, 4, 4, 72),
    "super": Workload("super", 128, 6144, 48, 24576, 8192, 2, 2, 32),
}
CONFIGS["tiny-full"] = replace(CONFIGS["tiny"], name="tiny-full", variant="full")
CONFIGS["odd-full"] = replace(CONFIGS["odd"], name="odd-full", variant="full")
CONFIGS["nano-full"] = replace(CONFIGS["nano"], name="nano-full", variant="full")
CONFIGS.update(_sweep())


def custom(name="custom", **kw):
    base = dict(n_blocks=2, hidden=256, heads=4, mlp=1024, tokens=64, shards=2,
                steps=1, distinct=None)
    base.update(kw)
    if base["distinct"] is None:
        base["distinct"] = base["n_blocks"]
    return Workload(name=name, **base)


def block_param_descs(w: Workload):
    """(name, shape, dtype code) in registration order."""
    d, f = w.hidden, w.mlp
    if w.variant == "full":
        hd = d // w.heads
        return [
            ("norm1.weight", (d,), F32), ("ada1.shift", (d,), F32),
            ("ada1.scale", (d,), F32), ("ada1.gate", (d,), F32),
            ("attn.qkv.weight", (3 * d, d), BF16), ("attn.qkv.bias", (3 * d,), BF16),
            ("attn.q_norm.weight", (hd,), F32), ("attn.k_norm.weight", (hd,), F32),
            ("attn.out.weight", (d, d), BF16), ("attn.out.bias", (d,), BF16),
            ("norm2.weight", (d,), F32), ("ada2.shift", (d,), F32),
            ("ada2.scale", (d,), F32), ("ada2.gate", (d,), F32),
            ("mlp.fc1.weight", (f, d), BF16), ("mlp.fc1.bias", (f,), BF16),
            ("mlp.fc2.weight", (d, f), BF16), ("mlp.fc2.bias", (d,), BF16),
        ]
    return [
        ("norm1.weight", (d,), F32), ("ada1.shift", (d,), F32),
        ("ada1.scale", (d,), F32), ("ada1.gate", (d,), F32),
        ("attn.qkv.weight", (3 * d, d), BF16), ("attn.out.weight", (d, d), BF16),
        ("norm2.weight", (d,), F32), ("ada2.shift", (d,), F32),
        ("ada2.scale", (d,), F32), ("ada2.gate", (d,), F32),
        ("mlp.fc1.weight", (f, d), BF16), ("mlp.fc2.weight", (d, f), BF16),
    ]


def cfg_flags(w: Workload):
    """Keyword arguments of dlo.dit_cfg for the workload's block variant."""
    full = w.variant == "full"
    return {"rope": full, "qk_norm": full}


def oracle_rope_base(w: Workload):
    """rope_base argument of the oracle's block forward for this variant."""
    return 10000.0 if w.variant == "full" else 0.0


def block_param_descs_quantized(w: Workload, kind: str):
    """The same block with its four linears kept in a 1-byte layout, as
    online quantisation finalizes them ([D5] "Request and loading
    constraints"): kind "mxfp8" is an fp8 (e4m3) weight with one e8m0 scale
    per 32 weights along the input dimension, "int8" an int8 weight with one
    fp32 scale per output row.  The QKV and fc1 weights are given as
    transposed views ([in, out] storage seen as [out, in]), the others
    contiguous; the f32 vectors are unchanged.  Shapes only: these blocks are
    moved and reassembled, not computed with."""
    out = []
    for name, shape, code in block_param_descs(w):
        if code != BF16:
            out.append((name, shape, code))
            continue
        o, i = shape
        transposed = name in ("attn.qkv.weight", "mlp.fc1.weight")
        wcode = FP8_E4M3 if kind == "mxfp8" else I8
        out.append((name, shape, wcode, (1, o)) if transposed else (name, shape, wcode))
        if kind == "mxfp8":
            out.append((name + ".scale", (o, i // 32), E8M0))
        else:
            out.append((name + ".scale", (o,), F32))
    return out


def _generator(device, seed, block, index):
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + block) * 64 + index + 1)
    return g


def gen_block(w: Workload, block: int, seed: int = 0, device="cpu"):
    """dict name -> tensor for host block `block` (already reduced mod distinct)."""
    out = {}
    for idx, (name, shape, code) in enumerate(block_param_descs(w)):
        if name.startswith("norm"):
            t = torch.ones(shape, dtype=torch.float32, device=device)
        elif name.endswith("_norm.weight"):
            t = 1.0 + 0.1 * torch.randn(shape, generator=_generator(device, seed, block, idx),
                                        dtype=torch.float32, device=device)
        elif code == F32:
            t = 0.1 * torch.randn(shape, generator=_generator(device, seed, block, idx),
                                  dtype=torch.float32, device=device)
        else:
            t = (0.02 * torch.randn(shape, generator=_generator(device, seed, block, idx),
                                    dtype=torch.float32, device=device)).to(torch.bfloat16)
        out[name] = t
    return out


def gen_x(w: Workload, seed: int = 0, device="cpu"):
    g = _generator(device, seed, 1 << 20, 63)
    return torch.randn((w.batch * w.tokens, w.hidden), generator=g,
                       dtype=torch.float32, device=device)
