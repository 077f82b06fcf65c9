"""Benchmark of the streamed per-block weight stream on GB300.

One bench step is one denoising step of the workload: every block once,
each block's weights streamed host->device into a slot (prefetch of block
i+1 overlapping block i's forward) and the block forward run on them.

Prints one JSON line:
  value       streamed block forwards per second (whole job, all ranks),
              inputs (pinned host shards, x on the device) in place before
              the timed region, the engine as it runs in use; the K timed
              steps run as 5 regions (each bracketed by a device
              synchronisation) and value is the median region's rate;
  e2e         the same, with x copied from pinned host memory (PinnedIO
              buffers) and the result read back every step inside the timed
              region;
  h2d_gbs     bytes moved host->device / copy-stream busy time, from a
              second pass of the same steps with an event pair around every
              prefetch (the copy statistics come from that pass);
  exposed_transfer_ms_per_step  streamed minus all-resident step time;
  roofline    the dominant operation: where the link bounds the block, the
              host->device copy against the measured pinned cudaMemcpyAsync
              ceiling of this machine; where compute does, fc2 (the largest
              linear, on CTA pairs) timed alone against the measured bf16
              peak;
  roofline_h2d, roofline_compute  both of these, always;
  cpu_baseline the CPU oracle on a bounded sample of the same workload.

--impl reference times the CPU oracle (the reference arm of this build):
each step is one oracle block forward of the same workload on the host
cores (for blocks above 1e11 FLOPs a bounded 1/H share of one, see
oracle_sample); under torchrun only rank 0 runs it.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "streamed block-fwd/s; H2D GB/s vs roofline; exposed transfer ms/step (1×GB300)"
UNIT = "block-fwd/s"
DEFAULT_CONFIG = "super"
# DRAM bytes (read + written) per launch of fc2 from an ncu capture of that
# shape (M, K, N, on CTA pairs): python bench.py --only fc2 --config super
# --reps 3, then ncu --set full --clock-control none -k regex:gemm_pair -s 2
# -c 1 on the same command (4.343 GB read, 0.194 GB written)
FC2_DRAM_BYTES = {(8192, 24576, 6144, True): 3_064_119_000 + 189_118_720}
REGIONS = 5          # timed regions per pass; value is the median region


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: enough for about 1.5 s, at least 20; "
                         "the reference arm: 20)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--copy-mode", default="auto", choices=["auto", "dma", "kernel", "staged"])
    ap.add_argument("--copy-ctas", type=int, default=0)
    ap.add_argument("--two-copy-streams", action="store_true",
                    help="prefetches into slot 1 on a second copy stream")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--gen-device", default=None, help="cpu or cuda (default: by size)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true",
                    help="do not sample nvidia-smi during the timed region (diagnostics)")
    ap.add_argument("--dump-copies", action="store_true",
                    help="add every timed prefetch's duration to the JSON line")
    ap.add_argument("--pretouch", type=int, default=1,
                    help="1: read every pinned host block once from the GPU before timing")
    ap.add_argument("--verify", type=int, default=1,
                    help="1: after the shards are written, time every host block's copy and "
                         "relocate the slow ones (setup, untimed)")
    ap.add_argument("--heal", default="auto", choices=["auto", "on", "off"],
                    help="move host blocks whose copies turn slow while the stream runs "
                         "(auto: for blocks of 128 MB or more, where timing every copy costs "
                         "nothing measurable)")
    ap.add_argument("--only", default=None,
                    choices=["linear", "qkv", "fc2", "outproj", "attention", "norm", "copy",
                             "forward"],
                    help="run one kernel of the workload's block `--reps` times (for ncu)")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--gemm-pair", default="auto", choices=["auto", "on", "off"],
                    help="GEMM kernel of the linears: by shape (auto), CTA pairs for all (on), "
                         "single CTAs for all (off)")
    ap.add_argument("--launch-overlap", default="auto", choices=["auto", "on", "off"],
                    help="programmatic dependent launch between the forward's kernels "
                         "(auto: for blocks below 1e11 FLOPs)")
    ap.add_argument("--source", default="shards", choices=["shards", "pageable", "registered"],
                    help="shards: pinned host shards (default); pageable / registered: the "
                         "rank-local path with one shard, blocks by parameter address")
    ap.add_argument("--source-pages", default="huge", choices=["huge", "base"],
                    help="--source registered: the parameters' memory as huge pages (a "
                         "huge-page-backed mapping) or the tensors' own base pages")
    ap.add_argument("--layout", default="dit", choices=["dit", "mxfp8", "int8"],
                    help="with --only copy: the block's linears as bf16 (dit) or in a 1-byte layout")
    ap.add_argument("--sweep", action="store_true",
                    help="run the transfer-vs-compute sweep (36 cells), one JSON line per cell")
    ap.add_argument("--sweep-d", default="1664,3328,6656")
    ap.add_argument("--sweep-t", default="256,4096,16384")
    ap.add_argument("--sweep-s", default="1,2,4,8")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def union_ms(spans):
    """Total length of the union of [start, end] intervals (ms)."""
    total, cur_s, cur_e = 0.0, None, None
    for s, e in sorted(spans):
        if cur_e is None or s > cur_e:
            if cur_e is not None:
                total += cur_e - cur_s
            cur_s, cur_e = s, e
        else:
            cur_e = max(cur_e, e)
    if cur_e is not None:
        total += cur_e - cur_s
    return total


def region_sizes(steps, regions=REGIONS):
    """Splits `steps` timed steps into up to `regions` regions, as evenly as
    possible (the earlier regions take the remainder)."""
    n = max(1, min(regions, steps))
    return [steps // n + (1 if i < steps % n else 0) for i in range(n)]


def median_region(sizes, ms):
    """Index of the median region by rate (steps per ms)."""
    order = sorted(range(len(sizes)), key=lambda i: sizes[i] / ms[i])
    return order[len(order) // 2]


def timed_regions(step, stream, sizes, ws):
    """Runs sum(sizes) steps as one timed region, bracketed by a barrier and
    a device synchronisation on both sides, with a CUDA event on `stream`
    (the stream the steps end on) after every sizes[i] steps, so that the
    regions follow each other without a pause (the stream stays in its
    steady state); returns each region's time in ms, the maximum over
    ranks."""
    import torch
    barrier(ws)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(sizes) + 1)]
    ev[0].record(stream)
    for i, k in enumerate(sizes):
        for _ in range(k):
            step()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    return [max_over_ranks(ev[i].elapsed_time(ev[i + 1]), ws) for i in range(len(sizes))]


def max_over_ranks(v, ws):
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while a region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.pre = None

    def start(self):
        """Starts sampling and returns once the first sample is in (at most
        3 s), so that the samples kept come from the region that follows."""
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        import select
        ready, _, _ = select.select([self.proc.stdout], [], [], 3.0)
        if ready:
            self.pre = self.proc.stdout.readline()   # the sample taken before the region

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        lines = out.splitlines()
        adjacent = False
        if not any(len(l.split(",")) >= 9 for l in lines):
            # a region shorter than the sampling interval: the samples just
            # before and just after it stand in, marked as such
            adjacent = True
            lines = [self.pre or ""]
            try:
                lines += subprocess.run(
                    ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                     "-i", str(self.index)], capture_output=True, text=True,
                    timeout=10).stdout.splitlines()
            except (OSError, subprocess.SubprocessError):
                pass
        sm, smax, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            try:
                power.append(float(f[3]))
            except ValueError:
                pass
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        res = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
               "reasons": sorted(reasons), "samples": len(sm),
               "power_w": statistics.median(power) if power else None}
        if adjacent:
            res["adjacent"] = "region shorter than the 200 ms sampling interval: samples " \
                              "taken just before and just after it"
        return res


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return d.get("bf16_tflops"), d.get("bf16_tflops_sustained"), d.get("hbm_gbs"), "measured"
    except (OSError, ValueError):
        return 1900.0, 1700.0, 6800.0, "fallback"


FULL_ORACLE_FLOPS = 1e11   # blocks up to this run whole in the oracle samples


def oracle_sample(w, seed=0, gen_device="cpu"):
    """One bounded piece of the fp64 oracle's work on host block 0 of `w`:
    returns (run, share, text), run() doing the piece once, share the
    fraction of one block forward's FLOPs it is.

    A block of at most FULL_ORACLE_FLOPS runs whole (oracle.block_forward,
    share 1).  A larger one (Nano, Super, the T = 16384 sweep cells, where
    one oracle forward takes minutes) is sampled as 1/H of a block, H the
    head count: the oracle's QKV projection and attention for head 0 over
    all T tokens of the first batch item (1/H of those FLOPs), then its
    out-projection, gated residual, second norm, MLP (GELU included) and
    gated residual on round(B*T/H) token rows (the out-projection's input
    is head 0's attention output in its columns, zeros in the others).
    The first norm runs over all T rows (a little more than 1/H of it);
    share is the piece's exact dense-contraction FLOPs over the block's."""
    import numpy as np
    import oracle
    from layerwise_weight_offload_gb300 import workloads as W
    p = {k: v.float().cpu().numpy() for k, v in W.gen_block(w, 0, seed, device=gen_device).items()}
    x = W.gen_x(w, seed, device=gen_device).cpu().numpy()
    threads = oracle.default_threads()
    rb = W.oracle_rope_base(w)
    if w.flops_per_block() <= FULL_ORACLE_FLOPS:
        def run():
            oracle.block_forward(x, p, w.batch, w.tokens, w.hidden, w.heads, w.mlp, w.eps,
                                 threads=threads, rope_base=rb)
        return run, 1.0, "one fp64 oracle block forward of host block 0 of %s" % w.name, threads
    d, f, T, H = w.hidden, w.mlp, w.tokens, w.heads
    hd = d // H
    r = max(1, round(w.batch * T / H))
    wqkv = p["attn.qkv.weight"]
    w_head = np.ascontiguousarray(np.concatenate([wqkv[0:hd], wqkv[d:d + hd],
                                                  wqkv[2 * d:2 * d + hd]]))
    x0, xr = x[:T], x[:r]

    def run():
        h = oracle.rmsnorm_mod(x0, p["norm1.weight"], p["ada1.shift"], p["ada1.scale"], w.eps)
        qkv_h = oracle.linear(h, w_head, threads)
        o_h = oracle.attention(qkv_h, 1, T, hd, 1, threads)
        o_r = np.zeros((r, d))
        o_r[:, :hd] = o_h[np.arange(r) % T]
        y = oracle.linear(o_r, p["attn.out.weight"], threads)
        x1 = xr.astype(np.float64) + p["ada1.gate"].astype(np.float64) * y
        h2 = oracle.rmsnorm_mod(x1, p["norm2.weight"], p["ada2.shift"], p["ada2.scale"], w.eps)
        u = oracle.gelu_tanh_array(oracle.linear(h2, p["mlp.fc1.weight"], threads))
        y2 = oracle.linear(u, p["mlp.fc2.weight"], threads)
        return x1 + p["ada2.gate"].astype(np.float64) * y2

    flops = 2 * T * d * 3 * hd + 4 * T * T * hd + 2 * r * (d * d + 2 * d * f)
    text = ("1/%d of an fp64 oracle block forward of host block 0 of %s: QKV projection and "
            "attention of head 0 over all %d tokens, out-projection, norms, MLP and residuals "
            "on %d token rows (%.3g FLOPs of the block's %.3g)"
            % (H, w.name, T, r, flops, w.flops_per_block()))
    return run, flops / w.flops_per_block(), text, threads


def oracle_block_rate(w, seconds, seed=0, gen_device="cpu"):
    """CPU oracle block forwards per second on a bounded sample: the
    oracle_sample piece of host block 0, repeated until `seconds` have
    passed (at least once), counted as `share` block forwards each."""
    run, share, text, threads = oracle_sample(w, seed, gen_device)
    n, t0 = 0, time.perf_counter()
    while True:
        run()
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return n * share / el, n, el, threads, text


def oracle_extras(w, seed=0, seconds=3.0):
    """The oracle's other two figures: its shard-reassembly throughput on the
    bf16 group of one block of `w` (element-wise copies, one thread), and its
    block-forward rate on one thread, taken on the tiny workload (a
    one-thread forward of the larger ones takes minutes)."""
    import numpy as np
    import oracle
    from layerwise_weight_offload_gb300 import workloads as W
    rng = np.random.default_rng(seed)
    n = w.bf16_numel()
    flat = rng.integers(0, 256, size=2 * n, dtype=np.uint8)
    shards = oracle.shard(flat, n, 2, w.shards)
    S = oracle.shard_numel(n, w.shards)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.reassemble(shards, S, 2)
        reps += 1
        if time.perf_counter() - t0 >= seconds / 2:
            break
    gbs = reps * w.shards * S * 2 / ((time.perf_counter() - t0) * 1e9)
    t = W.CONFIGS["tiny"]
    p = {k: v.float().numpy() for k, v in W.gen_block(t, 0, seed).items()}
    x = W.gen_x(t, seed).numpy()
    k, t0 = 0, time.perf_counter()
    while True:
        oracle.block_forward(x, p, t.batch, t.tokens, t.hidden, t.heads, t.mlp, t.eps, threads=1)
        k += 1
        if time.perf_counter() - t0 >= seconds / 2:
            break
    return {"oracle_reassemble_gbs": gbs,
            "oracle_reassemble_sample": "%d reassemblies of the %s bf16 group (%d shards)"
                                        % (reps, w.name, w.shards),
            "one_thread_tiny_block_fwd_per_s": k / (time.perf_counter() - t0),
            "one_thread_sample": "%d fp64 oracle forwards of a tiny block on 1 thread" % k}


def run_reference(args, ws, rank):
    """The oracle as the reference arm: K timed steps (after W untimed) of
    one oracle_sample piece each on the host cores, counted as `share`
    block forwards per step."""
    if rank != 0:
        return
    from layerwise_weight_offload_gb300 import workloads as W
    w = W.CONFIGS[args.config]
    run, share, text, threads = oracle_sample(w, args.seed)
    if args.steps is None:
        args.steps = 20
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    el = time.perf_counter() - t0
    v = args.steps * share / el
    sample = "%d steps, each %s" % (args.steps, text)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": DATA, "config": workload_config(w, args, ws),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


DATA = ("synthetic: seeded torch.randn, bf16 linear weights ~N(0,0.02), f32 adaLN ~N(0,0.1), "
        "norm gains 1, x ~N(0,1)")


def workload_config(w, args, ws=1):
    """The workload as both arms name it (the same dict in each)."""
    mb = (w.bf16_numel() * 2 + w.f32_numel() * 4) * w.n_blocks / 1e6
    return {"workload": "%s: %d blocks/step (%d distinct host blocks), hidden %d, %d heads, "
                        "mlp %d, %d tokens, batch %d, %d shards per dtype group, %d denoising "
                        "steps in the workload" % (w.name, w.n_blocks, w.distinct, w.hidden,
                                                   w.heads, w.mlp, w.tokens, w.batch, w.shards,
                                                   w.steps),
            "name": w.name, "copy_mode": args.copy_mode, "host_source": args.source,
            "gemm_pair": args.gemm_pair, "launch_overlap": args.launch_overlap,
            "l2": "streamed weights %.0f MB per step > 129 MB L2" % mb,
            "parallelism": "replicas" if ws > 1 else "single GPU"}


def h2d_ceiling_gbs(torch, nbytes=1 << 30, reps=10):
    """Pinned host -> device cudaMemcpyAsync ceiling of this machine (best of reps)."""
    from layerwise_weight_offload_gb300.stack import PinnedBuffer
    buf = PinnedBuffer(nbytes)
    src = buf.view(0, nbytes)
    src.fill_(1)
    dst = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    best = float("inf")
    with torch.cuda.stream(s):
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            dst.copy_(src, non_blocking=True)
            b.record(s)
            b.synchronize()
            best = min(best, a.elapsed_time(b))
    s.synchronize()
    del dst
    buf.close()
    return nbytes / best / 1e6


def apply_gemm_pair(dlo, args):
    dlo.set_gemm_pair_mode({"auto": dlo.GEMM_PAIR_AUTO, "on": dlo.GEMM_PAIR_ON,
                            "off": dlo.GEMM_PAIR_OFF}[args.gemm_pair])
    dlo.set_launch_overlap({"auto": -1, "on": 1, "off": 0}[args.launch_overlap])


def run_ours(args, ws, rank, local):
    import torch
    from layerwise_weight_offload_gb300 import build as B
    B.build()
    from layerwise_weight_offload_gb300 import dlo, workloads as W
    apply_gemm_pair(dlo, args)
    from layerwise_weight_offload_gb300.stack import (HostBlocks, StreamedStack, ResidentStack,
                                                      PinnedIO, IOHealer)

    torch.cuda.set_device(local)
    w = W.CONFIGS[args.config]
    mode = {"auto": dlo.COPY_AUTO, "dma": dlo.COPY_DMA, "kernel": dlo.COPY_KERNEL,
            "staged": dlo.COPY_STAGED}[args.copy_mode]
    bf16_peak, bf16_sust, hbm_peak, peak_src = measured_peaks()
    ceiling = h2d_ceiling_gbs(torch)

    gen_dev = args.gen_device or ("cuda" if w.distinct * w.bf16_numel() > 2e9 else "cpu")
    if args.source != "shards":
        w = W.Workload(**{**w.__dict__, "shards": 1})
    host = HostBlocks(w, seed=args.seed, gen_device=gen_dev,
                      keep_params=args.source != "shards")
    bytes_per_block = sum(g.shard_bytes * w.shards for g in host.plan.groups())
    pretouch_s = None
    if args.pretouch:
        # setup, untimed: one device-side pass over every pinned host block
        t0 = time.perf_counter()
        host.pretouch()
        pretouch_s = time.perf_counter() - t0
    host_verify = None
    if args.verify and args.source == "shards":
        # setup, untimed: every host block's copy timed after the weights are
        # in place; the slow ones move to fresh host ranges
        t0 = time.perf_counter()
        host_verify = host.verify()
        host_verify["seconds"] = time.perf_counter() - t0
    heal = args.source == "shards" and (
        args.heal == "on" or (args.heal == "auto" and bytes_per_block >= 128 << 20))

    def make_stack(timing):
        if args.source != "shards":
            from layerwise_weight_offload_gb300.stack import SourceStack
            return SourceStack(host, transport=args.source, timing=timing,
                               pages=args.source_pages)
        return StreamedStack(host, copy_mode=mode, copy_ctas=args.copy_ctas, timing=timing,
                             two_copy_streams=args.two_copy_streams, heal=heal)

    x0 = W.gen_x(w, args.seed, device="cuda")
    x = x0.clone()
    cur = torch.cuda.current_stream()

    def run_steps(stack, n):
        stack.compute.wait_stream(cur)
        for _ in range(n):
            stack.step(x)
        cur.wait_stream(stack.compute)

    # Two passes of the same length.  The first measures the stream as it
    # runs in use (no per-copy timing events: a timing event recorded between
    # two block copies on the copy queue costs the link ~3% of a 25 MB copy);
    # it gives `value`, the step time and the clocks.  The second records an
    # event pair around every prefetch for the copy statistics (H2D GB/s,
    # busy time, overlap, the copy-time distribution).
    st = make_stack(False)
    run_steps(st, args.warmup)
    torch.cuda.synchronize()
    if args.steps is None:
        # enough timed steps for REGIONS regions of about 1.5 s of device
        # time each (at least 20 steps), so that every region's clock
        # samples and copies are many; one more untimed step measures the
        # step time
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st.compute)
        st.step(x)
        e1.record(st.compute)
        torch.cuda.synchronize()
        est = e0.elapsed_time(e1)
        args.steps = int(max_over_ranks(
            max(20, min(50000, math.ceil(REGIONS * 1500.0 / max(est, 1e-3)))), ws))
    sizes = region_sizes(args.steps)
    stats0 = st.engine.query()
    clocks = ClockSampler(local)
    if not args.no_clocks:
        clocks.start()
    region_ms = timed_regions(lambda: st.step(x), st.compute, sizes, ws)
    clk = clocks.stop()
    stats1 = st.engine.query()
    n_fwd = w.n_blocks * args.steps
    rates = [w.n_blocks * k / (ms / 1e3) for k, ms in zip(sizes, region_ms)]
    med = median_region(sizes, region_ms)
    value = ws * w.n_blocks * sizes[med] / (region_ms[med] / 1e3)
    ms_step = region_ms[med] / sizes[med]
    total_ms = sum(region_ms)
    chosen = dlo.COPY_MODE_NAMES[stats1.chosen_mode]
    # the library's own kernels in the timed region: every forward's launches
    # plus the copy-kernel launches of the prefetches the timed forwards issued
    gpu_launches = (n_fwd * dlo.forward_launches(st.cfg) +
                    stats1.n_copy_kernel_launches - stats0.n_copy_kernel_launches)

    # second pass: the same steps with every prefetch timed
    stt = make_stack(True)
    x.copy_(x0)
    run_steps(stt, args.warmup)
    torch.cuda.synchronize()
    n_copies_before = len(stt.engine.copy_times()[0])
    dropped_before = stt.engine.query().timed_dropped
    t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0e.record(stt.compute)
    for _ in range(args.steps):
        stt.step(x)
    t1e.record(stt.compute)
    torch.cuda.synchronize()
    ms_timed_step = t0e.elapsed_time(t1e) / args.steps
    stats_t = stt.engine.query()
    copy_ms, copy_bytes = stt.engine.copy_times()
    spans_all = stt.engine.copy_spans()
    # the prefetches enqueued by the timed forwards (the last one prefetches
    # block 0 of the next step); the setup and warm-up ones are excluded.
    # The timing record keeps the newest entries: shift by what it dropped.
    first = n_copies_before - (stats_t.timed_dropped - dropped_before)
    if first < 0:
        raise RuntimeError("timing record too small for %d timed prefetches" % n_fwd)
    copy_ms, copy_bytes = copy_ms[first:first + n_fwd], copy_bytes[first:first + n_fwd]
    spans = spans_all[first:first + n_fwd]
    # prefetches into the two slots run on two copy streams and may overlap:
    # the copy engines' busy time is the union of the intervals
    busy_ms = union_ms(spans)
    h2d = sum(copy_bytes) / (busy_ms * 1e6) if busy_ms > 0 else None
    qs = sorted(copy_ms)
    copy_dist = {"min": qs[0], "p50": qs[len(qs) // 2],
                 "p99": qs[min(len(qs) - 1, int(math.ceil(0.99 * len(qs))) - 1)],
                 "max": qs[-1], "n": len(qs),
                 "slow_over_2x_p50": sum(1 for v in qs if v > 2 * qs[len(qs) // 2]),
                 "first": copy_ms[:3], "last": copy_ms[-3:]} if qs else None
    chosen_t = dlo.COPY_MODE_NAMES[stats_t.chosen_mode]
    heal_log_t = list(getattr(stt, "heal_log", []))
    stt.close()

    # all-resident reference run: same kernels, no transfer, the same regions
    rs = ResidentStack(host)
    xr = x0.clone()
    rs.stream.wait_stream(cur)
    for _ in range(args.warmup):
        rs.step(xr)
    clocks_r = ClockSampler(local)
    if not args.no_clocks:
        clocks_r.start()
    res_region_ms = timed_regions(lambda: rs.step(xr), rs.stream, sizes, ws)
    clk_res = clocks_r.stop()
    rmed = median_region(sizes, res_region_ms)
    res_ms_step = res_region_ms[rmed] / sizes[rmed]
    exposed = ms_step - res_ms_step
    copy_per_step = busy_ms / args.steps
    overlap = 1.0 - exposed / copy_per_step if copy_per_step > 0 else None

    # block roofline: max(bytes / link ceiling, flops / bf16 peak), the
    # peak being the measured burst figure (the sustained one as a second
    # field: the streamed step is a long run under the power cap)
    flops = w.flops_per_block()
    t_link = bytes_per_block / (ceiling * 1e9)
    t_comp = flops / (bf16_peak * 1e12)
    t_comp_sust = flops / (bf16_sust * 1e12)
    t_roof = max(t_link, t_comp)
    roof_frac = (w.n_blocks * t_roof * 1e3) / ms_step
    roof_frac_sust = (w.n_blocks * max(t_link, t_comp_sust) * 1e3) / ms_step

    # fc2 alone (T x f -> d, gated residual), event-timed on its stream: the
    # top kernel of the step's launch list on the large workloads (its
    # operands, 403 MB of A at Super, exceed L2)
    M, K, N = w.batch * w.tokens, w.mlp, w.hidden
    a = torch.randn(M, K, device="cuda").to(torch.bfloat16)
    wt = (0.02 * torch.randn(N, K, device="cuda")).to(torch.bfloat16)
    xr2 = torch.randn(M, N, device="cuda")
    gate = 0.1 * torch.randn(N, device="cuda")
    nws = dlo.op_linear_workspace_bytes(M, N, K, dlo.EPI_RESID_F32)
    lws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda")
    ls = torch.cuda.Stream()
    ls.wait_stream(cur)
    for _ in range(3):
        dlo.op_linear(a, M, K, wt, N, dlo.EPI_RESID_F32, xr2, gate, ls, lws, nws)
    l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 20
    l0.record(ls)
    for _ in range(reps):
        dlo.op_linear(a, M, K, wt, N, dlo.EPI_RESID_F32, xr2, gate, ls, lws, nws)
    l1.record(ls)
    torch.cuda.synchronize()
    lin_ms = l0.elapsed_time(l1) / reps
    lin_tflops = 2.0 * M * K * N / (lin_ms * 1e-3) / 1e12
    lin_pair = bool(dlo.op_linear_on_pairs(M, N, K, dlo.EPI_RESID_F32))
    del a, wt, xr2, lws

    # end to end through the public API: x in from pinned host, result out
    e2e = None
    if not args.no_e2e:
        # End to end, as a serving loop runs it: every step's input is copied
        # from pinned host memory and its result read back inside the timed
        # region, double-buffered, so that step s+1's input lands and step
        # s's result returns while step s computes.  The input goes through
        # the weight stream's copy queue (between the block copies, rather
        # than beside them on a second host-to-device queue); the result
        # returns on a data stream (the other direction of the link).
        # the step's input and its two result buffers in the library's
        # huge-page pinned memory, each copy direction checked (PinnedIO)
        xb = x0.numel() * x0.element_size()
        io = PinnedIO(xb, 3)
        io_rates = io.verify(0.5 * ceiling)
        xh = io.tensor(0, x0.shape, x0.dtype)
        xh.copy_(x0.cpu())
        yh = [io.tensor(1 + i, x0.shape, x0.dtype) for i in range(2)]
        xd = [torch.empty_like(x) for _ in range(2)]
        data = torch.cuda.Stream()
        h2d_ev = [torch.cuda.Event() for _ in range(2)]
        done_ev = [torch.cuda.Event() for _ in range(2)]
        rb_ev = [torch.cuda.Event() for _ in range(2)]
        # timing events around every input copy and result read-back
        io_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
                 for _ in range(args.steps)]
        step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        in_q = st.copy if hasattr(st, "copy") else data
        # Host ranges can turn slow after the check above, during the pass:
        # the input and result copies that have completed are read after each
        # step is queued (no wait on the GPU), and a buffer whose copy ran
        # over 4x the link time moves to fresh huge-page ranges (IOHealer);
        # the copies queued after the move use the new place.
        io_healer = IOHealer(io, ceiling)
        io_checked = 0

        def io_heal(upto):
            nonlocal xh, io_checked
            while io_checked < upto and io_ev[io_checked][3].query():
                k = io_checked
                io_checked += 1
                times = [(0, io_ev[k][0].elapsed_time(io_ev[k][1])),
                         (1 + (k & 1), io_ev[k][2].elapsed_time(io_ev[k][3]))]
                for i in io_healer.observe(times):
                    if not io_healer.move(k, i, dict(times)[i], 0.25 * ceiling):
                        continue
                    if i == 0:
                        xh = io.tensor(0, x0.shape, x0.dtype)
                    else:
                        yh[i - 1] = io.tensor(i, x0.shape, x0.dtype)
        # untimed: one step on each device buffer, so that the forward's cached
        # CUDA graphs for these buffers exist before the timed region
        st.compute.wait_stream(cur)
        for b in range(2):
            xd[b].copy_(x0)
            st.compute.wait_stream(cur)
            st.step(xd[b])
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        barrier(ws)
        clocks_e = ClockSampler(local)
        if not args.no_clocks:
            clocks_e.start()
        e0.record(in_q)
        with torch.cuda.stream(in_q):
            io_ev[0][0].record(in_q)
            xd[0].copy_(xh, non_blocking=True)
            io_ev[0][1].record(in_q)
        h2d_ev[0].record(in_q)
        for s in range(args.steps):
            b = s & 1
            st.compute.wait_event(h2d_ev[b])
            if s == 0:
                step_ev[0].record(st.compute)
            st.step(xd[b])
            done_ev[b].record(st.compute)
            step_ev[s + 1].record(st.compute)
            with torch.cuda.stream(data):
                data.wait_event(done_ev[b])
                io_ev[s][2].record(data)
                yh[b].copy_(xd[b], non_blocking=True)
                io_ev[s][3].record(data)
                rb_ev[b].record(data)
            if s + 1 < args.steps:
                # the other buffer's last reader was step s-1: its result
                # read-back must be done before the next input lands there
                with torch.cuda.stream(in_q):
                    if s >= 1:
                        in_q.wait_event(rb_ev[b ^ 1])
                    io_ev[s + 1][0].record(in_q)
                    xd[b ^ 1].copy_(xh, non_blocking=True)
                    io_ev[s + 1][1].record(in_q)
                    h2d_ev[b ^ 1].record(in_q)
            io_heal(s)
        data.wait_stream(in_q)
        e1.record(data)
        torch.cuda.synchronize()
        clk_e2e = clocks_e.stop()
        e_ms = max_over_ranks(e0.elapsed_time(e1), ws)
        x_in_ms = sorted(ev[0].elapsed_time(ev[1]) for ev in io_ev)
        y_out_ms = sorted(ev[2].elapsed_time(ev[3]) for ev in io_ev)
        # compute-stream time of each step (from the end of the previous one,
        # so a step that waited for its input counts the wait)
        e_steps = [step_ev[i].elapsed_time(step_ev[i + 1]) for i in range(args.steps)]
        e_step_ms = sorted(e_steps)
        # the value pass's regions over the same steps: the first from before
        # step 0's input copy, the last to the end of the last read-back, so
        # that the regions add up to the whole pass
        bounds = [0]
        for k in sizes:
            bounds.append(bounds[-1] + k)
        marks = [e0] + [step_ev[b] for b in bounds[1:-1]] + [e1]
        e_region_ms = [max_over_ranks(marks[i].elapsed_time(marks[i + 1]), ws)
                       for i in range(len(sizes))]
        e_rates = [ws * w.n_blocks * k / (ms / 1e3) for k, ms in zip(sizes, e_region_ms)]
        emed = median_region(sizes, e_region_ms)
        e2e = {"value": e_rates[emed], "unit": UNIT,
               "whole_pass_value": ws * n_fwd / (e_ms / 1e3),
               "block_fwd_per_s_per_region": e_rates,
               "timing": "median of the value pass's regions over the same steps (the first "
                         "from before step 0's input copy, the last to the end of the last "
                         "read-back: together the whole pass, whole_pass_value)",
               "h2d_bytes_per_step": xb + w.n_blocks * bytes_per_block,
               "d2h_bytes_per_step": xb,
               "clocks": clk_e2e,
               "x_in_ms": {"p50": x_in_ms[len(x_in_ms) // 2], "max": x_in_ms[-1]},
               "result_out_ms": {"p50": y_out_ms[len(y_out_ms) // 2], "max": y_out_ms[-1]},
               "step_ms": {"p50": e_step_ms[len(e_step_ms) // 2], "max": e_step_ms[-1],
                           "min": e_step_ms[0], "first": e_steps[:3],
                           "before_first": e0.elapsed_time(step_ev[0])},
               "io_buffers": {"kind": "PinnedIO: huge-page pinned host memory, surveyed, each "
                                      "copy direction verified",
                              "h2d_gbs": [round(a, 1) for a, _ in io_rates],
                              "d2h_gbs": [round(b, 1) for _, b in io_rates],
                              "relocated": io.relocated, "failed": io.failed,
                              "moved_during_pass": io_healer.log,
                              "moved_note": "(step, buffer 0 = input / 1, 2 = results, copy ms, "
                                            "new place fast)"},
               "note": "h2d counts x plus every streamed weight shard of the step; x in and "
                       "the result out are double-buffered; x goes through the weight copy "
                       "stream, the result returns on a data stream; run after the value, "
                       "timed-copy and resident passes (clocks: sampled during this pass)"}
        del xh, yh
        io.close()

    status = dlo.kernel_status()
    if status != 0:
        raise RuntimeError("a kernel wait timed out (device status %d)" % status)
    st.close()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, n, el, threads, text = oracle_block_rate(w, args.cpu_seconds, args.seed,
                                                    gen_device="cuda")
        cpu = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": "%d x (%s) in %.1f s; the oracle's reassembly is not included"
                         % (n, text, el),
               **oracle_extras(w, args.seed)}

    # the dominant operation: the block's host->device copy where the link
    # bounds the step, else the top GEMM (fc2) timed alone
    roof_h2d = {"name": None, "bound": "h2d", "peak": ceiling, "unit": "GB/s",
                "traffic": None,
                "peak_source": "pinned cudaMemcpyAsync 1 GiB ceiling measured in this run",
                "bytes_per_launch": bytes_per_block,
                "timing": "CUDA events around every prefetch of the timed steps "
                          "(copy_stats_pass); busy time per block"}
    fc2_traffic = FC2_DRAM_BYTES.get((M, K, N, lin_pair))
    roof_gemm = {"name": ("gemm_pair_kernel<2>" if lin_pair else "gemm_tcgen05_kernel<2>")
                 + " (fc2, gated residual)", "bound": "tensor", "achieved": lin_tflops,
                 "peak": bf16_peak, "unit": "TFLOP/s", "frac": lin_tflops / bf16_peak,
                 "traffic": fc2_traffic,
                 "traffic_note": ("dram__bytes_read.sum + dram__bytes_write.sum per launch, "
                                  "from an ncu capture of this shape" if fc2_traffic
                                  else "no ncu capture of this shape"),
                 "flops_per_launch": 2 * M * K * N, "algorithmic_bytes_per_launch":
                     2 * M * K + 2 * N * K + 8 * M * N,
                 "peak_source": peak_src + " burst bf16 (the kernel is timed alone)",
                 "shape": [M, K, N], "ms": lin_ms,
                 "timing": "20 back-to-back launches alone on one stream, CUDA events"}
    copy_name = {"kernel": "copy_reassemble_kernel",
                 "staged": "cudaMemcpyAsync into staging (copy engines), then a device gather"}.get(
        chosen, "cudaMemcpyAsync (copy engines)")
    # per launch: one block's bytes over the busy time per block
    achieved = (sum(copy_bytes) / len(copy_bytes)) / (busy_ms / len(copy_ms) * 1e6) \
        if copy_ms and busy_ms > 0 else None
    roof_h2d.update(name=copy_name, achieved=achieved,
                    frac=achieved / ceiling if achieved else None)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": DATA, "config": workload_config(w, args, ws), "chosen_copy_mode": chosen,
        "timing": {"regions": len(sizes), "steps_per_region": sizes,
                   "streamed_ms_per_region": region_ms,
                   "streamed_block_fwd_per_s_per_region": [ws * r for r in rates],
                   "streamed_ms_per_step_all_steps": total_ms / args.steps,
                   "resident_ms_per_region": res_region_ms,
                   "note": "the K timed steps run back to back as these regions (CUDA events "
                           "between them, one synchronisation before and after); value, "
                           "ms_per_step and resident_ms_per_step are the median region's"},
        "h2d_gbs": h2d, "h2d_ceiling_gbs": ceiling,
        "h2d_nominal_pcie5_x16_gbs": 63.0,
        "exposed_transfer_ms_per_step": exposed,
        "exposed_transfer_fraction_of_step": exposed / ms_step,
        "resident_ms_per_step": res_ms_step,
        "copy_busy_ms_per_step": copy_per_step, "overlap_fraction": overlap,
        "block_roofline_fraction": roof_frac,
        "block_roofline_fraction_sustained_peak": roof_frac_sust,
        "block_roofline": {"bytes_per_block": bytes_per_block, "flops_per_block": flops,
                           "t_link_ms": t_link * 1e3, "t_compute_ms": t_comp * 1e3,
                           "t_compute_sustained_ms": t_comp_sust * 1e3,
                           "bf16_peak_tflops": bf16_peak, "bf16_sustained_tflops": bf16_sust,
                           "peak_source": peak_src + " burst bf16 (the sustained figure for "
                                          "block_roofline_fraction_sustained_peak)",
                           "bound": "h2d" if t_link >= t_comp else "tensor"},
        "auto_race_us_per_forward": {"dma": stats1.race_dma_us, "kernel": stats1.race_kernel_us},
        "copy_stats_pass": {
            "ms_per_step": ms_timed_step, "chosen_copy_mode": chosen_t,
            "note": "h2d_gbs, copy_busy_ms_per_step, overlap_fraction, copy_ms_distribution "
                    "and roofline come from this second pass of the same steps, with an event "
                    "pair recorded around every prefetch; value, ms_per_step and clocks come "
                    "from the first pass, without them"},
        "copy_ms_distribution": copy_dist, "pretouch_s": pretouch_s,
        "host_verify": host_verify,
        "heal": {"enabled": heal,
                 "moves_value_pass": [list(m) for m in getattr(st, "heal_log", [])],
                 "moves_copy_stats_pass": [list(m) for m in heal_log_t],
                 "note": "(forwards so far, host block, moved to a range that streamed at "
                         "speed); the value pass's moves include those of its warm-up and of "
                         "the e2e pass, which runs on the same stack"},
        "host_huge_page_fraction": host.buf.huge_fraction(),
        "host_huge_ranges_used_fraction": host.buf.good_fraction(),
        "host_range_survey": host.buf.survey_summary(),
        "source_path": ({"transport": args.source, "pages": args.source_pages,
                         "direct_prefetches": stats1.n_direct_prefetches,
                         "packed_prefetches": stats1.n_packed_prefetches,
                         "pack_ms_per_packed_block": (stats1.pack_ms - stats0.pack_ms) /
                         max(1, stats1.n_packed_prefetches - stats0.n_packed_prefetches)}
                        if args.source != "shards" else None),
        "copy_ms_all": copy_ms if args.dump_copies else None,
        "roofline": roof_h2d if t_link >= t_comp else roof_gemm,
        "roofline_h2d": roof_h2d,
        "roofline_compute": roof_gemm,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": gpu_launches,
        "clocks": clk,
        "clocks_resident_pass": clk_res,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_only(args):
    """One kernel of the workload's block, `reps` event-timed launches on one
    stream; prints the mean time.  Sized by the workload, one host block."""
    import torch
    from layerwise_weight_offload_gb300 import build as B
    B.build()
    from layerwise_weight_offload_gb300 import dlo, workloads as W
    apply_gemm_pair(dlo, args)
    from layerwise_weight_offload_gb300.stack import HostBlocks, ResidentStack
    w = W.CONFIGS[args.config]
    w = W.Workload(**{**w.__dict__, "distinct": 1, "n_blocks": 1})
    M, d, f, H = w.batch * w.tokens, w.hidden, w.mlp, w.heads
    s = torch.cuda.Stream()
    dev = "cuda"
    if args.only == "linear":
        a = torch.randn(M, d, device=dev).to(torch.bfloat16)
        wt = (0.02 * torch.randn(f, d, device=dev)).to(torch.bfloat16)
        out = torch.empty(M, f, dtype=torch.bfloat16, device=dev)
        fn = lambda: dlo.op_linear(a, M, d, wt, f, dlo.EPI_GELU_BF16, out, None, s)
    elif args.only == "qkv":
        # the QKV linear's shape (its V-transposing epilogue runs only inside
        # the block forward; the bf16 store stands in for it)
        a = torch.randn(M, d, device=dev).to(torch.bfloat16)
        wt = (0.02 * torch.randn(3 * d, d, device=dev)).to(torch.bfloat16)
        out = torch.empty(M, 3 * d, dtype=torch.bfloat16, device=dev)
        fn = lambda: dlo.op_linear(a, M, d, wt, 3 * d, dlo.EPI_BF16, out, None, s)
    elif args.only == "fc2":
        a = torch.randn(M, f, device=dev).to(torch.bfloat16)
        wt = (0.02 * torch.randn(d, f, device=dev)).to(torch.bfloat16)
        x = torch.randn(M, d, device=dev)
        gate = 0.1 * torch.randn(d, device=dev)
        nws = dlo.op_linear_workspace_bytes(M, d, f, dlo.EPI_RESID_F32)
        ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)
        fn = lambda: dlo.op_linear(a, M, f, wt, d, dlo.EPI_RESID_F32, x, gate, s, ws, nws)
    elif args.only == "outproj":
        a = torch.randn(M, d, device=dev).to(torch.bfloat16)
        wt = (0.02 * torch.randn(d, d, device=dev)).to(torch.bfloat16)
        x = torch.randn(M, d, device=dev)
        gate = 0.1 * torch.randn(d, device=dev)
        nws = dlo.op_linear_workspace_bytes(M, d, d, dlo.EPI_RESID_F32)
        ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)
        fn = lambda: dlo.op_linear(a, M, d, wt, d, dlo.EPI_RESID_F32, x, gate, s, ws, nws)
    elif args.only == "attention":
        qkv = torch.randn(M, 3 * d, device=dev).to(torch.bfloat16)
        o = torch.empty(M, d, dtype=torch.bfloat16, device=dev)
        nb = dlo.op_attention_scratch_bytes(w.batch, w.tokens, d)
        sc = torch.empty(nb, dtype=torch.uint8, device=dev)
        fn = lambda: dlo.op_attention(qkv, w.batch, w.tokens, d, H, o, sc, nb, s)
    elif args.only == "norm":
        x = torch.randn(M, d, device=dev)
        g = torch.ones(d, device=dev)
        z = torch.zeros(d, device=dev)
        h = torch.empty(M, d, dtype=torch.bfloat16, device=dev)
        fn = lambda: dlo.op_rmsnorm_mod(x, M, d, g, z, z, 1e-6, h, s)
    elif args.only == "copy" and args.layout != "dit":
        return run_copy_layout(args, w)
    else:
        host = HostBlocks(w, seed=args.seed, gen_device="cuda")
        if args.only == "copy":
            dst = torch.empty(host.plan.info().slot_bytes, dtype=torch.uint8, device=dev)
            ptrs = host.shard_ptrs(0)
            mode = dlo.COPY_DMA if args.copy_mode == "dma" else dlo.COPY_KERNEL
            fn = lambda: dlo.reassemble(host.plan, ptrs, dst, mode, s)
        else:
            rs = ResidentStack(host, stream=s)
            x = W.gen_x(w, args.seed, device=dev)
            fn = lambda: rs.block(0, x)
    for _ in range(2):          # first calls: module loading, attributes, graph capture
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(args.reps):
        fn()
    e1.record(s)
    torch.cuda.synchronize()
    assert dlo.kernel_status() == 0
    print(json.dumps({"only": args.only, "config": args.config, "reps": args.reps,
                      "gemm_pair": args.gemm_pair, "launch_overlap": args.launch_overlap,
                      "ms_per_rep": e0.elapsed_time(e1) / args.reps}), flush=True)


def run_copy_layout(args, w):
    """Reassembly of one block whose linears are in a 1-byte layout (fp8 +
    e8m0 block scales, or int8 + fp32 row scales; some weights transposed
    views): random bytes in surveyed pinned shards, both copy modes timed
    over `reps` prefetch-sized reassemblies each."""
    import numpy as np
    import torch
    from layerwise_weight_offload_gb300 import dlo, workloads as W
    from layerwise_weight_offload_gb300.stack import PinnedBuffer
    descs = W.block_param_descs_quantized(w, args.layout)
    plan = dlo.Plan(descs, w.shards)
    groups = plan.groups()
    sizes = [g.shard_alloc_bytes for g in groups for _ in range(w.shards)]
    buf = PinnedBuffer(sum(-(-n // 256) * 256 for n in sizes), spare=0.5, defer=True)
    offs = buf.place_surveyed(sizes)
    ptrs = [buf.ptr + o for o in offs]
    rng = np.random.default_rng(args.seed)
    srcs = []
    for p in range(plan.info().n_params):
        pi = plan.param(p)
        srcs.append(rng.integers(0, 256, size=pi.storage_numel * dlo.ESIZE[pi.dtype],
                                 dtype=np.uint8))
    plan.shard_host([x.ctypes.data for x in srcs], ptrs)
    nbytes = sum(g.shard_bytes * w.shards for g in groups)
    dst = torch.empty(plan.info().slot_bytes, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    ceiling = h2d_ceiling_gbs(torch)
    res = {}
    for name, mode in (("dma", dlo.COPY_DMA), ("kernel", dlo.COPY_KERNEL)):
        for _ in range(2):
            dlo.reassemble(plan, ptrs, dst, mode, s)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(args.reps):
            dlo.reassemble(plan, ptrs, dst, mode, s)
        e1.record(s)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.reps
        res[name] = {"ms_per_block": ms, "gbs": nbytes / (ms * 1e6),
                     "frac_of_ceiling": nbytes / (ms * 1e6) / ceiling}
    assert dlo.kernel_status() == 0
    print(json.dumps({"only": "copy", "config": args.config, "layout": args.layout,
                      "shards": w.shards, "bytes_per_block": nbytes,
                      "groups": [(g.dtype, g.shard_bytes) for g in groups],
                      "h2d_ceiling_gbs": ceiling, "reps": args.reps, **res}), flush=True)
    buf.close()


def run_sweep(args):
    """The transfer-vs-compute sweep: for every (hidden d, tokens T, shards s)
    cell, 16 blocks per step streamed through the engine (AUTO copy mode)
    and the same blocks all resident; prints one JSON line per cell with the
    streamed and resident step times, exposed transfer, overlap and the
    block-roofline fraction.  Weights are drawn once per d and re-sharded
    per s; one set of pinned shards serves all T."""
    import torch
    from layerwise_weight_offload_gb300 import build as B
    B.build()
    from layerwise_weight_offload_gb300 import dlo, workloads as W
    apply_gemm_pair(dlo, args)
    from layerwise_weight_offload_gb300.stack import HostBlocks, StreamedStack, ResidentStack
    bf16_peak, bf16_sust, _, _ = measured_peaks()
    ceiling = h2d_ceiling_gbs(torch)
    for d in [int(v) for v in args.sweep_d.split(",")]:
        base = W.CONFIGS["sweep-d%d-t256-s1" % d]
        params = []
        for hb in range(base.distinct):
            p = W.gen_block(base, hb, args.seed, device="cuda")
            params.append({k: v.cpu().contiguous() for k, v in p.items()})
        torch.cuda.empty_cache()
        for s in [int(v) for v in args.sweep_s.split(",")]:
            w0 = W.CONFIGS["sweep-d%d-t256-s%d" % (d, s)]
            host = HostBlocks(w0, params=params)
            host.pretouch()
            verify = host.verify()
            bytes_hb = sum(g.shard_bytes * s for g in host.plan.groups())
            for T in [int(v) for v in args.sweep_t.split(",")]:
                w = W.CONFIGS["sweep-d%d-t%d-s%d" % (d, T, s)]
                host.w = w
                x = W.gen_x(w, args.seed, device="cuda")
                cur = torch.cuda.current_stream()
                steps = 3 if T < 16384 else 2
                warm = 3

                heal = bytes_hb >= 128 << 20

                def timed_pass(timing):
                    # the step time without per-copy timing events (as the
                    # stream runs in use; blocks of 128 MB or more heal, which
                    # times every copy at no measurable cost); with them, the
                    # copy statistics
                    stk = StreamedStack(host, copy_mode=dlo.COPY_AUTO, timing=timing,
                                        heal=heal)
                    stk.compute.wait_stream(cur)
                    for _ in range(warm):
                        stk.step(x)
                    torch.cuda.synchronize()
                    nb = len(stk.engine.copy_times()[0]) if timing else 0
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stk.compute)
                    for _ in range(steps):
                        stk.step(x)
                    b.record(stk.compute)
                    torch.cuda.synchronize()
                    return stk, nb, a.elapsed_time(b) / steps

                st, _, ms = timed_pass(False)
                moves = [list(m) for m in st.heal_log]
                st.close()
                st, n_before, _ = timed_pass(True)
                cms, cby = st.engine.copy_times()
                cms = cms[n_before:n_before + w.n_blocks * steps]
                cby = cby[n_before:n_before + w.n_blocks * steps]
                busy = union_ms(st.engine.copy_spans()[n_before:n_before + w.n_blocks * steps])
                chosen = dlo.COPY_MODE_NAMES[st.engine.query().chosen_mode]
                st.close()
                rs = ResidentStack(host)
                xr = W.gen_x(w, args.seed, device="cuda")
                rs.stream.wait_stream(cur)
                rs.step(xr)
                r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                r0.record(rs.stream)
                for _ in range(steps):
                    rs.step(xr)
                r1.record(rs.stream)
                torch.cuda.synchronize()
                res = r0.elapsed_time(r1) / steps
                del rs
                bytes_block = sum(g.shard_bytes * s for g in host.plan.groups())
                t_link = bytes_block / (ceiling * 1e9)
                t_roof = max(t_link, w.flops_per_block() / (bf16_peak * 1e12))
                t_roof_s = max(t_link, w.flops_per_block() / (bf16_sust * 1e12))
                copy_step = busy / steps
                exposed = ms - res
                print(json.dumps({
                    "cell": w.name, "hidden": d, "tokens": T, "shards": s, "blocks": w.n_blocks,
                    "streamed_ms_per_step": ms, "resident_ms_per_step": res,
                    "exposed_transfer_ms_per_step": exposed,
                    "copy_ms_per_step": copy_step,
                    "h2d_gbs": sum(cby) / (busy * 1e6) if busy > 0 else None,
                    "overlap_fraction": 1 - exposed / copy_step if copy_step > 0 else None,
                    "block_fwd_per_s": w.n_blocks / (ms / 1e3),
                    "block_roofline_fraction": w.n_blocks * t_roof * 1e3 / ms,
                    "block_roofline_fraction_sustained_peak": w.n_blocks * t_roof_s * 1e3 / ms,
                    "bound": "h2d" if t_link >= w.flops_per_block() / (bf16_peak * 1e12)
                    else "tensor",
                    "copy_mode": chosen, "copy_max_ms": max(cms) if cms else None,
                    "host_verify_relocated": verify["relocated"],
                    "heal_moves": moves + [list(m) for m in st.heal_log]}), flush=True)
                del x, xr
                torch.cuda.empty_cache()
            host.close()
            del host
    if dlo.kernel_status() != 0:
        raise RuntimeError("a kernel wait timed out")


def main():
    args = parse()
    if args.only:
        run_only(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    ws, rank, local = dist_env()
    if args.warmup < 3:
        args.warmup = 3
    if ws > 1:
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return
        else:
            import torch
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_ours(args, ws, rank, local)
    if ws > 1 and args.impl != "reference":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
