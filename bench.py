"""Benchmark of one MLA decode step (one layer) on GB300.

A step is the whole hot path on one batch of synthetic input:
    mla_absorb_q -> mla_decode_paged -> mla_combine_splits -> mla_project_uv
(--fused runs mla_combine_project, the merge inside the W_UV projection,
instead of the last two; it measured slightly slower in the step.)
(mla_decode_paged is one kernel launch for B <= 448, or B <= 352 with
grouped latents: the decode kernel computes its own split; larger batches
add a plan kernel before it.)
Each step is one CUDA-graph replay (the kernels chain by programmatic
dependent launch); the decode kernel is also timed alone, by events around
replays of a graph holding only it.

Default workload: DeepSeek-V3 dims, B=16, Lq=1, H=128, all seq_lens 4096,
64-token pages, contiguous block tables.  Its 75.5 MB cache fits in the
129 MB L2, so the timed loop rotates through 4 copies of the cache (302 MB),
which keeps every step's cache reads coming from HBM; it also rotates
through copies of W_UK and W_UV (2.2x the L2 in all: 9 copies, 302 MB, on
this workload), so that, as in a model with many layers, no step finds its
weights in L2.

Prints ONE JSON line (rank 0).  `value` is latent-KV GB/s of the whole step:
the latent cache bytes one step reads (every cached row once, 1152 B per
token) over the step time.  The step's other algorithmic bytes (weights,
queries, outputs), TFLOP/s, tokens/s and the decode kernel's roofline ride
along.  `--impl reference` times the fp64 CPU oracle on a bounded sample of
the same workload instead.

--kv fp8 runs the same step over the FP8 cache (mla_decode_paged_fp8: E4M3
latent codes with power-of-two block scales, bf16 RoPE key, 656 B a token);
`value` then counts those bytes.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--kv bf16|fp8]
                       [--impl ours|reference]
For N > 1 launch with torchrun; each rank runs its own batch (weak scaling, no
collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MLA decode latent-KV GB/s & TFLOPS per layer, % of GB300 roofline; tokens/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

WORKLOAD_TEXT = {
    "tiny": "tiny MLA decode B=2 Lq=1 H=16 seq {37,200}",
    "dsv3": "DeepSeek-V3-dim decode B=16 Lq=1 H=128 seq 4096 contiguous",
    "long": "long-context decode B=16 Lq=1 H=128 seq U[32768,65536] shuffled pages",
    "spec": "speculative decode B=64 Lq=2 causal H=128 seq U[1024,16384] shuffled pages",
    "gla": "grouped-latent decode G=2 B=32 Lq=1 H=128 seq 8192 contiguous",
    "prefill": "decompress branch: a 1024-token chunk after 3072 cached tokens, B=1 H=128",
}


def rotation_copies(nbytes):
    """Copies of an input of nbytes that a timed loop rotates through so
    that no step finds it in L2: at least 2.2x the L2 in all."""
    return max(1, math.ceil(2.2 * L2_BYTES / nbytes))


def workload_text(args):
    text = WORKLOAD_TEXT[args.workload]
    return text + ", FP8 E4M3 cache" if getattr(args, "kv", "bf16") == "fp8" else text


DECODE_SOURCES = ("mla_latent_kv_10_gb300/csrc/mla_decode.cu", "mla_latent_kv_10_gb300/csrc/ptx.cuh",
                  "mla_latent_kv_10_gb300/csrc/mla_internal.h", "include/mla.h")


def decode_source_sha():
    """sha256 over the decode kernel's translation unit: its .cu and every
    header of this repository it includes, in a fixed order."""
    import hashlib
    h = hashlib.sha256()
    for rel in DECODE_SOURCES:
        h.update(rel.encode())
        h.update(open(os.path.join(ROOT, rel), "rb").read())
    return h.hexdigest()


def decode_traffic(workload, kv="bf16"):
    """DRAM bytes per decode launch from the committed ncu summary of this
    workload, if it was taken on the current decode sources (else None)."""
    name = workload if kv == "bf16" else "%s_%s" % (workload, kv)
    path = os.path.join(ROOT, "profiles", "decode_kernel_%s.json" % name)
    if not os.path.exists(path):
        return None
    rec = json.load(open(path))
    if rec.get("sources_sha256") != decode_source_sha():
        return None
    return rec["dram_bytes_per_launch"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [l.strip().split(",") for l in self.f.read().splitlines() if l.strip()]
        self.f.close()
        os.unlink(self.f.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def roofline_entry(dec_bytes, dec_flops, dec_ms, peaks, traffic, peak_src, kernel="mla_decode_paged"):
    """The binding roof of the decode kernel: the larger of its HBM fraction
    (algorithmic bytes / time against the measured copy bandwidth) and its
    tensor fraction (algorithmic FLOPs / time against the measured bf16
    rate, the burst figure since the kernel is timed alone)."""
    gbs = dec_bytes / (dec_ms * 1e-3) / 1e9
    tfs = dec_flops / (dec_ms * 1e-3) / 1e12
    hbm, tc = peaks["hbm_gbs"], peaks["bf16_tflops"]
    if tfs / tc > gbs / hbm:
        ach, peak, unit, bound = tfs, tc, "TFLOP/s", "tensor"
    else:
        ach, peak, unit, bound = gbs, hbm, "GB/s", "hbm"
    return {"bound": bound, "achieved": ach, "peak": peak, "unit": unit, "frac": ach / peak,
            "traffic": traffic, "peak_source": peak_src, "kernel": kernel}


def max_over_ranks(value, dist, device):
    """The largest of one number over all ranks: a job's time is its slowest
    rank's.  `dist` is torch.distributed with an initialised group (NCCL on
    GPUs, gloo on host cores), or None for a single process."""
    if dist is None:
        return value
    import torch
    x = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(x, op=dist.ReduceOp.MAX)
    return float(x.item())


def job_rate(world, units_per_rank, ms):
    """Whole-job throughput (units per second): what all ranks processed,
    over the max-over-ranks time in milliseconds."""
    return world * units_per_rank / (ms * 1e-3)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args, world, rank):
    """The fp64 oracle timed on host cores over a bounded sample."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    from mla_latent_kv_10_gb300 import accounting as acc
    from mla_latent_kv_10_gb300.inputs import workload

    case = workload(args.workload, kv=args.kv)
    d = case.dims
    seq = case.seq_lens.tolist()
    B, H = d["B"], d["H"]
    kv_bytes = acc.latent_kv_bytes(seq, kv=args.kv)
    step_flops = acc.step_flops(seq, d["Lq"], H, d["G"])
    nt = oracle.num_threads()
    ref_decode = oracle.decode_fp8 if args.kv == "fp8" else oracle.decode
    tensors = case.tensors()
    if args.kv == "fp8":  # read the FP8 rows once, outside the timed calls
        tensors["cache"] = oracle.fp8_as_bf16_cache(case.cache)
        ref_decode = oracle.decode
    rng = np.random.default_rng(0)
    # size one step's sample so the whole run stays within minutes
    pairs_per_step = max(nt, 1)
    times = []
    work = 0.0
    for i in range(args.warmup + args.steps):
        bs = rng.integers(0, B, pairs_per_step)
        hs = rng.integers(0, H, pairs_per_step)
        sel = list(zip(bs.tolist(), hs.tolist()))
        t0 = time.perf_counter()
        ref_decode(d, **tensors, sel=sel, nthreads=nt)
        dt = time.perf_counter() - t0
        frac = sum(seq[b] for b, _ in sel) / (sum(seq) * H)
        if i >= args.warmup:
            times.append(dt)
            work += frac
    total = sum(times)
    value = kv_bytes * work / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / work,  # time the oracle would take for one whole step
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "tflops": step_flops * work / total / 1e12,
        "config": {"workload": workload_text(args), "step": "fused" if args.fused else "four calls", "B": B,
                   "Lq": d["Lq"], "H": H, "G": d["G"], "kv": args.kv,
                   "parallelism": "replicas" if world > 1 else "single"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": nt, "kind": "oracle",
                         "sample": "%d random (sequence, head) pairs per step; metric scaled by the "
                                   "fraction of the step's work they cover%s" % (
                                       pairs_per_step, "; the FP8 rows dequantised once before the timed "
                                       "calls" if args.kv == "fp8" else "")},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def e2e_pipelined(args, mla, torch, dev, stream, case, t, caches, weights, fp8):
    """Mean ms per step of the end-to-end loop (see main), and the H2D / D2H
    bytes each step copies.  The step's inputs (q_nope, q_rope, block table,
    lengths) sit in one pinned host buffer and go up in one copy into one
    device buffer, of which the call gets views."""
    d = case.dims
    keys = ("q_nope", "q_rope", "block_table", "seq_lens")
    src = case.tensors()
    offs, off = {}, 0
    for k in keys:  # 16-byte aligned pieces
        offs[k] = off
        off += (src[k].numel() * src[k].element_size() + 15) // 16 * 16
    h_in = torch.empty(off, dtype=torch.uint8).pin_memory()
    for k in keys:
        n = src[k].numel() * src[k].element_size()
        h_in[offs[k]:offs[k] + n].copy_(src[k].contiguous().view(-1).view(torch.uint8))
    dev_in = [torch.empty(off, dtype=torch.uint8, device=dev) for _ in range(2)]

    def views(buf):
        return {k: buf[offs[k]:offs[k] + src[k].numel() * src[k].element_size()].view(src[k].dtype).view(src[k].shape)
                for k in keys}

    ins = [views(b) for b in dev_in]
    bb = [mla.DecodeBuffers(d, dev) for _ in range(2)]
    h_out = [torch.empty(bb[0].out.shape, dtype=bb[0].out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(src[k].numel() * src[k].element_size() for k in keys)
    d2h = h_out[0].numel() * h_out[0].element_size()
    cs = torch.cuda.Stream(dev)
    ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("in", "done", "out")}
    for j in range(2):  # every event has been recorded once before it is waited on
        for n in ev:
            ev[n][j].record(stream)

    def upload(j):  # on cs: the inputs into set j once the step that last read them is done
        cs.wait_event(ev["done"][j])
        dev_in[j].copy_(h_in, non_blocking=True)
        ev["in"][j].record(cs)

    def run(i, n):
        j = i % 2
        stream.wait_event(ev["in"][j])
        stream.wait_event(ev["out"][j])  # the result two steps back has been read from this buffer
        x = ins[j]  # one mla_decode_step call (the separate calls when a split count is forced)
        w_uk, w_uv = weights[i % len(weights)]
        mla.decode_step(d, bb[j], x["q_nope"], x["q_rope"], w_uk, w_uv, caches[i % len(caches)],
                        x["block_table"], x["seq_lens"], num_splits=args.splits, stream=stream,
                        fused=args.fused, fp8=fp8)
        ev["done"][j].record(stream)
        with torch.cuda.stream(cs):
            if i + 1 < n:
                upload(1 - j)  # the next step's inputs, while this step computes
            cs.wait_event(ev["done"][j])
            h_out[j].copy_(bb[j].out, non_blocking=True)
            ev["out"][j].record(cs)

    with torch.cuda.stream(cs):
        upload(0)
    for i in range(3):
        run(i, 3)
    torch.cuda.synchronize(dev)
    # steady state: at least 200 steps (a loop of a few dozen carries about
    # half a millisecond of start-up in its first steps)
    n = max(args.steps, 200)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    cs.wait_stream(stream)  # the first step's copies inside the timed region too
    with torch.cuda.stream(cs):
        upload(0)
    for i in range(n):
        run(i, n)
    stream.wait_stream(cs)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    for j in range(2):
        status = mla.mla_get_device_status(bb[j].workspace)
        if status != 0:
            raise SystemExit("device status in the end-to-end loop: %s" % mla.mla_status_string(status))
    return e0.elapsed_time(e1) / n, h2d, d2h, n


def cpu_baseline(case, budget_s=12.0, kv="bf16"):
    """Oracle on a bounded sample of the workload, scaled to GB/s."""
    import numpy as np
    import oracle
    from mla_latent_kv_10_gb300 import accounting as acc

    d = case.dims
    seq = case.seq_lens.tolist()
    nt = oracle.num_threads()
    B, H = d["B"], d["H"]
    rng = np.random.default_rng(1)
    kv_bytes = acc.latent_kv_bytes(seq, kv=kv)
    tensors = case.tensors()
    if kv == "fp8":  # the FP8 rows read once (the oracle's reading), then the same decode
        tensors["cache"] = oracle.fp8_as_bf16_cache(case.cache)
    n_pairs = nt
    sel = list(zip(rng.integers(0, B, n_pairs).tolist(), rng.integers(0, H, n_pairs).tolist()))
    t0 = time.perf_counter()
    oracle.decode(d, **tensors, sel=sel, nthreads=nt)
    t1 = time.perf_counter() - t0
    rounds = max(1, int(budget_s / max(t1, 1e-3)) - 1)
    total_t, frac = t1, sum(seq[b] for b, _ in sel) / (sum(seq) * H)
    if rounds > 1 and t1 < budget_s / 2:
        sel2 = list(zip(rng.integers(0, B, n_pairs * rounds).tolist(), rng.integers(0, H, n_pairs * rounds).tolist()))
        t0 = time.perf_counter()
        oracle.decode(d, **tensors, sel=sel2, nthreads=nt)
        total_t += time.perf_counter() - t0
        frac += sum(seq[b] for b, _ in sel2) / (sum(seq) * H)
        n_pairs += len(sel2)
    return {"value": kv_bytes * frac / total_t / 1e9, "unit": "GB/s", "cores": nt, "kind": "oracle",
            "sample": "%d random (sequence, head) pairs of the same workload, %.1f s; scaled by the "
                      "fraction of the step's work they cover" % (n_pairs, total_t)}


def prefill_accounting(seq, Lq, H, G, max_pages):
    """Algorithmic FLOPs and bytes of the decompress branch: the up-projections
    of every cached token (K and V: 2 * 2 * 128 * d_g per token and head)
    and causal attention (2 * (128 + 64) + 2 * 128 per visible (query, key)
    pair and head); bytes: the cache rows, both weights, K and V written
    (whole pages) and read (the pages some query sees), queries in, output
    out."""
    d_g = 512 // G
    tok = sum(seq)
    pages = sum((n + 63) // 64 for n in seq)
    dec_flops = tok * H * 2 * 2 * 128 * d_g
    pairs = sum(sum(n - Lq + l + 1 for l in range(Lq)) for n in seq)
    att_flops = pairs * H * (2 * 192 + 2 * 128)
    kv = pages * 64 * H * 128 * 2 * 2
    dec_bytes = tok * 1152 + 2 * H * 128 * d_g * 2 + kv
    att_bytes = kv + pages * 64 * 64 * 2 + len(seq) * Lq * H * (192 + 128) * 2 + len(seq) * Lq * H * 4
    return dec_flops, att_flops, dec_bytes, att_bytes


def run_prefill(args, world, rank, local):
    """The decompress branch timed as a step: mla_decompress_kv then
    mla_prefill_attend, one CUDA-graph replay per step, each kernel also
    timed alone (graphs of one launch)."""
    import torch
    import mla_latent_kv_10_gb300 as mla
    from mla_latent_kv_10_gb300.inputs import workload

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mla.load_library()
    case = workload("prefill")
    d = case.dims
    seq = case.seq_lens.tolist()
    t = {k: v.to(dev) for k, v in case.tensors().items()}
    bufs = mla.PrefillBuffers(d, dev)
    stream = torch.cuda.current_stream(dev)

    def dec():
        mla.mla_decompress_kv(d, t["cache"], t["block_table"], t["seq_lens"], t["W_UK"], t["W_UV"], bufs.k_nope,
                              bufs.v, bufs.workspace)

    def att():
        mla.mla_prefill_attend(d, t["q_nope"], t["q_rope"], t["cache"], t["block_table"], t["seq_lens"],
                               bufs.k_nope, bufs.v, bufs.out, bufs.lse, bufs.workspace)

    for _ in range(args.warmup):
        dec()
        att()
    torch.cuda.synchronize(dev)
    status = mla.mla_get_device_status(bufs.workspace, stream)
    if status != 0:
        raise SystemExit("device status after warm-up: %s" % mla.mla_status_string(status))
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    graphs = {k: torch.cuda.CUDAGraph() for k in ("step", "dec", "att")}
    with torch.cuda.stream(side):
        with torch.cuda.graph(graphs["step"], stream=side):
            dec()
            att()
        with torch.cuda.graph(graphs["dec"], stream=side):
            dec()
        with torch.cuda.graph(graphs["att"], stream=side):
            att()
    stream.wait_stream(side)
    torch.cuda.synchronize(dev)
    for g in graphs.values():
        for _ in range(max(3, args.warmup)):
            g.replay()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    ms = {}
    for k in ("step", "dec", "att"):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            graphs[k].replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms[k] = e0.elapsed_time(e1) / args.steps
    clocks = sampler.stop()
    status = mla.mla_get_device_status(bufs.workspace, stream)

    # end to end through the public API with host buffers, as for the
    # decode: the new tokens' queries, the block table and lengths (one
    # packed pinned buffer) H2D and the output D2H every step, on a copy
    # stream overlapping the step before (double-buffered), plain calls
    keys = ("q_nope", "q_rope", "block_table", "seq_lens")
    src = case.tensors()
    offs, off = {}, 0
    for k in keys:
        offs[k] = off
        off += (src[k].numel() * src[k].element_size() + 15) // 16 * 16
    h_in = torch.empty(off, dtype=torch.uint8).pin_memory()
    for k in keys:
        n = src[k].numel() * src[k].element_size()
        h_in[offs[k]:offs[k] + n].copy_(src[k].contiguous().view(-1).view(torch.uint8))
    dev_in = [torch.empty(off, dtype=torch.uint8, device=dev) for _ in range(2)]
    ins = [{k: b[offs[k]:offs[k] + src[k].numel() * src[k].element_size()].view(src[k].dtype).view(src[k].shape)
            for k in keys} for b in dev_in]
    pb = [bufs, mla.PrefillBuffers(d, dev)]
    h_out = [torch.empty(bufs.out.shape, dtype=bufs.out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(src[k].numel() * src[k].element_size() for k in keys)
    d2h = h_out[0].numel() * h_out[0].element_size()
    cs = torch.cuda.Stream(dev)
    ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("in", "done", "out")}
    for j in range(2):
        for n in ev:
            ev[n][j].record(stream)

    def upload(j):
        cs.wait_event(ev["done"][j])
        dev_in[j].copy_(h_in, non_blocking=True)
        ev["in"][j].record(cs)

    def e2e_step(i, n):
        j = i % 2
        stream.wait_event(ev["in"][j])
        stream.wait_event(ev["out"][j])
        x, b = ins[j], pb[j]
        mla.mla_decompress_kv(d, t["cache"], x["block_table"], x["seq_lens"], t["W_UK"], t["W_UV"], b.k_nope, b.v,
                              b.workspace)
        mla.mla_prefill_attend(d, x["q_nope"], x["q_rope"], t["cache"], x["block_table"], x["seq_lens"], b.k_nope,
                               b.v, b.out, b.lse, b.workspace)
        ev["done"][j].record(stream)
        with torch.cuda.stream(cs):
            if i + 1 < n:
                upload(1 - j)
            cs.wait_event(ev["done"][j])
            h_out[j].copy_(b.out, non_blocking=True)
            ev["out"][j].record(cs)

    with torch.cuda.stream(cs):
        upload(0)
    for i in range(3):
        e2e_step(i, 3)
    torch.cuda.synchronize(dev)
    e2e_n = max(args.steps, 20)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    cs.wait_stream(stream)
    with torch.cuda.stream(cs):
        upload(0)
    for i in range(e2e_n):
        e2e_step(i, e2e_n)
    stream.wait_stream(cs)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_n
    for b in pb:
        st2 = mla.mla_get_device_status(b.workspace)
        if st2 != 0:
            raise SystemExit("device status in the end-to-end loop: %s" % mla.mla_status_string(st2))
    peaks, peak_src = load_peaks()
    dec_flops, att_flops, dec_bytes, att_bytes = prefill_accounting(seq, d["Lq"], d["H"], d["G"], d["max_pages"])
    if rank != 0:
        return
    tf = lambda f, m: f / (m * 1e-3) / 1e12
    line = {
        "metric": "MLA prefill (decompress branch) TFLOP/s", "value": tf(dec_flops + att_flops, ms["step"]),
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms["step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) cache and queries, N(0,1/d_g) weights)",
        "config": {"workload": WORKLOAD_TEXT["prefill"], "B": d["B"], "Lq": d["Lq"], "H": d["H"], "G": d["G"],
                   "seq_len": seq, "l2": "K and V (%.0f MB each) exceed L2" % (bufs.k_nope.numel() * 2 / 1e6)},
        "kernels": {
            "decompress": {"ms": ms["dec"], "tflops": tf(dec_flops, ms["dec"]),
                           "tensor_frac": tf(dec_flops, ms["dec"]) / peaks["bf16_tflops"],
                           "gbs": dec_bytes / (ms["dec"] * 1e-3) / 1e9, "flops": dec_flops, "bytes": dec_bytes},
            "attend": {"ms": ms["att"], "tflops": tf(att_flops, ms["att"]),
                       "tensor_frac": tf(att_flops, ms["att"]) / peaks["bf16_tflops"],
                       "gbs": att_bytes / (ms["att"] * 1e-3) / 1e9, "flops": att_flops, "bytes": att_bytes},
            "timing": "events around replays of one-launch graphs",
        },
        "roofline": {"bound": "tensor", "achieved": tf(att_flops, ms["att"]), "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": tf(att_flops, ms["att"]) / peaks["bf16_tflops"], "traffic": None,
                     "kernel": "prefill_attn_kernel", "peak_source": peak_src},
        "e2e": {"value": tf(dec_flops + att_flops, e2e_ms), "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_n,
                "how": "the two calls a step; inputs H2D in one packed copy and the output D2H on a copy stream "
                       "overlapping the step before (double-buffered), all inside the timed region"},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "device_status": mla.mla_status_string(status),
        "cpu_baseline": {"omitted": "the fp64 oracle recomputes a decompressed key and value per (query, key) "
                                    "pair: one (sequence, head) pair of this workload is hours of CPU time; the "
                                    "decode workloads' lines carry the oracle baseline"},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="dsv3", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--fused", action="store_true", help="one fused combine + projection launch")
    ap.add_argument("--kv", default="bf16", choices=["bf16", "fp8"], help="cache format of the decode")
    args = ap.parse_args()
    world, rank, local = dist_env()
    if args.workload == "prefill":
        if args.kv != "bf16":
            raise SystemExit("the decompress branch reads the bf16 cache")
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the decode "
                                  "workloads; the prefill line is a supplementary measurement"}))
            return
        return run_prefill(args, world, rank, local)
    if args.impl == "reference":
        return run_reference(args, world, rank)

    import torch
    import mla_latent_kv_10_gb300 as mla
    from mla_latent_kv_10_gb300 import accounting as acc
    from mla_latent_kv_10_gb300.inputs import workload

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    mla.load_library()

    # every rank decodes a replica of the same batch (weak scaling)
    fp8 = args.kv == "fp8"
    case = workload(args.workload, kv=args.kv)
    d = case.dims
    seq = case.seq_lens.tolist()
    B, Lq, H, G = d["B"], d["Lq"], d["H"], d["G"]
    t = {k: v.to(dev) for k, v in case.tensors().items()}
    cache_bytes = t["cache"].numel() * t["cache"].element_size()
    copies = rotation_copies(cache_bytes)
    caches = [t["cache"]] + [t["cache"].clone() for _ in range(copies - 1)]
    # the weights rotate too, so that no step finds its W_UK and W_UV in L2
    # (a model with many layers reads each layer's weights from HBM)
    w_bytes = sum(t[k].numel() * t[k].element_size() for k in ("W_UK", "W_UV"))
    wcopies = rotation_copies(w_bytes)
    weights = [(t["W_UK"], t["W_UV"])] + [(t["W_UK"].clone(), t["W_UV"].clone()) for _ in range(wcopies - 1)]
    nrot = max(copies, wcopies)  # step graphs: step c uses cache copy c % copies, weights c % wcopies
    bufs = mla.DecodeBuffers(d, dev)
    stream = torch.cuda.current_stream(dev)

    kv_bytes = acc.latent_kv_bytes(seq, kv=args.kv)
    step_bytes = acc.step_bytes(seq, Lq, H, G, kv=args.kv)
    step_flops = acc.step_flops(seq, Lq, H, G)
    dec_bytes = acc.decode_bytes(seq, Lq, H, G, kv=args.kv)
    dec_flops = acc.decode_flops(seq, Lq, H, G, causal=bool(d["causal"]))

    def pre(c):
        mla.mla_absorb_q(d, t["q_nope"], t["q_rope"], weights[c % wcopies][0], bufs.q_cat)

    decode = mla.mla_decode_paged_fp8 if fp8 else mla.mla_decode_paged

    def dec(c):
        decode(d, bufs.q_cat, caches[c], t["block_table"], t["seq_lens"], args.splits, bufs.o_part,
               bufs.lse_part, bufs.workspace)

    def post(c):
        w_uv = weights[c % wcopies][1]
        if not args.fused:
            mla.mla_combine_splits(d, bufs.o_part, bufs.lse_part, bufs.workspace, bufs.o_lat, bufs.lse)
            mla.mla_project_uv(d, bufs.o_lat, w_uv, bufs.out)
        else:
            mla.mla_combine_project(d, bufs.o_part, bufs.lse_part, bufs.workspace, w_uv, bufs.out,
                                    bufs.o_lat, bufs.lse)

    def step(i):
        pre(i)
        dec(i % copies)
        post(i)

    # warm-up through the plain API (sets kernel attributes, checks status)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    status = mla.mla_get_device_status(bufs.workspace, stream)
    if status != 0:
        raise SystemExit("device status after warm-up: %s" % mla.mla_status_string(status))

    # The timed loops replay CUDA graphs of the same calls (no host launch
    # overhead): one graph per step (per cache copy).  The decode kernel's
    # own duration: a graph of DEC_CHAIN decode launches back to back over
    # the rotating cache copies, events around each replay, divided by the
    # launches (each launch waits for the one before it to complete before
    # touching memory; only its on-chip set-up overlaps the tail of the one
    # before, as between the kernels of a step); and, for reference, events
    # around replays of a graph holding a single decode launch (which adds
    # the graph's launch latency).
    DEC_CHAIN = 8
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        g_step = [torch.cuda.CUDAGraph() for _ in range(nrot)]
        g_one = [torch.cuda.CUDAGraph() for _ in range(copies)]
        g_chain = torch.cuda.CUDAGraph()
        for c in range(nrot):
            with torch.cuda.graph(g_step[c], stream=side):
                pre(c)
                dec(c % copies)
                post(c)
        for c in range(copies):
            with torch.cuda.graph(g_one[c], stream=side):
                dec(c)
        with torch.cuda.graph(g_chain, stream=side):
            for j in range(DEC_CHAIN):
                dec(j % copies)
    stream.wait_stream(side)
    torch.cuda.synchronize(dev)

    for i in range(max(nrot, args.warmup)):
        g_step[i % nrot].replay()
        g_one[i % copies].replay()
        g_chain.replay()
    torch.cuda.synchronize(dev)

    def event_pair():
        return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    ev_one = [event_pair() for _ in range(args.steps)]
    ev_chain = [event_pair() for _ in range(args.steps)]
    t_start, t_end = event_pair()
    s_start, s_end = event_pair()
    sampler = ClockSampler(local)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    t_start.record(stream)
    for i in range(args.steps):
        g_step[i % nrot].replay()
    t_end.record(stream)
    for i in range(args.steps):
        ev_chain[i][0].record(stream)
        g_chain.replay()
        ev_chain[i][1].record(stream)
    for i in range(args.steps):
        ev_one[i][0].record(stream)
        g_one[(i + args.steps) % copies].replay()  # continue the rotation of cache copies
        ev_one[i][1].record(stream)
    torch.cuda.synchronize(dev)
    # a sustained run of about a second of steps, so that the clock record
    # spans many samples under load
    step_ms_est = t_start.elapsed_time(t_end) / args.steps
    n_sus = max(args.steps, int(1000.0 / max(step_ms_est, 1e-3)))
    s_start.record(stream)
    for i in range(n_sus):
        g_step[i % nrot].replay()
    s_end.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if pg:
        pg.barrier()
    total_ms = t_start.elapsed_time(t_end)
    dec_ms = sum(a.elapsed_time(b) for a, b in ev_chain) / (args.steps * DEC_CHAIN)
    dec_ms_one = sum(a.elapsed_time(b) for a, b in ev_one) / args.steps
    sus_ms = s_start.elapsed_time(s_end) / n_sus
    total_ms = max_over_ranks(total_ms, pg, dev)
    ms = total_ms / args.steps
    status = mla.mla_get_device_status(bufs.workspace, stream)

    # end to end through the public API with host buffers: every step's
    # inputs H2D from pinned memory, the step by one mla_decode_step call,
    # its result D2H (no graph).  As a serving loop would, the inputs of
    # step i+1 go up on a copy stream while step i computes, and the result
    # of step i comes down there once it is done: two sets of device inputs
    # and outputs, events between the streams.
    e2e_ms, h2d, d2h, e2e_steps = e2e_pipelined(args, mla, torch, dev, stream, case, t, caches, weights, fp8)
    e2e_ms = max_over_ranks(e2e_ms, pg, dev)

    peaks, peak_src = load_peaks()
    hbm = peaks["hbm_gbs"]
    achieved = dec_bytes / (dec_ms * 1e-3) / 1e9
    tflops_dec = dec_flops / (dec_ms * 1e-3) / 1e12
    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": job_rate(world, kv_bytes, ms) / 1e9,
        "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8 e4m3 cache, f16 latent products, fp32 accumulation" if fp8 else "bf16",
        "data": ("synthetic (seeded random E4M3 codes, power-of-two block scales and N(0,1) RoPE key; "
                 "N(0,1) queries, N(0,1/d_g) weights)" if fp8 else
                 "synthetic (seeded N(0,1) cache and queries, N(0,1/d_g) weights)"),
        "config": {"workload": workload_text(args), "step": "fused" if args.fused else "four calls", "B": B,
                   "Lq": Lq, "H": H, "G": G, "kv": args.kv,
                   "seq_len_mean": sum(seq) / len(seq), "page_size": 64,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs larger than L2: %d rotating cache copies (%.0f MB), %d rotating copies of "
                         "W_UK and W_UV (%.0f MB)" % (copies, copies * cache_bytes / 1e6, wcopies,
                                                     wcopies * w_bytes / 1e6)},
        "value_counts": "latent KV cache bytes read per step (%d B, %d B a token) over the step time"
                        % (kv_bytes, acc.row_bytes(args.kv)),
        "step_gbs": job_rate(world, step_bytes, ms) / 1e9,
        "step_bytes": step_bytes,
        "tflops": job_rate(world, step_flops, ms) / 1e12,
        "tokens_per_s": job_rate(world, B * Lq, ms),
        "roofline_frac_step": max(step_bytes / (ms * 1e-3) / 1e9 / hbm,
                                  step_flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"]),
        "decode_kernel": {"ms": dec_ms, "gbs": achieved, "tflops": tflops_dec,
                          "hbm_frac": achieved / hbm,  # on the cache format's bytes
                          "tensor_frac": tflops_dec / peaks["bf16_tflops"],
                          "bytes": dec_bytes, "flops": dec_flops,
                          "ms_single_launch_graph": dec_ms_one,
                          "timing": "mean per launch over %d-launch graphs (events around each replay); "
                                    "ms_single_launch_graph: events around one-launch graphs" % DEC_CHAIN},
        "roofline": roofline_entry(dec_bytes, dec_flops, dec_ms, peaks, decode_traffic(args.workload, args.kv),
                                   peak_src, kernel="mla_decode_paged_fp8" if fp8 else "mla_decode_paged"),
        "e2e": {"value": job_rate(world, kv_bytes, e2e_ms) / 1e9, "unit": "GB/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "how": "one mla_decode_step call a step; the step's inputs H2D from pinned memory in one copy and "
                       "its output D2H, on a copy stream overlapping the step before (double-buffered), all "
                       "inside the timed region"},
        "gpu_launches": mla.launches_per_step(case.dims, fused=args.fused) * args.steps,
        "timing": "one CUDA-graph replay per step: absorb, decode, combine, projection (absorb, decode and "
                  "projection chained by programmatic dependent launch; --fused: one combine + projection "
                  "kernel); gpu_launches counts the kernels of the timed steps",
        "sustained": {"steps": n_sus, "ms_per_step": sus_ms, "seconds": sus_ms * n_sus / 1e3,
                      "note": "step graphs replayed back to back for about a second after the timed "
                              "region, inside the clock record"},
        "clocks": clocks,
        "device_status": mla.mla_status_string(status),
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(case, kv=args.kv)
    print(json.dumps(line))
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
