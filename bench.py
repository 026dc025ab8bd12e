"""Benchmark: fp8 paged MQA logits (sparse-attention indexer), KV positions
scored per second on GB300, with the roofline fraction of the kernel.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|mtp2|mtp4|skewed|indexer_g1|...|indexer_g8]

One step = one call of the hot path (per-CTA schedule + TMA/tcgen05 logits
kernel) over the whole batch, inputs resident in HBM.  By default the timed
steps cycle through three resident copies of the workload (together several
times larger than L2, so no step finds its inputs in L2) and are launched back
to back between one pair of CUDA events on the launching stream; ``--l2
flush`` instead writes 256 MiB before every step and times each launch alone.  Under torchrun every rank runs its own batch of the same
shape (different seed): weak scaling, no data-path collective; the time is the
max over ranks.  ``--impl reference`` times the CPU oracle (fp64, all host
cores) on bounded samples of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
METRIC = "KV positions scored/s and HBM GB/s (fraction of roofline), fp8 paged MQA logits"
UNIT = "positions/s"
FLUSH_BYTES = 256 << 20

WORKLOAD_TEXT = {
    "decode": "decode: batch 64, next_n 1, 64 heads, head_dim 128, 64-token kv_fused blocks "
              "(64x128 e4m3 + 64 fp32 scales), seq_lens U[1024,32768], pages shuffled in a "
              "shared pool, q,k ~N(0,1)->e4m3, s_p ~U[0.5,2], w ~N(0,1)/8, fp32 out",
    "mtp2": "MTP verify: batch 32, next_n 2, 64 heads, seq_lens U[8192,65536], decode layout",
    "mtp4": "MTP verify: batch 32, next_n 4, 64 heads, seq_lens U[8192,65536], decode layout",
    "skewed": "skewed: 16 requests, next_n 1, 64 heads, one 131072, three empty, twelve "
              "U[512,4096]",
    "topk_decode": "indexer top-k selection: 64 logits rows of 32768 (lengths U[1024,32768]), "
                   "k 2048, indices of the largest meaningful logits",
    "mxfp4_decode": "MXFP4 paged MQA logits, decode shape: batch 64, next_n 1, 64 heads, head_dim "
                    "128, 64-token blocks (64x64 E2M1 code bytes + 64x4 E8M0 scales), seq_lens "
                    "U[1024,32768], pages shuffled in a shared pool, codes uniform, scales "
                    "2^-4..2^4, w ~N(0,1)/8, bf16 out",
    "nvfp4_g8": "single-head NVFP4 indexer_scores: 256 groups of 8 rows, E2M1 codes with E4M3 "
                "scales per 16 values, pages of 4096 code bytes then 512 scale bytes, "
                "context_lengths U[0,65536] (8 zeros), fp32 scores [2048, 65536]",
}


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def make_problem(workload: str, rank: int):
    from sparse_attention_indexer_logits_gb300 import workloads as W
    off = 1000 * rank
    if workload == "decode":
        return W.decode(seed=1 + off, poison=False)
    if workload in ("mtp2", "mtp4"):
        n = int(workload[-1])
        return W.mtp(next_n=n, seed=(2 if n == 4 else 3) + off, poison=False)
    if workload == "skewed":
        return W.skewed(seed=4 + off)
    if workload == "mxfp4_decode":
        return W.mxfp4_decode(seed=7 + off, poison=False)
    if workload == "topk_decode":
        return W.topk_decode(seed=13 + off)
    if workload.startswith("nvfp4_g"):
        return W.indexer_nvfp4(group_size=int(workload[len("nvfp4_g"):]), seed=6 + off,
                               poison=False)
    if workload.startswith("indexer_g"):
        return W.indexer(group_size=int(workload[len("indexer_g"):]), seed=5 + off, poison=False)
    raise SystemExit(f"unknown workload {workload}")


# Sources each kernel is built from (the shared headers included): a recorded
# traffic figure stays valid while these are unchanged.
KERNEL_SOURCES = {
    "fp8_logits_kernel": ("fp8_logits.cuh", "fp8_logits.cu", "fp8_logits_h8.cu", "fp8_logits_h16.cu",
                          "fp8_logits_h32.cu", "fp8_logits_h64.cu", "window.cuh"),
    "bf16_scores_kernel": ("bf16_scores.cu",),
    "nvfp4_scores_kernel": ("nvfp4_scores.cu",),
    "topk_kernel": ("topk.cu",),
    "mxfp4_logits_kernel": ("mxfp4_logits.cu", "window.cuh"),
}
SHARED_SOURCES = ("common.cuh", "ptx.cuh", "kernels.h")


def kernel_fingerprint(kernel: str) -> str:
    h = hashlib.sha256()
    d = os.path.join(ROOT, "sparse_attention_indexer_logits_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[kernel] + SHARED_SOURCES):
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def recorded_traffic(kernel: str, workload: str):
    """dram bytes per launch from a committed ncu capture of the current kernel
    source, or None when the kernel changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(kernel, {}).get(workload)
    if not e or e.get("fingerprint") != kernel_fingerprint(kernel):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        with open(self.file.name) as f:
            lines = [l.strip() for l in f if l.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in lines:
            parts = [x.strip() for x in l.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def oracle_baseline(p, seconds_budget: float, workload: str):
    """The CPU oracle (fp64, all host cores) on a bounded sample of the same
    workload: whole requests in order until about `seconds_budget` of wall
    time has been spent.  Returns (positions/s, cores, sample description)."""
    import oracle
    from tests.helpers import sub_problem
    cores = os.cpu_count() or 1
    if workload.startswith("indexer"):
        raise SystemExit("oracle baseline is only wired for the fp8 workloads")
    done_pos, spent, used = 0, 0.0, []
    order = list(range(p.batch))
    while spent < seconds_budget and order:
        take = order[:cores]
        order = order[cores:]
        sp = sub_problem(p, take)
        if sp.positions == 0:
            continue
        t0 = time.perf_counter()
        oracle.fp8_paged_mqa_logits(sp.q, sp.kv_fused, sp.weights, sp.seq_lens, sp.block_table,
                                    next_n=sp.next_n, max_context=int(sp.seq_lens.max()),
                                    with_mag=False, nthreads=cores)
        spent += time.perf_counter() - t0
        done_pos += sp.positions
        used += take
    return done_pos / spent, cores, f"{len(used)} of {p.batch} requests ({done_pos} positions), " \
                                   f"{spent:.1f} s wall on {cores} threads"


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is a bounded sample."""
    import oracle
    from tests.helpers import sub_problem
    if rank != 0:
        return
    p = make_problem(args.workload, 0)
    cores = os.cpu_count() or 1
    total_budget = 90.0
    per_step = max(0.02, total_budget / max(1, args.steps + args.warmup))
    # calibrate: positions per second of the oracle on this host
    cal = sub_problem(p, list(range(min(cores, p.batch))))
    cal_sl = np.minimum(cal.seq_lens, 2048).astype(np.int32)
    t0 = time.perf_counter()
    oracle.fp8_paged_mqa_logits(cal.q, cal.kv_fused, cal.weights, cal_sl, cal.block_table,
                                next_n=cal.next_n, max_context=2048, with_mag=False,
                                nthreads=cores)
    rate = int(cal_sl.sum()) / (time.perf_counter() - t0)
    per_req = max(64, int(rate * per_step / cores))
    times, positions = [], []
    start = 0
    for step in range(args.warmup + args.steps):
        idx = [(start + i) % p.batch for i in range(cores)]
        start = (start + cores) % p.batch
        sp = sub_problem(p, idx)
        sl = np.minimum(sp.seq_lens, per_req).astype(np.int32)
        t0 = time.perf_counter()
        oracle.fp8_paged_mqa_logits(sp.q, sp.kv_fused, sp.weights, sl, sp.block_table,
                                    next_n=sp.next_n, max_context=max(1, int(sl.max())),
                                    with_mag=False, nthreads=cores)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
            positions.append(int(sl.sum()))
    value = sum(positions) / sum(times)
    sample = (f"per step {cores} requests of the workload, each clipped to its first "
              f"{per_req} positions (fp64 oracle, {cores} threads)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(args.workload, p, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def reduce_over_ranks(seconds: float, positions: int, dist, device):
    """Whole-job timing across ranks: the slowest rank's time and the sum of
    the positions every rank scored (identity without a process group)."""
    if dist is None:
        return seconds, positions
    t = torch.tensor([seconds, float(positions)], dtype=torch.float64, device=device)
    tmax = t[:1].clone()
    dist.all_reduce(tmax, op=dist.ReduceOp.MAX)
    psum = t[1:].clone()
    dist.all_reduce(psum, op=dist.ReduceOp.SUM)
    return float(tmax.item()), int(psum.item())


def config_of(workload, p, world, l2="rotate", copies=3, launch="graph"):
    l2_text = (f"flushed before every timed step ({FLUSH_BYTES >> 20} MiB write)" if l2 == "flush"
               else f"inputs larger than L2: {copies} resident copies of the workload used in "
                    f"rotation, back-to-back launches")
    launch_text = ("each step launched alone between its own events" if l2 == "flush" else
                   "the K calls captured into one CUDA graph before the timed region, which "
                   "replays it" if launch == "graph" else
                   "the K calls issued from Python inside the timed region")
    cfg = {"workload": WORKLOAD_TEXT.get(workload, workload),
           "l2": l2_text, "launch": launch_text,
           "parallelism": "replicas" if world == 1 else f"dp{world} (independent batches)"}
    if hasattr(p, "k"):
        cfg.update({"rows": int(p.logits.shape[0]), "k": p.k, "max_context": p.max_context,
                    "positions_per_step": p.positions})
    elif hasattr(p, "next_n"):
        cfg.update({"batch": p.batch, "next_n": p.next_n, "num_heads": p.num_heads,
                    "head_dim": 128, "positions_per_step": p.positions,
                    "max_context": p.max_context})
    else:
        cfg.update({"groups": p.groups, "group_size": p.group_size,
                    "positions_per_step": p.positions, "max_context": p.max_context})
    return cfg


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--l2", default="rotate", choices=["rotate", "flush"],
                    help="rotate: cycle through --copies resident input sets (together larger "
                         "than L2) with back-to-back launches; flush: write 256 MiB between steps")
    ap.add_argument("--copies", type=int, default=3)
    ap.add_argument("--launch", default="graph", choices=["graph", "eager"],
                    help="graph: the K timed calls are captured once into a CUDA graph before "
                         "the timed region, which replays it (device throughput, no host cost "
                         "per call); eager: the K calls are issued from Python inside the "
                         "timed region")
    ap.add_argument("--out-dtype", default="float32", choices=["float32", "bfloat16"],
                    help="fp8 workloads: element type of the logits (the output_dtype option)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = _env_int("RANK", 0)
    world = _env_int("WORLD_SIZE", 1)
    local_rank = _env_int("LOCAL_RANK", 0)
    dist = None
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference":
            dist.init_process_group("gloo")
        else:
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    if args.impl == "reference":
        run_reference(args, rank, world)
        if dist is not None:
            dist.destroy_process_group()
        return

    sys.path.insert(0, ROOT)
    import __graft_entry__
    __graft_entry__.build()
    import sparse_attention_indexer_logits_gb300 as pml

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    p = make_problem(args.workload, rank)
    from sparse_attention_indexer_logits_gb300 import workloads as W
    is_topk = isinstance(p, W.TopkProblem)
    is_mx = isinstance(p, W.Mxfp4Problem)
    is_fp8 = hasattr(p, "next_n") and not is_mx
    is_nvfp4 = isinstance(p, W.Nvfp4Problem)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    copies = args.copies if args.l2 == "rotate" else 1
    out_dtype = torch.bfloat16 if (is_fp8 and args.out_dtype == "bfloat16") else torch.float32
    if is_topk:
        def device_set():
            return dict(x=t(p.logits), sl=t(p.seq_lens),
                        out=torch.zeros((p.logits.shape[0], p.k), dtype=torch.int32, device=dev))
        sets = [device_set() for _ in range(copies)]

        def step(d, stream=None):
            pml.pml_topk_logits(d["x"], d["sl"], p.rows_per_request, p.max_context, p.k,
                                indices=d["out"], stream=stream)
        kernel = "topk_kernel"
        bound_name = "hbm"
    elif is_mx:
        def device_set():
            return dict(q=t(p.q), qsf=t(p.q_sf), kv=t(p.kv), w=t(p.weights), sl=t(p.seq_lens),
                        bt=t(p.block_table),
                        out=torch.zeros((p.batch * p.next_n, p.max_context), dtype=torch.bfloat16,
                                        device=dev))
        sets = [device_set() for _ in range(copies)]

        def step(d, stream=None):
            pml.pml_fp4_paged_mqa_logits(d["q"], d["qsf"], d["kv"], d["w"], d["sl"], d["bt"],
                                         d["out"], p.max_context, p.next_n, stream=stream)
        kernel = "mxfp4_logits_kernel"
        bound_name = "hbm"
    elif is_fp8:
        def device_set():
            return dict(q=t(p.q), kv=t(p.kv_fused), w=t(p.weights), sl=t(p.seq_lens),
                        bt=t(p.block_table),
                        out=torch.zeros((p.batch * p.next_n, p.max_context), dtype=out_dtype,
                                        device=dev))
        sets = [device_set() for _ in range(copies)]

        def step(d, stream=None):
            pml.pml_fp8_paged_mqa_logits_ex(d["q"], d["kv"], d["w"], d["sl"], d["bt"], d["out"],
                                            p.max_context, p.next_n, stream=stream)
        kernel = "fp8_logits_kernel"
        bound_name = "hbm"
    elif is_nvfp4:
        def device_set():
            kb = t(p.key_buf)
            return dict(q=t(p.query), qs=t(p.query_scales), kb=kb,
                        sb=kb if p.fused else t(p.scale_buf), bt=t(p.block_table),
                        cl=t(p.context_lengths), rq=t(p.requests),
                        out=torch.zeros((p.rows, p.max_context), dtype=torch.float32, device=dev))
        sets = [device_set() for _ in range(copies)]

        def step(d, stream=None):
            pml.pml_indexer_scores_nvfp4(d["q"], d["qs"], d["kb"][p.key_off:], p.page_stride_bytes,
                                         d["sb"][p.scale_off:], p.scale_page_stride_bytes,
                                         p.num_pages, d["bt"], d["cl"], d["rq"], d["out"],
                                         p.max_context, stream=stream)
        kernel = "nvfp4_scores_kernel"
        bound_name = "hbm"
    else:
        def device_set():
            return dict(q=t(p.query.view(np.int16)).view(torch.bfloat16), kc=t(p.key_cache),
                        bt=t(p.block_table), cl=t(p.context_lengths), rq=t(p.requests),
                        out=torch.zeros((p.rows, p.max_context), dtype=torch.float32, device=dev))
        sets = [device_set() for _ in range(copies)]

        def step(d, stream=None):
            pml.pml_indexer_scores_bf16(d["q"], d["kc"], p.page_stride_bytes, p.num_pages, d["bt"],
                                        d["cl"], d["rq"], d["out"], p.max_context, stream=stream)
        kernel = "bf16_scores_kernel"
        bound_name = "hbm"

    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev) \
        if args.l2 == "flush" else None
    stream = torch.cuda.current_stream()
    pml.pml_device_status(clear=True)
    for i in range(args.warmup):
        if flush is not None:
            flush.zero_()
        step(sets[i % copies])
    torch.cuda.synchronize()

    graph = None
    if flush is not None:
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    else:
        starts = [torch.cuda.Event(enable_timing=True)]
        ends = [torch.cuda.Event(enable_timing=True)]
        if args.launch == "graph":
            # the K calls, captured once: the same kernels and arguments as the
            # eager loop, without the per-call host work in the timed region
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for i in range(args.steps):
                    step(sets[i % copies])
            graph.replay()
            torch.cuda.synchronize()
            stream = torch.cuda.current_stream()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank if world > 1 else _visible_index()) as clocks:
        if flush is not None:
            for i in range(args.steps):
                flush.zero_()
                starts[i].record(stream)
                step(sets[0])
                ends[i].record(stream)
        elif graph is not None:
            # a ~1 ms device spin ahead of the start event keeps the GPU busy
            # while the host submits the graph, so the timed region holds the
            # K calls and not the graph's launch latency
            torch.cuda._sleep(2_000_000)
            starts[0].record(stream)
            graph.replay()
            ends[0].record(stream)
        else:
            starts[0].record(stream)
            for i in range(args.steps):
                step(sets[i % copies])
            ends[0].record(stream)
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    durs_ms = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
    total_s = sum(durs_ms) / 1e3
    status = pml.pml_device_status(clear=True)
    if status:
        raise SystemExit(f"device status word set during the bench: {status:#x}")

    total_s, positions_all = reduce_over_ranks(total_s, p.positions, dist, dev)
    value = positions_all * args.steps / total_s
    avg_launch_s = total_s / args.steps

    # ---- end to end through the public API with host buffers (pinned)
    e2e = None
    if is_topk:
        d0 = sets[0]
        inputs = ((d0["x"], torch.from_numpy(p.logits).pin_memory()),
                  (d0["sl"], torch.from_numpy(p.seq_lens).pin_memory()))
        hout = torch.empty(d0["out"].shape, dtype=torch.int32).pin_memory()
        h2d = sum(h.numel() * h.element_size() for _, h in inputs)
        d2h = hout.numel() * hout.element_size()

        def e2e_step():
            for d, h in inputs:
                d.copy_(h, non_blocking=True)
            step(d0)
            hout.copy_(d0["out"], non_blocking=True)
    elif is_mx:
        d0 = sets[0]
        bufs = [(d0["q"], p.q), (d0["qsf"], p.q_sf), (d0["kv"], p.kv), (d0["w"], p.weights),
                (d0["sl"], p.seq_lens), (d0["bt"], p.block_table)]
        inputs = tuple((d, torch.from_numpy(np.ascontiguousarray(a)).pin_memory()) for d, a in bufs)
        hout = torch.empty(d0["out"].shape, dtype=torch.bfloat16).pin_memory()
        h2d = sum(h.numel() * h.element_size() for _, h in inputs)
        d2h = hout.numel() * hout.element_size()

        def e2e_step():
            for d, h in inputs:
                d.copy_(h, non_blocking=True)
            step(d0)
            hout.copy_(d0["out"], non_blocking=True)
    elif is_fp8:
        hq, hkv, hw = (torch.from_numpy(a).pin_memory() for a in (p.q, p.kv_fused, p.weights))
        hsl, hbt = torch.from_numpy(p.seq_lens).pin_memory(), torch.from_numpy(p.block_table).pin_memory()
        d0 = sets[0]
        hout = torch.empty(d0["out"].shape, dtype=out_dtype).pin_memory()
        inputs = ((d0["q"], hq), (d0["kv"], hkv), (d0["w"], hw), (d0["sl"], hsl), (d0["bt"], hbt))
        h2d = sum(h.numel() * h.element_size() for _, h in inputs)
        d2h = hout.numel() * hout.element_size()

        def e2e_step():
            for d, h in inputs:
                d.copy_(h, non_blocking=True)
            step(d0)
            hout.copy_(d0["out"], non_blocking=True)
    elif is_nvfp4:
        d0 = sets[0]
        bufs = [(d0["q"], p.query), (d0["qs"], p.query_scales), (d0["kb"], p.key_buf),
                (d0["bt"], p.block_table), (d0["cl"], p.context_lengths), (d0["rq"], p.requests)]
        if not p.fused:
            bufs.append((d0["sb"], p.scale_buf))
        inputs = tuple((d, torch.from_numpy(np.ascontiguousarray(a)).pin_memory()) for d, a in bufs)
        hout = torch.empty(d0["out"].shape, dtype=torch.float32).pin_memory()
        h2d = sum(h.numel() * h.element_size() for _, h in inputs)
        d2h = hout.numel() * hout.element_size()

        def e2e_step():
            for d, h in inputs:
                d.copy_(h, non_blocking=True)
            step(d0)
            hout.copy_(d0["out"], non_blocking=True)
    else:
        hq = torch.from_numpy(p.query.view(np.int16)).pin_memory()
        hkc = torch.from_numpy(p.key_cache).pin_memory()
        hbt, hcl, hrq = (torch.from_numpy(a).pin_memory() for a in (p.block_table, p.context_lengths, p.requests))
        d0 = sets[0]
        hout = torch.empty(d0["out"].shape, dtype=torch.float32).pin_memory()
        inputs = ((d0["q"].view(torch.int16), hq), (d0["kc"], hkc), (d0["bt"], hbt), (d0["cl"], hcl),
                  (d0["rq"], hrq))
        h2d = sum(h.numel() * h.element_size() for _, h in inputs)
        d2h = hout.numel() * hout.element_size()

        def e2e_step():
            for d, h in inputs:
                d.copy_(h, non_blocking=True)
            step(d0)
            hout.copy_(d0["out"], non_blocking=True)
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    es.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    ee.record(stream)
    torch.cuda.synchronize()
    e2e_s, _ = reduce_over_ranks(es.elapsed_time(ee) / 1e3, 0, dist, dev)
    e2e = {"value": positions_all * args.e2e_steps / e2e_s, "unit": UNIT,
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    hbm_peak, bf16_peak, peak_kind = measured_peaks()
    alg_bytes = (p.algorithmic_bytes(out_dtype.itemsize) if (is_fp8 and not is_topk)
                 else p.algorithmic_bytes())   # MXFP4: bf16 logits
    achieved_gbs = alg_bytes / avg_launch_s / 1e9
    roof = {"bound": bound_name, "achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s",
            "frac": achieved_gbs / hbm_peak, "traffic": recorded_traffic(kernel, args.workload),
            "peak_source": f"{peak_kind} hbm_gbs (burst copy); kernel time = timed region / steps",
            "algorithmic_bytes_per_launch": alg_bytes,
            "algorithmic_flops_per_launch": p.algorithmic_flops(),
            "kernel": kernel, "avg_launch_us": avg_launch_s * 1e6}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": (("e4m3 x e4m3 -> f32" + (" -> bf16 out" if out_dtype == torch.bfloat16 else ""))
                      if is_fp8 else
                      ("mxfp4 (e2m1 x e8m0/32) -> f16 or bf16 x same -> f32 -> bf16 out" if is_mx else
                       "nvfp4 (e2m1 x e2m1, e4m3 scale per 16, block-scaled MMA) -> f32" if is_nvfp4
                                      else ("f32 logits -> int32 indices" if is_topk
                                            else "bf16 x bf16 -> f32"))),
            "data": "synthetic (seeded generators; no public dataset on the pages)",
            "config": dict(config_of(args.workload, p, world, args.l2, copies, args.launch),
                           **({"output_dtype": args.out_dtype} if is_fp8 else {})),
            "clocks": clocks.summary(), "gpu_launches": args.steps,
            "e2e": e2e, "roofline": roof,
            "logits_per_s": positions_all * getattr(p, "next_n", 1) * args.steps / total_s,
        }
        if not args.no_cpu_baseline and world >= 1 and is_fp8:
            v, cores, sample = oracle_baseline(p, 15.0, args.workload)
            line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                    "sample": sample}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def _visible_index() -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    if vis and vis.split(",")[0].strip().isdigit():
        return int(vis.split(",")[0])
    return torch.cuda.current_device()


if __name__ == "__main__":
    main()
