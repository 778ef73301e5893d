"""Benchmark: KDA training forward + backward throughput (token*heads/s) on GB300.

One step = kda_fwd + kda_bwd (every kernel of the path) over the packed
8 x 1024-token, 96-head workload (K = V = 128), synthetic seeded inputs
(kda_inputs.py), already resident in HBM. Each input tensor is larger than the
129 MB L2, so no flush is needed between steps. Timing: CUDA events on the
launching stream, W untimed warm-up steps, then exactly K timed steps between
a barrier + synchronize on both sides; the max over ranks is reported.

Also reported on the same JSON line:
  roofline      the dominant kernel's achieved algorithmic HBM bytes/s against
                the measured copy bandwidth (MEASURED_PEAKS.json);
  e2e           the same metric with inputs in pinned host memory, copied in and
                all results copied out inside the timed region;
  cpu_baseline  the FP64 oracle timed on this host on a bounded sample;
  clocks        nvidia-smi SM clocks and throttle reasons sampled while timing.

``--impl reference`` times the oracle itself (the only reference implementation
of this method available here) as the reference arm.
Multi-GPU (torchrun, N > 1): every rank runs its own copy of the workload on its
own GPU with no collective on the data path (weak scaling, replicas).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "packed_8x1024_h96"
METRIC = "KDA fwd+bwd token·heads/s (1 GB300) and fraction of roofline"
UNIT = "token·heads/s"
DIM = 128
# operand type of the tensor-core products (FP32 accumulation; the state and its adjoint are FP32)
MMA_KIND = "tf32"


def algorithmic_bytes(total_tokens, hqk, hv, units):
    """Compulsory HBM bytes of one forward and one backward (each tensor read or
    written once): per token 1536 Hqk + 2054 Hv, per unit 4 states of 64 KiB."""
    fwd_tok = 512 * hqk + 512 * hv + 2 * hv + 256 * hv
    bwd_tok = (512 * hqk + 512 * hv + 2 * hv + 256 * hv) + 512 * hqk + 512 * hv + 2 * hv
    state = DIM * DIM * 4
    return {"fwd": total_tokens * fwd_tok + units * 2 * state,
            "bwd": total_tokens * bwd_tok + units * 2 * state}


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": float(d["hbm_gbs"]), "src": "measured"}
    return {"hbm_gbs": 6800.0, "src": "fallback"}


def kernel_source_sha(name):
    path = os.path.join(ROOT, "linear_attention_gated_gb300", "csrc", name)
    if not os.path.exists(path):
        return None
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def ncu_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, or None if absent, taken
    on a different version of the kernel's source, or scaled to another workload."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path)).get(kernel)
    if not d or d.get("source_sha") != kernel_source_sha(d.get("source", "")) or d.get("workload") != workload:
        return None
    return d.get("bytes_per_launch")


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value, world, device=None):
    """Largest value over all ranks (the slowest rank sets the job's time)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank, world, max_seconds):
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return units_per_rank * world / max_seconds


def oracle_sample_run(x, heads, r):
    """Time the FP64 oracle's forward + backward on the given query/key heads."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    from kda_test_utils import FWD_KEYS, slice_heads
    y = slice_heads(x, heads, r)
    f = {k: (v.double().numpy() if hasattr(v, "double") else v) for k, v in y.items()}
    t0 = time.perf_counter()
    oracle.forward(*[f[k] for k in FWD_KEYS], cu_seqlens=f.get("cu_seqlens"))
    oracle.backward(*[f[k] for k in FWD_KEYS], f["do"], f["dfinal_state"], cu_seqlens=f.get("cu_seqlens"))
    return time.perf_counter() - t0, oracle.num_threads()


def cpu_baseline(x, w, target_s=12.0):
    """Oracle on a bounded sample: the first query/key heads (all sequences), grown
    until one timed run takes at least about 10 s (or covers every head)."""
    r = w.hv // w.hqk
    token_heads_per_qk = x["q"].shape[0] * x["q"].shape[1] * r
    nh = 1
    dt, cores = oracle_sample_run(x, list(range(nh)), r)
    while dt < 10.0 and nh < w.hqk:
        nh = min(w.hqk, max(nh + 1, int(nh * target_s / max(dt, 1e-3))))
        dt, cores = oracle_sample_run(x, list(range(nh)), r)
    th = nh * token_heads_per_qk
    return {"value": th / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{w.name}: query/key heads 0..{nh - 1} of {w.hqk} (all sequences), "
                      f"{th} token·heads, FP64 forward + backward, {dt:.1f} s"}


def run_reference(args, world, rank):
    import kda_inputs as ki
    if rank != 0:
        return
    w = ki.WORKLOADS[args.workload]
    x = ki.workload_inputs(args.workload)
    r = w.hv // w.hqk
    heads = list(range(min(2, w.hqk)))
    th = len(heads) * x["q"].shape[0] * x["q"].shape[1] * r
    for _ in range(args.warmup):
        oracle_sample_run(x, heads, r)
    times = []
    cores = 0
    for _ in range(args.steps):
        dt, cores = oracle_sample_run(x, heads, r)
        times.append(dt)
    total = sum(times)
    value = th * args.steps / total
    sample = (f"{w.name}: query/key heads {heads} of {w.hqk} (all sequences) per step, "
              f"{th} token·heads, FP64 forward + backward")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "sample": sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="named workload of kda_inputs.WORKLOADS (default: the packed 8 x 1024, 96-head one)")
    ap.add_argument("--decode", type=int, default=0, metavar="N",
                    help="instead of the training step, time decode steps (T = 1) of N sequences x 96 heads")
    ap.add_argument("--decode-state", default="bf16", choices=["bf16", "fp32"])
    ap.add_argument("--prefill", action="store_true",
                    help="instead of the training step, time inference prefill of the workload from a state pool")
    ap.add_argument("--prefill-checkpoint", type=int, default=0, metavar="N",
                    help="prefill: BF16 state checkpoints every N tokens (a multiple of 16; 0 = none)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.decode:
        bench_decode(args)
        return
    if args.prefill:
        bench_prefill(args)
        return

    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import torch

    import kda_inputs as ki
    from linear_attention_gated_gb300 import kda_bwd, kda_fwd, load_library
    from linear_attention_gated_gb300 import build as cuda_build

    cuda_build.build()
    load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = ki.WORKLOADS[args.workload]
    x = ki.workload_inputs(args.workload)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    cu_cpu = x["cu_seqlens"]  # None for the fixed [B, T] layout
    B, T = x["q"].shape[:2]
    N = cu_cpu.numel() - 1 if cu_cpu is not None else B
    Ttot = B * T
    units = N * w.hv
    token_heads = Ttot * w.hv
    stream = torch.cuda.current_stream(dev)

    o = torch.empty_like(d["v"])
    hT = torch.empty_like(d["h0"])
    grads = (torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"]),
             torch.empty_like(d["g"]), torch.empty_like(d["beta"]), torch.empty_like(d["A_log"]),
             torch.empty_like(d["dt_bias"]), torch.empty_like(d["h0"]))
    ctx = None

    def step(evs=None):
        nonlocal ctx
        if evs:
            evs[0].record(stream)
        _, _, ctx = kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
                            d["h0"], cu_seqlens=d["cu_seqlens"], out=o, final_state_out=hT,
                            context_out=ctx, cu_seqlens_cpu=cu_cpu)
        if evs:
            evs[1].record(stream)
        kda_bwd(ctx, d["do"], d["dfinal_state"], out=grads)
        if evs:
            evs[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    barrier(world)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0])
                           if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local)
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize(dev)
    barrier(world)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop()
    elapsed = t_start.elapsed_time(t_end) / 1e3
    elapsed = max_over_ranks(elapsed, world, dev)
    fwd_ms = [e[0].elapsed_time(e[1]) for e in evs]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in evs]
    value = job_value(token_heads * args.steps, world, elapsed)

    ab = algorithmic_bytes(Ttot, w.hqk, w.hv, units)
    peaks = read_peaks()
    fwd_avg, bwd_avg = statistics.mean(fwd_ms), statistics.mean(bwd_ms)
    dom, dom_ms = ("kda_bwd_kernel", bwd_avg) if bwd_avg >= fwd_avg else ("kda_fwd_kernel", fwd_avg)
    dom_bytes = ab["bwd"] if dom == "kda_bwd_kernel" else ab["fwd"]
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": ncu_traffic(dom, args.workload),
                "kernel": dom, "peak_src": peaks["src"],
                "algorithmic_bytes_per_launch": dom_bytes, "avg_launch_ms": dom_ms,
                "step_frac": (ab["fwd"] + ab["bwd"]) / (elapsed / args.steps) / 1e9 / peaks["hbm_gbs"],
                "fwd_ms": fwd_avg, "bwd_ms": bwd_avg}
    launches_per_step = 2 + (1 if w.hv != w.hqk else 0) + 1  # fwd, bwd, param reduce, GQA reduce

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(x, d, dev, stream, kda_fwd, kda_bwd, token_heads, world)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * elapsed / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp32", "data": "synthetic",
            "config": {"workload": args.workload, "sequences": N, "tokens": Ttot, "Hqk": w.hqk, "Hv": w.hv,
                       "head_dim": DIM, "token_heads_per_gpu": token_heads, "io_dtype": "bf16",
                       "state_dtype": "fp32", "mma": MMA_KIND, "l2": f"a forward moves {ab['fwd'] / 1e6:.0f} MB and a backward "
                       f"{ab['bwd'] / 1e6:.0f} MB, each > 129 MB of L2 (largest token tensor "
                       f"{d['v'].numel() * 2 / 1e6:.0f} MB), no flush",
                       "parallelism": f"replicas x{world}"},
            "roofline": roofline, "gpu_launches": launches_per_step * args.steps, "clocks": clocks,
            "e2e": e2e}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(x, w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def bench_decode(args):
    """Decode steps of N sequences x 96 value heads (one token each) against one
    state pool, updated in place; prints one JSON line with HBM roofline."""
    import torch

    from linear_attention_gated_gb300 import build as cuda_build
    from linear_attention_gated_gb300 import kda_decode, load_library

    cuda_build.build()
    load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    N, H = args.decode, 96
    gen = torch.Generator("cpu").manual_seed(7)
    def bf(*shape):
        return torch.randn(shape, generator=gen).to(torch.bfloat16).to(dev)
    q, k, v, g, beta = bf(N, 1, H, DIM), bf(N, 1, H, DIM), bf(N, 1, H, DIM), bf(N, 1, H, DIM), bf(N, 1, H)
    A_log = (torch.rand((H,), generator=gen) * math.log(16.0)).to(dev)
    dt_bias = (0.1 * torch.randn((H, DIM), generator=gen)).to(dev)
    sdt = torch.bfloat16 if args.decode_state == "bf16" else torch.float32
    state = (0.05 * torch.randn((N, H, DIM, DIM), generator=gen)).to(sdt).to(dev)
    o = torch.empty_like(v)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        kda_decode(q, k, v, g, beta, A_log, dt_bias, state, out=o, use_gate_in_kernel=True, beta_is_logit=True)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        kda_decode(q, k, v, g, beta, A_log, dt_bias, state, out=o, use_gate_in_kernel=True, beta_is_logit=True)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    sec = t0.elapsed_time(t1) / 1e3 / args.steps
    esz = 2 if sdt == torch.bfloat16 else 4
    # per unit: the state read and written once, q, k (its query/key head), v, g read, o written, beta
    bytes_step = N * H * (2 * esz * DIM * DIM + 4 * 2 * DIM + 2 * DIM + 2)
    peaks = read_peaks()
    achieved = bytes_step / sec / 1e9
    line = {"metric": "KDA decode token\u00b7heads/s (1 GB300)", "value": N * H / sec, "unit": UNIT,
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec,
            "higher_is_better": True, "dtype": "fp32", "data": "synthetic",
            "config": {"workload": f"decode_{N}x{H}", "sequences": N, "Hqk": H, "Hv": H, "head_dim": DIM,
                       "state_dtype": args.decode_state,
                       "l2": f"state pool {N * H * DIM * DIM * esz / 1e6:.0f} MB > 129 MB, no flush"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "traffic": None, "kernel": "kda_decode_kernel",
                         "peak_src": peaks["src"], "algorithmic_bytes_per_launch": bytes_step},
            "gpu_launches": args.steps, "clocks": clocks}
    print(json.dumps(line), flush=True)


def bench_prefill(args):
    """Inference prefill of the named workload from a state pool (slot n per
    sequence, FP32 or BF16 per --decode-state, updated in place), optionally
    with BF16 state checkpoints; prints one JSON line with HBM roofline."""
    import itertools

    import torch

    import kda_inputs as ki
    from linear_attention_gated_gb300 import build as cuda_build
    from linear_attention_gated_gb300 import kda_prefill, load_library

    cuda_build.build()
    load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = ki.WORKLOADS[args.workload]
    x = ki.workload_inputs(args.workload)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    cu_cpu = x["cu_seqlens"]
    B, T = x["q"].shape[:2]
    N = cu_cpu.numel() - 1 if cu_cpu is not None else B
    lens = (cu_cpu[1:] - cu_cpu[:-1]).tolist() if cu_cpu is not None else [T] * B
    Ttot = sum(lens)
    sdt = torch.bfloat16 if args.decode_state == "bf16" else torch.float32
    state = d["h0"].to(sdt).contiguous()
    ck = ck_starts = ck_cpu = None
    n_ck = 0
    if args.prefill_checkpoint:
        per = [(L + args.prefill_checkpoint - 1) // args.prefill_checkpoint for L in lens]
        ck_cpu = torch.tensor([0] + list(itertools.accumulate(per)), dtype=torch.int64)
        n_ck = int(ck_cpu[-1])
        ck = torch.empty((n_ck, w.hv, DIM, DIM), dtype=torch.bfloat16, device=dev)
        ck_starts = ck_cpu.to(dev)
    o = torch.empty_like(d["v"])
    stream = torch.cuda.current_stream(dev)
    def step():
        kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], state,
                    cu_seqlens=d["cu_seqlens"], checkpoints=ck, checkpoint_cu_starts=ck_starts,
                    checkpoint_every_n_tokens=args.prefill_checkpoint, out=o, use_gate_in_kernel=True,
                    beta_is_logit=True, cu_seqlens_cpu=cu_cpu, checkpoint_cu_starts_cpu=ck_cpu)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    sec = t0.elapsed_time(t1) / 1e3 / args.steps
    esz = 2 if sdt == torch.bfloat16 else 4
    # q, k read per query/key head; v, g, beta read and o written per value head; every unit's state
    # read and written once; each checkpoint written once
    bytes_step = (Ttot * (512 * w.hqk + (256 * 3 + 2) * w.hv) + N * w.hv * 2 * esz * DIM * DIM
                  + n_ck * w.hv * 2 * DIM * DIM)
    peaks = read_peaks()
    achieved = bytes_step / sec / 1e9
    line = {"metric": "KDA prefill token·heads/s (1 GB300)", "value": Ttot * w.hv / sec, "unit": UNIT,
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec,
            "higher_is_better": True, "dtype": "fp32", "data": "synthetic",
            "config": {"workload": f"prefill_{args.workload}", "sequences": N, "tokens": Ttot, "Hqk": w.hqk,
                       "Hv": w.hv, "head_dim": DIM, "state_dtype": args.decode_state,
                       "checkpoint_every_n_tokens": args.prefill_checkpoint,
                       "l2": f"a prefill moves {bytes_step / 1e6:.0f} MB > 129 MB of L2, no flush"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"],
                         "traffic": ncu_traffic("kda_fwd_kernel_prefill", f"prefill_{args.workload}_"
                                                f"{args.decode_state}_ck{args.prefill_checkpoint}"),
                         "kernel": "kda_fwd_kernel (prefill)",
                         "peak_src": peaks["src"], "algorithmic_bytes_per_launch": bytes_step},
            "gpu_launches": args.steps, "clocks": clocks}
    print(json.dumps(line), flush=True)


def measure_e2e(x, d, dev, stream, kda_fwd, kda_bwd, token_heads, world, steps=64):
    """Inputs in pinned host memory; each step goes through the C-ABI call
    kda_step_host, which copies that step's inputs in, runs the forward and the
    backward and copies o, the final state and every gradient out. Two arenas
    take the steps in turn on shared copy-in, compute and copy-out streams, so
    step i+1's inputs and step i-1's outputs travel while step i computes; the
    timed region covers every step's copies and kernels, including the pipeline's
    fill (the first copy-in and the first kernels, before any copy-out) and its
    drain, about 10 ms in all on the packed 8 x 1024-token, 96-head workload, i.e.
    0.15 ms of each of the 64 steps."""
    import torch
    from linear_attention_gated_gb300 import HostStep
    names_in = ["q", "k", "v", "g", "beta", "A_log", "dt_bias", "h0", "do", "dfinal_state"]
    host_in = [x[k].pin_memory() for k in names_in]
    cu_cpu = x["cu_seqlens"]
    B, T, Hqk = x["q"].shape[:3]
    Hv = x["v"].shape[2]
    streams = [torch.cuda.Stream(dev) for _ in range(3)]
    runners = [HostStep(B, T, Hqk, Hv, cu_seqlens_cpu=cu_cpu, device=dev, stream=streams[0],
                        h2d_stream=streams[1], d2h_stream=streams[2]) for _ in range(2)]
    outs = [r.empty_outputs() for r in runners]
    h2d = sum(t.numel() * t.element_size() for t in host_in) + (cu_cpu.numel() * 8 if cu_cpu is not None else 0)
    d2h = sum(t.numel() * t.element_size() for t in outs[0])
    for i in range(2):  # warm-up: each arena once
        runners[i](*host_in, out=outs[i])
    for r in runners:
        r.synchronize()
    barrier(world)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for s_ in streams:
        s_.wait_stream(stream)
    for i in range(steps):
        runners[i % 2](*host_in, out=outs[i % 2])
    for s_ in streams:
        stream.wait_stream(s_)
    b.record(stream)
    torch.cuda.synchronize(dev)
    el = max_over_ranks(a.elapsed_time(b) / 1e3, world, dev)
    for r in runners:
        r.status()
    return {"value": job_value(token_heads, world, el / steps), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "api": "kda_step_host",
            "overlap": "two arenas taken in turn; copy-in, compute and copy-out streams; "
                       "the pipeline's fill and drain inside the timed region"}


if __name__ == "__main__":
    main()
