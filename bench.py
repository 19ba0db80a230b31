"""Benchmark: MoE-layer tokens/s (route + permute + expert FFN + combine) on B300, with the
roofline fraction of the dominant kernel and the fp64 oracle timed on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config v3_prefill] [--impl ours|reference]

One step = one moe_layer_forward (gate GEMM, routing, permutation, routed + shared SwiGLU
experts, combine) over one batch of synthetic inputs already resident in HBM. N > 1 runs N
independent replicas (one per GPU, launched by torch.distributed.run), weak scaling: the layer
forward of one GPU's batch has no cross-GPU exchange.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s (route+permute+expert FFN+combine); % of roofline"
# A timed region at least this long runs under the power cap: use the sustained bf16 peak.
LONG_REGION_MS = 500.0
# The oracle's CPU timing (both the cpu_baseline of our arm and every step of the reference
# arm): samples of this many random tokens of the batch, each timed once.
CPU_SAMPLE_TOKENS = 32
CPU_SAMPLES = 16


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--config", default="v3_prefill")
    p.add_argument("--tokens", type=int, default=None,
                   help="override the config's batch size T (profiling cases)")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-stages", action="store_true")
    p.add_argument("--no-graph", action="store_true",
                   help="launch every step eagerly instead of replaying a captured CUDA graph")
    return p.parse_args()


# ---------------------------------------------------------------- distributed plumbing
def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.init_process_group(backend="nccl")
    return world, rank, local


def max_over_ranks(v: float, world: int, device=None) -> float:
    """Slowest rank's value (the job takes as long as its slowest replica)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(ms_max: float, world: int, tokens_per_step: int, steps: int) -> float:
    """Whole-job throughput: the tokens every replica processed over the slowest replica's time."""
    return world * tokens_per_step * steps / (ms_max / 1e3)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- peaks, clocks
def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6400.0, bf16=1800.0, bf16_sus=1400.0, source="fallback")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.lines, self.proc = index, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        sm, mx, power, reasons = [], None, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
                power.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------- work accounting
def layer_work(cfg, counts, kept_rows: int) -> dict:
    """Algorithmic FLOPs and bytes of one layer forward (no credit for permutation copies)."""
    T, H, N, I, S, K = cfg.T, cfg.hidden, cfg.n_routed, cfg.inter, cfg.n_shared, cfg.top_k
    eb = cfg.elem_bytes
    touched = int(sum(1 for c in counts if c > 0))
    flops = 2.0 * T * H * N + 6.0 * H * I * (kept_rows + T * S)
    bytes_ = (2.0 * T * H * eb + N * H * eb + (touched + S) * 3.0 * H * I * eb
              + T * N * 4.0 + T * K * 8.0)
    return dict(flops=flops, bytes=bytes_, touched=touched,
                up_flops=4.0 * H * I * (kept_rows + T * S),
                down_flops=2.0 * H * I * (kept_rows + T * S),
                up_weight_bytes=(touched + S) * 2.0 * H * I * eb,
                down_weight_bytes=(touched + S) * 1.0 * H * I * eb,
                weight_bytes=(touched + S) * 3.0 * H * I * eb)


GEMM_SOURCES = ("gemm_tc.cu", "common.cuh", "internal.h")


def strip_comments(text: str) -> str:
    """C/C++ source without // and /* */ comments (string literals with comment markers are not
    expected in these files), blank lines and trailing spaces."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    out = []
    for line in text.splitlines():
        i = line.find("//")
        if i >= 0:
            line = line[:i]
        line = line.rstrip()
        if line.strip():
            out.append(line)
    return "\n".join(out)


def code_digest(*paths: str) -> str:
    """sha256 over the code of the given source files (comments and blank lines removed): a
    comment edit keeps it, any change to the code of any of the files does not."""
    import hashlib
    h = hashlib.sha256()
    for path in paths:
        with open(path, encoding="utf-8") as fh:
            h.update(os.path.basename(path).encode() + b"\0")
            h.update(strip_comments(fh.read()).encode() + b"\0")
    return h.hexdigest()


def gemm_digest() -> str:
    """Digest of the code the tensor-core GEMM kernels are built from: the kernel file, the
    inline-PTX helpers it includes and the argument layout it shares with the host."""
    csrc = os.path.join(ROOT, "mixture_experts_routing_sigmoid_b300", "csrc")
    return code_digest(*(os.path.join(csrc, f) for f in GEMM_SOURCES))


def traffic_per_launch(workload: str):
    """DRAM bytes (read + write) of one launch of the up GEMM on this workload, from the committed
    ncu capture of that workload; None when there is no capture of it or the kernel code has
    changed since the counters were taken. A capture taken on a smaller case of the same kernel
    carries its scale factor to the full launch (`scale_to`)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get("tc_gemm_kernel<MODE_UP>")
    if not d or d.get("source_code_digest") != gemm_digest():
        return None
    c = d.get("captures", {}).get(workload)
    if c is None:
        return None
    return float(c["dram_read_bytes"] + c["dram_write_bytes"]) * float(c.get("scale_to", 1.0))


def config_of(args):
    from moe_inputs import CONFIGS
    cfg = CONFIGS[args.config]
    if args.tokens is not None:
        cfg = cfg.replace(name=f"{cfg.name}_t{args.tokens}", T=args.tokens)
    return cfg


def workload_name(cfg) -> str:
    return (f"{cfg.name}: T={cfg.T} H={cfg.hidden} N={cfg.n_routed} G={cfg.n_groups} "
            f"Gk={cfg.topk_groups} K={cfg.top_k} S={cfg.n_shared} I={cfg.inter} "
            f"{cfg.score_fn} {cfg.dtype}")


# ---------------------------------------------------------------- our arm
def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    import mixture_experts_routing_sigmoid_b300 as moe
    from moe_inputs import CONFIGS, make_weights, make_x

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = config_of(args)
    T, H, K, N = cfg.T, cfg.hidden, cfg.top_k, cfg.n_routed
    w = make_weights(cfg, device=dev, seed=0)
    x = make_x(cfg, device=dev, seed=0)
    out = torch.empty_like(x)
    ws = torch.empty(moe.moe_workspace_size(cfg, T), dtype=torch.uint8, device=dev)
    want_stats = cfg.name == "v1"  # the v1 layer also reports f, P, L_B, L_Z
    counts = torch.empty(N, dtype=torch.int32, device=dev)
    lbz = torch.empty(3, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(s):
        moe.moe_layer_forward(cfg, T, x, w, out, counts if want_stats else None,
                              lbz if want_stats else None, ws, s)

    for _ in range(args.warmup):
        step(stream)
    st = moe.moe_get_error(stream)
    if st != 0:
        raise RuntimeError(f"device error {st} during warm-up")

    # ---- device-timed region (inputs resident in HBM; expert weights far above L2). By default
    # the K steps are captured once into a CUDA graph (launch overheads matter for small decode
    # batches) and the graph is replayed once untimed, then once timed. The headline region runs
    # the layer as a user would, with no instrumentation; a second timed region of the same K
    # steps records CUDA events at every stage boundary (on the launching stream, as graph
    # nodes), and the per-kernel times and the roofline come from it.
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed_region(with_stages: bool, sample_clocks: bool):
        if with_stages:
            moe.moe_stage_timing_start(args.steps)
        graph = None
        launches0 = moe.moe_kernel_launches()
        launches = 0
        if not args.no_graph:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, capture_error_mode="relaxed"):
                cs = torch.cuda.current_stream(dev)
                for _ in range(args.steps):
                    step(cs)
            launches = moe.moe_kernel_launches() - launches0  # what each replay runs
            graph.replay()
            torch.cuda.synchronize(dev)
        barrier(world)
        torch.cuda.synchronize(dev)
        clk = ClockSampler(local) if sample_clocks else None
        if clk is not None:
            clk.__enter__()
        ev0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for _ in range(args.steps):
                step(stream)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        if clk is not None:
            clk.__exit__(None, None, None)
        if graph is None:
            launches = moe.moe_kernel_launches() - launches0
        barrier(world)
        ms_ = ev0.elapsed_time(ev1)
        stages_, ncalls_ = moe.moe_stage_timing_stop() if with_stages else ({}, 0)
        del graph
        st_ = moe.moe_get_error(stream)
        if st_ != 0:
            raise RuntimeError(f"device error {st_} in the timed region")
        return ms_, launches, clk, stages_, ncalls_

    ms, launches, clk, _, _ = timed_region(False, True)
    stages, ncalls, ms_staged = {}, 0, None
    if not args.no_stages:
        ms_staged, _, _, stages, ncalls = timed_region(True, False)
    ms_max = max_over_ranks(ms, world, dev)
    ms_step = ms_max / args.steps
    tok_s = job_tokens_per_s(ms_max, world, T, args.steps)

    # routing outcome of this batch (for the work accounting)
    idx = torch.empty((T, K), dtype=torch.int32, device=dev)
    wt = torch.empty((T, K), dtype=torch.float32, device=dev)
    moe.moe_route(cfg, T, x, w, None, None, idx, wt, ws, stream)
    offs = torch.empty(N + 1, dtype=torch.int32, device=dev)
    rt = torch.empty(T * K, dtype=torch.int32, device=dev)
    sr = torch.empty(T * K, dtype=torch.int32, device=dev)
    moe.moe_permute(cfg, T, idx, wt, None, offs, rt, sr, None, ws, stream)
    offs_h = offs.cpu().numpy()
    kept_rows = int(offs_h[-1])
    work = layer_work(cfg, np.diff(offs_h), kept_rows)
    pk = peaks()

    result = {
        "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype,
        "data": "synthetic (seeded; random-init weights of the layer's shapes)",
        "config": {"workload": workload_name(cfg), "T": T, "hidden": H, "n_routed": N,
                   "top_k": K, "n_shared": cfg.n_shared, "inter": cfg.inter,
                   "parallelism": "replicas" if world > 1 else "single-gpu",
                   "l2": "inputs larger than L2: expert weights touched per step %.2f GB "
                         "(L2 126 MB), no flush" % (work["weight_bytes"] / 1e9),
                   "kept_rows": kept_rows, "touched_experts": work["touched"]},
        "gpu_launches": launches,
        "launch": ("CUDA graph of the timed steps" if not args.no_graph else "eager")
                  + "; kernels start while the kernel ahead of them finishes (dependent launches)",
    }
    # Tensor peak: the measured sustained bf16 rate when the timed region is long (the GPU
    # then runs under its power cap, as the sustained measurement did), else the burst rate.
    sustained = ms_max >= LONG_REGION_MS
    bf16_peak = pk["bf16_sus"] if sustained else pk["bf16"]
    bf16_kind = ("bf16 sustained" if sustained else "bf16 burst") + ", " + pk["source"]
    t_flop = work["flops"] / (bf16_peak * 1e12)
    t_byte = work["bytes"] / (pk["hbm_gbs"] * 1e9)
    t_roof = max(t_flop, t_byte)
    result["layer_roofline"] = {
        "flops": work["flops"], "bytes": work["bytes"], "roofline_ms": t_roof * 1e3,
        "frac": t_roof * 1e3 / ms_step, "tflops": work["flops"] / (ms_step * 1e-3) / 1e12,
        "weight_gbs": work["weight_bytes"] / (ms_step * 1e-3) / 1e9,
        "bound": "tensor" if t_flop >= t_byte else "hbm",
        "peaks": f"{bf16_kind} ({bf16_peak} TFLOP/s), HBM copy ({pk['hbm_gbs']} GB/s)",
        "frac_vs_burst_peak": max(work["flops"] / (pk["bf16"] * 1e12), t_byte) * 1e3 / ms_step}
    result["clocks"] = clk.summary()

    # ---- the dominant kernel (the SwiGLU up GEMM) against its own roofline
    if stages and ncalls:
        per = {k: v / ncalls for k, v in stages.items()}
        up = per["up"]
        traffic = traffic_per_launch(cfg.name)
        if result["layer_roofline"]["bound"] == "tensor":
            up_tf = work["up_flops"] / (up * 1e-3) / 1e12
            result["roofline"] = {
                "kernel": "tc_gemm_kernel<MODE_UP> (grouped SwiGLU up projection, tcgen05)",
                "bound": "tensor", "achieved": up_tf, "peak": bf16_peak, "unit": "TFLOP/s",
                "frac": up_tf / bf16_peak, "traffic": traffic,
                "peak_kind": bf16_kind,
                "frac_of_burst": up_tf / pk["bf16"], "avg_launch_ms": up,
                "algorithmic_flops_per_launch": work["up_flops"]}
        else:
            gbs = work["up_weight_bytes"] / (up * 1e-3) / 1e9
            result["roofline"] = {
                "kernel": "tc_gemm_kernel<MODE_UP> (grouped SwiGLU up projection, tcgen05)",
                "bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / pk["hbm_gbs"], "traffic": traffic,
                "peak_kind": "HBM copy, " + pk["source"], "avg_launch_ms": up,
                "algorithmic_bytes_per_launch": work["up_weight_bytes"]}
        dn = per["down"]
        result["kernels"] = {
            "avg_ms": per,
            "share_of_step": {k: v / ms_step for k, v in per.items()},
            "up_tflops": work["up_flops"] / (up * 1e-3) / 1e12,
            "down_tflops": work["down_flops"] / (dn * 1e-3) / 1e12,
            "up_weight_gbs": work["up_weight_bytes"] / (up * 1e-3) / 1e9,
            "down_weight_gbs": work["down_weight_bytes"] / (dn * 1e-3) / 1e9,
            "timing": "CUDA events at the stage boundaries of a second timed region of the same "
                      "K steps (graph-replayed, launching stream); its step time is "
                      "ms_per_step_with_stage_events",
            "ms_per_step_with_stage_events": ms_staged / args.steps}

    # ---- end to end through the C ABI: every step copies its input from pinned host memory and
    # its output back. Double-buffered on two copy streams, so that step i+1's input and step
    # i-1's output move while step i computes (the copies are inside the timed region).
    if not args.no_e2e:
        xh = x.cpu().pin_memory()
        xd = [torch.empty_like(x) for _ in range(2)]
        od = [torch.empty_like(out) for _ in range(2)]
        oh = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def e2e_run(main, nsteps):
            start = torch.cuda.Event()
            start.record(main)
            h2d_s.wait_event(start)
            d2h_s.wait_event(start)
            h2d_done = [torch.cuda.Event() for _ in range(2)]
            comp_done = [torch.cuda.Event() for _ in range(2)]
            d2h_done = [torch.cuda.Event() for _ in range(2)]
            for i in range(nsteps):
                b = i % 2
                if i >= 2:
                    h2d_s.wait_event(comp_done[b])     # step i-2 has read xd[b]
                with torch.cuda.stream(h2d_s):
                    xd[b].copy_(xh, non_blocking=True)
                h2d_done[b].record(h2d_s)
                main.wait_event(h2d_done[b])
                if i >= 2:
                    main.wait_event(d2h_done[b])       # step i-2's output has left od[b]
                moe.moe_layer_forward(cfg, T, xd[b], w, od[b], None, None, ws, main)
                comp_done[b].record(main)
                d2h_s.wait_event(comp_done[b])
                with torch.cuda.stream(d2h_s):
                    oh[b].copy_(od[b], non_blocking=True)
                d2h_done[b].record(d2h_s)
            for b in range(min(nsteps, 2)):
                main.wait_event(d2h_done[b])

        e2e_run(stream, args.warmup)
        graph = None
        if not args.no_graph:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, capture_error_mode="relaxed"):
                e2e_run(torch.cuda.current_stream(dev), args.steps)
            graph.replay()
        barrier(world)
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            e2e_run(stream, args.steps)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        del graph
        e2e_ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
        result["e2e"] = {"value": job_tokens_per_s(e2e_ms, world, T, args.steps), "unit": "tokens/s",
                         "h2d_bytes_per_step": xh.numel() * xh.element_size(),
                         "d2h_bytes_per_step": oh[0].numel() * oh[0].element_size(),
                         "overlap": "inputs and outputs double-buffered on two copy streams"}

    # ---- the oracle on the host cores (rank 0, N = 1 only), bounded sample
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # about 10 s of host work: CPU_SAMPLES samples of CPU_SAMPLE_TOKENS tokens each, the
        # same per-sample recipe as the reference arm's steps
        result["cpu_baseline"] = oracle_baseline(cfg, x, w, n_tokens=CPU_SAMPLE_TOKENS,
                                                 steps=CPU_SAMPLES, seed=1)
    return result


def oracle_baseline(cfg, x, w, n_tokens: int, steps: int, seed: int = 0, repeat: int = 1) -> dict:
    """Time the fp64 oracle (as it stands) on `steps` samples of `n_tokens` tokens each, each
    sample run `repeat` times (a longer timed span without staging more expert weights).

    The experts a sample touches are copied to host memory before its timed calls."""
    import numpy as np
    import torch

    import oracle
    rng = np.random.default_rng(seed)
    f64 = (lambda t: None if t is None else t.double().cpu().numpy())
    wg, gb, sb = f64(w["w_gate"]), f64(w["gate_logit_bias"]), f64(w["select_bias"])
    host = {}
    for s_ in range(cfg.n_shared):
        host[("s", s_)] = (w["w13_shared"][s_].cpu(), w["w2_shared"][s_].cpu())
    ew = (lambda e: host[("r", e)])
    sw = (lambda s: host[("s", s)])
    total_s, total_tok = 0.0, 0
    xs_all = f64(x) if cfg.capacity_drop else None
    for _ in range(steps):
        tok = np.sort(rng.choice(cfg.T, size=min(n_tokens, cfg.T), replace=False))
        # untimed: route the sample once to learn which experts to stage on the host
        xr = f64(x[torch.as_tensor(tok).long().to(x.device)])
        u = oracle.gate_logits(xs_all if cfg.capacity_drop else xr, wg, gb)
        idx, _, _ = oracle.route(cfg.replace(T=u.shape[0]), oracle.scores(u, cfg.score_fn), sb)
        for e in np.unique(idx):
            if ("r", int(e)) not in host:
                host[("r", int(e))] = (w["w13"][int(e)].cpu(), w["w2"][int(e)].cpu())
        t0 = time.perf_counter()
        for _ in range(repeat):
            if cfg.capacity_drop:
                oracle.layer_forward(cfg, xs_all, wg, gb, sb, ew, sw, tokens=tok)
            else:
                oracle.layer_forward(cfg.replace(T=len(tok)), xr, wg, gb, sb, ew, sw)
        total_s += time.perf_counter() - t0
        total_tok += len(tok) * repeat
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return {"value": total_tok / total_s, "unit": "tokens/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{steps} x {n_tokens} random tokens of the {cfg.name} batch"
                      + (f", each sample timed {repeat} times" if repeat > 1 else "") + ": gate logits, "
                      f"routing, {cfg.top_k} routed + {cfg.n_shared} shared SwiGLU experts and "
                      f"the combine in fp64; the expert weights a sample touches are staged in "
                      f"host memory before its timed call (staging not timed)"
                      + ("; gate and routing over the whole batch for the drop"
                         if cfg.capacity_drop else ""),
            "seconds": total_s}


# ---------------------------------------------------------------- reference arm
def run_reference(args, world, rank, local):
    """The oracle, as it stands, on the host cores: same metric / unit / config as our arm."""
    import torch
    from moe_inputs import CONFIGS, make_weights, make_x
    cfg = config_of(args)
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    w = make_weights(cfg, device=dev, seed=0)
    x = make_x(cfg, device=dev, seed=0)
    if args.warmup:
        oracle_baseline(cfg, x, w, n_tokens=CPU_SAMPLE_TOKENS, steps=1, seed=99)
    # one step = one sample of CPU_SAMPLE_TOKENS tokens, as in our arm's cpu_baseline
    cb = oracle_baseline(cfg, x, w, n_tokens=CPU_SAMPLE_TOKENS, steps=args.steps, seed=1)
    ms_step = cb["seconds"] / args.steps * 1e3
    return {"metric": METRIC, "value": cb["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; random-init weights of the layer's shapes)",
            "config": {"workload": workload_name(cfg), "T": cfg.T, "hidden": cfg.hidden,
                       "n_routed": cfg.n_routed, "top_k": cfg.top_k,
                       "n_shared": cfg.n_shared, "inter": cfg.inter,
                       "parallelism": "host cores"},
            "impl": "reference",
            "cpu_baseline": {"value": cb["value"], "unit": "tokens/s", "cores": cb["cores"],
                             "kind": "oracle", "sample": cb["sample"]},
            "e2e": {"value": cb["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    world, rank, local = dist_init(args)
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, world, rank, local)), flush=True)
    else:
        res = run_ours(args, world, rank, local)
        if rank == 0:
            print(json.dumps(res), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
