"""Benchmark: routing time of one microbatch (every site's forward + backward).

One step = one microbatch of the depth-routing path: the source appends
(inverse RMS), the forward of every routing site in order, and the backward of
every site in reverse (source gradients accumulated in the shared fp32 rows,
dq/dg reduced). Default workload: the 1B-shaped model (d=1280, 36 layers ->
73 sites, H=8, T=16x1024 tokens, bf16).

Prints ONE JSON line (rank 0). ``value`` is whole-job tokens/s with inputs
resident in HBM (each step captured as two CUDA graphs, forward and
backward, replayed back to back); ``e2e`` is the same metric through the
public API with the step's inputs copied from pinned host memory and its
parameter gradients copied back, inside the timed region.

Multi-GPU (torchrun): every rank routes its own microbatch (tokens shard with
no exchange in the routing path), weak scaling; time = max over ranks.

``--impl reference`` times the CPU oracle (its float32 build) on the host
cores instead: each step is one bounded token sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "route_bwd_traffic.json")
# GB300's nominal HBM3e bandwidth (~8 TB/s); fractions are also reported against it
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
METRIC = "routing ms per microbatch fwd+bwd (all sites), tokens/s, % of HBM roofline"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", default="1B")
    p.add_argument("--heads", type=int, default=None)
    p.add_argument("--tokens", type=int, default=None, help="override T (profiling cases)")
    p.add_argument("--sites", default="all",
                   help="all: every routing site; last: only the last one; an integer k: "
                        "only site k (profiling cases)")
    p.add_argument("--e2e-steps", type=int, default=None)
    p.add_argument("--cpu-seconds", type=float, default=15.0,
                   help="target wall time of the CPU-oracle sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--eager", action="store_true", help="no CUDA graphs")
    p.add_argument("--multi-read", type=int, metavar="Q", default=None,
                   help="time ar_route_fwd_multi instead: Q queries read the largest site's row "
                        "list of the workload in one pass (two-phase block inference, phase 1), "
                        "against Q single reads")
    p.add_argument("--report", metavar="DIR", default=None,
                   help="run every workload (each in its own process) and write DIR/report.json "
                        "and DIR/report.md")
    return p.parse_args()


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# Sources of the backward kernel each workload's roofline entry measures.
KERNEL_SOURCES = {
    "full": ("kernels_bwd.cuh", "common.cuh", "ar_internal.h", "launch_util.cuh", "shapes.h"),
    "coop": ("kernels_coop.cuh", "common.cuh", "ar_internal.h", "launch_util.cuh", "shapes.h"),
    "lr": ("kernels_lr.cuh", "common.cuh", "ar_internal.h", "launch_util.cuh", "shapes.h"),
}


def _code_only(text: str) -> str:
    """C++ source without comments and blank lines (comment edits keep the hash)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_hash(family: str = "full") -> str:
    """Hash of the code (not the comments) of a kernel family's sources."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "depth_wise_attention_ar_gb300", "csrc")
    for name in KERNEL_SOURCES[family]:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(config: str, H: int, bytes_per_launch: float, T: int):
    """DRAM bytes per backward launch at full size, from the small-case ncu
    captures recorded in profiles/route_bwd_traffic.json: the launch's
    algorithmic bytes, plus the forward output it reads per token (outside
    the byte model), less the write tail those captures found still dirty in
    L2 at the end of each launch. None when there is no record for the
    workload or the kernel's code changed since it was taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)["configs"]
        e = rec.get(f"{config}/H{H}")
        if e and e.get("kernel_hash") == kernel_hash(e.get("family", "full")):
            return bytes_per_launch + T * e["output_bytes_per_token"] - e["tail_bytes"]
    except (OSError, ValueError, KeyError):   # no record, or an unreadable one
        pass
    return None


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax = float(f[1])
            except ValueError:
                continue
            for nm, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_baseline(cfg, H, seconds: float, steps: int = 1, warmup: int = 0):
    """The oracle's float32 build (C, OpenMP over tokens, all host cores) on a
    token sample of the workload: every site's forward in order and every
    site's backward in reverse; `warmup` untimed runs, then the mean of
    `steps` timed runs."""
    import numpy as np

    import oracle
    import synth
    from oracle import schedule, storage

    oplan = schedule.block_plan(cfg.M, cfg.NB)
    run = list(cfg.sites) if cfg.sites is not None else list(range(len(oplan["sites"])))
    nrows = max(max(oplan["sites"][s]) for s in run) + 1
    f32 = np.float32

    def one(Ts):
        outs = [synth.storage_to_f64(synth.sublayer_output(1, j, Ts, cfg.d, cfg.dtype), cfg.dtype)
                for j in range(nrows)]
        rows = [x.astype(f32) for x in
                storage.block_bank(outs, {"row_ops": oplan["row_ops"][:nrows]}, cfg.dtype)]
        qs = {s: synth.site_query(1, s, cfg.r) for s in run}
        gouts = {s: synth.storage_to_f32(synth.site_dout(1, s, Ts, cfg.d, cfg.dtype), cfg.dtype)
                 for s in run}
        dsrc = {j: np.zeros((Ts, cfg.d), dtype=f32) for j in range(nrows)}
        t0 = time.perf_counter()
        for s in run:
            oracle.route_fwd([rows[j] for j in oplan["sites"][s]], qs[s], None, H, r=cfg.r,
                             precision="f32")
        for s in reversed(run):
            oracle.route_bwd([rows[j] for j in oplan["sites"][s]], qs[s], None, gouts[s], H,
                             r=cfg.r, dsrc=[dsrc[j] for j in oplan["sites"][s]],
                             precision="f32")
        return time.perf_counter() - t0

    threads = oracle.threads()
    # size the sample from two small probes: a run costs a + b * tokens (a:
    # per-call overheads, which dominate small runs)
    t1, t2 = 8 * threads, 32 * threads
    p1, p2 = one(t1), one(t2)
    b = max((p2 - p1) / (t2 - t1), 1e-9)
    a = max(p1 - b * t1, 0.0)
    Ts = int(min(cfg.T, max(t2, (seconds - a) / b)))
    Ts = max(threads, (Ts // threads) * threads)
    for _ in range(warmup):
        one(Ts)
    times = [one(Ts) for _ in range(steps)]
    dt = sum(times) / len(times)
    return {"value": Ts / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{Ts} of {cfg.T} tokens, every site forward + backward in reverse, "
                      f"float32 build of the oracle, {dt:.1f} s per sample"}, dt, Ts


def line_config(cfg, H, world, sites, run):
    """The `config` object of the JSON line, the same for both arms (`sites`:
    every site's row list; `run`: the sites that run)."""
    nrows = max(max(sites[s]) for s in run) + 1
    b = 2 if cfg.dtype == "bf16" else 4
    return {"workload": f"{cfg.name}-shaped routing microbatch", "T": cfg.T, "d": cfg.d, "H": H,
            "r": cfg.r, "sites": len(run), "sources_read": sum(len(sites[s]) for s in run),
            "global_batch_tokens": world * cfg.T, "parallelism": f"dp{world} (token shards)",
            "l2": f"inputs larger than L2 (bank {nrows * cfg.T * cfg.d * b / 1e9:.2f} GB)"}


def max_over_ranks(values, device="cpu"):
    """Element-wise maximum of per-rank timings (the slowest rank sets the
    step time); identity on a single process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def config_of(args, workload):
    import dataclasses
    cfg = workload.CONFIGS[args.config]
    if args.tokens:
        cfg = dataclasses.replace(cfg, T=args.tokens)
    if args.sites == "last":
        cfg = dataclasses.replace(cfg, sites=(cfg.M,))
    elif args.sites != "all":
        k = int(args.sites)
        if not 0 <= k <= cfg.M:
            raise SystemExit(f"--sites {k}: the workload has sites 0..{cfg.M}")
        cfg = dataclasses.replace(cfg, sites=(k,))
    return cfg


# (config, heads or None) of the report: the shaped workloads, the 1B head
# sweep, and the rows past the hot path
REPORT_RUNS = [("1B", None), ("1B", 1), ("1B", 4), ("1B", 16), ("350M", None), ("100M", None),
               ("lr_block", None), ("delta_8b", None), ("lr_page_1b", None), ("lr_page_4b", None)]


def report(args):
    """Every workload through this script, one process each; JSON + Markdown."""
    os.makedirs(args.report, exist_ok=True)
    lines = []
    for cfg, heads in REPORT_RUNS:
        cmd = [sys.executable, os.path.abspath(__file__), "--config", cfg, "--steps", str(args.steps),
               "--warmup", str(args.warmup), "--cpu-seconds", str(args.cpu_seconds)]
        if heads:
            cmd += ["--heads", str(heads)]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"{' '.join(cmd)} failed:\n{p.stderr[-2000:]}")
        lines.append(json.loads(p.stdout.strip().splitlines()[-1]))
    with open(os.path.join(args.report, "report.json"), "w") as f:
        json.dump(lines, f, indent=1)
    rows = ["| workload | H | ms / microbatch | tokens/s | of roofline | forward + appends (ms) | "
            "backward (ms, of roofline) | end to end (ms) | host link alone (GB/s) | SM MHz |",
            "|---|---|---|---|---|---|---|---|---|---|"]
    for L in lines:
        c, ph, e = L["config"], L["phases_ms"], L.get("e2e") or {}
        rows.append(f"| {c['workload']} | {c['H']} | {L['ms_per_step']:.2f} | {L['value']:,.0f} | "
                    f"{100 * L['step_roofline']['frac']:.1f} % | {ph['forward_and_appends']:.2f} | "
                    f"{ph['backward']:.2f} ({100 * L['roofline']['frac']:.1f} %) | "
                    f"{e.get('ms_per_step', float('nan')):.1f} | {e.get('h2d_gbs_alone', float('nan')):.0f} | "
                    f"{L['clocks'].get('sm_mhz')} |")
    rows.append("")
    rows.append("CPU oracle (float32 build, all host cores) on a token sample of each workload:")
    rows.append("")
    rows.append("| workload | H | oracle tokens/s | cores | GPU / oracle | sample |")
    rows.append("|---|---|---|---|---|---|")
    for L in lines:
        cb = L.get("cpu_baseline")
        if cb:
            c = L["config"]
            rows.append(f"| {c['workload']} | {c['H']} | {cb['value']:,.1f} | {cb['cores']} | "
                        f"{L['value'] / cb['value']:,.0f} | {cb['sample']} |")
    with open(os.path.join(args.report, "report.md"), "w") as f:
        f.write("\n".join(rows) + "\n")
    print("\n".join(rows))


def main():
    args = parse()
    if args.report:
        return report(args)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return reference_arm(args, rank, world)
    if args.multi_read:
        return multi_read(args)

    import torch
    import torch.distributed as dist

    import synth
    from depth_wise_attention_ar_gb300 import binding, workload

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    cfg = config_of(args, workload)
    H = args.heads or cfg.H
    inputs = synth.DeviceInputs(seed=1000 + rank, device=f"cuda:{local}")
    mb = workload.Microbatch(cfg, H, inputs, device=f"cuda:{local}")
    stream = torch.cuda.Stream()
    mbytes = workload.model_bytes(cfg, mb.plan, H)

    # warm-up (eager): fills the launch caches, checks the device error word
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup)):
            mb.step()
    torch.cuda.synchronize()
    if binding.ar_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    use_graph = not args.eager
    if use_graph:
        g_fwd, g_bwd = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_fwd, stream=stream):
            mb.forward()
        with torch.cuda.graph(g_bwd, stream=stream):
            mb.backward()
        run_fwd, run_bwd = g_fwd.replay, g_bwd.replay
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                run_fwd()
                run_bwd()
    else:
        def run_fwd():
            mb.forward()

        def run_bwd():
            mb.backward()
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        for k in range(K):
            ev[k][0].record(stream)
            run_fwd()
            ev[k][1].record(stream)
            run_bwd()
            ev[k][2].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    total_ms = ev[0][0].elapsed_time(ev[K - 1][2])
    fwd_ms = sum(ev[k][0].elapsed_time(ev[k][1]) for k in range(K)) / K
    bwd_ms = sum(ev[k][1].elapsed_time(ev[k][2]) for k in range(K)) / K
    if world > 1:
        total_ms, fwd_ms, bwd_ms = max_over_ranks([total_ms, fwd_ms, bwd_ms],
                                                  device=f"cuda:{local}")
    ms = total_ms / K
    per_step = sorted(ev[k][0].elapsed_time(ev[k][2]) for k in range(K))
    if binding.ar_device_error() != 0:
        raise RuntimeError("device error word set during the timed region")

    # end to end through the public API: inputs from pinned host memory
    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(args, mb, stream, run_fwd, run_bwd, world, local)

    hbm, peak_kind = peaks()
    n_bwd = len(mb.plan.run_sites)
    bwd_bytes = mbytes["bwd"]
    achieved = bwd_bytes / (bwd_ms * 1e-3) / 1e9
    # the record holds the mean over every site of the full workload: another
    # token count or site selection is a different launch mix
    traffic = (measured_traffic(args.config, H, bwd_bytes / n_bwd, cfg.T)
               if args.sites == "all" and not args.tokens else None)
    line = {
        "metric": METRIC,
        "value": world * cfg.T / (ms * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": cfg.dtype,
        "compute": f"fp32 arithmetic on {cfg.dtype} rows; fp32 gradient rows, lse, dq, dg",
        "data": "synthetic (seeded torch Philox on device; recipe of the 1B/100M/350M/LR models)",
        "config": line_config(cfg, H, world, mb.plan.sites, mb.plan.run_sites),
        "cuda_graphs": use_graph,
        "phases_ms": {"forward_and_appends": fwd_ms, "backward": bwd_ms},
        "step_ms_spread": {"median": per_step[K // 2], "min": per_step[0], "max": per_step[-1]},
        "model_bytes": mbytes,
        "step_roofline": {"achieved": mbytes["total"] / (ms * 1e-3) / 1e9, "peak": hbm,
                          "unit": "GB/s", "frac": mbytes["total"] / (ms * 1e-3) / 1e9 / hbm,
                          "frac_of_nominal": mbytes["total"] / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS,
                          "peak_source": peak_kind},
        "roofline": {"kernel": "the backward kernel (route_bwd_*; backward phase, incl. its dq/dg reduce)",
                     "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "nominal_peak": NOMINAL_HBM_GBS, "traffic": traffic,
                     "traffic_source": "ncu DRAM bytes of small-case backward launches "
                                       "(profiles/route_bwd_traffic.json): the algorithmic "
                                       "bytes per launch plus the forward output read per "
                                       "token, less the write tail still in L2 at each "
                                       "launch's end; null if the kernel changed since",
                     "launches_per_step": n_bwd,
                     "bytes_per_launch_avg": bwd_bytes / n_bwd,
                     "ms_per_launch_avg": bwd_ms / n_bwd,
                     "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json copy bandwidth)"},
        "gpu_launches": K * mb.kernel_launches(),
        "clocks": clk,
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb, _, _ = cpu_baseline(cfg, H, args.cpu_seconds)
        line["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def end_to_end(args, mb, stream, run_fwd, run_bwd, world, local):
    """Same step through the public API with host buffers: H2D of the step's
    inputs (source rows, upstream gradients, the packed per-site queries, norm
    weights and gates) from pinned memory, the routing step, D2H of the packed
    per-site dq/dg (and gate gradients) of every step.

    As a training loop's input pipeline would, the input copies run on their
    own stream and are double-buffered: two device buffer sets alternate between
    steps, the next step's inputs stream in while the current step computes,
    and each append / backward waits only for its own input. Every step's
    copies are inside the timed region. The step is issued eagerly, so that
    those waits sit between its launches."""
    import torch
    import torch.distributed as dist

    from depth_wise_attention_ar_gb300 import workload

    cfg, plan = mb.cfg, mb.plan
    sites = list(plan.run_sites)
    last = max(sites)
    mbs = [mb, workload.Microbatch(cfg, mb.H, mb.inputs, device=mb.device)]

    def pinned(t):
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        return h

    # host copies of one step's inputs (the same data feeds both buffer sets)
    h_small = pinned(mb.small_in)
    h_rows = {}                                  # inputs needed at step t of the forward
    for t in range(last + 1):
        lst = []
        if t < mb.n_rows and not (t == 0 and cfg.delta):
            lst.append(pinned(mb.outputs[t] if t in mb.outputs else mb.bank.rows[t]))
        if cfg.delta and t in mb.partial:
            lst.append(pinned(mb.partial[t]))
        h_rows[t] = lst
    h_dout = {s: pinned(mb.dout[s]) for s in sites}
    h_null = pinned(mb.null) if cfg.delta else None
    host_out = [torch.empty(mb.small_out.shape, dtype=torch.float32, pin_memory=True)
                for _ in range(2)]

    def dev_rows(M, t):
        lst = []
        if t < M.n_rows and not (t == 0 and cfg.delta):
            lst.append(M.outputs[t] if t in M.outputs else M.bank.rows[t])
        if cfg.delta and t in M.partial:
            lst.append(M.partial[t])
        return lst

    h2d = (h_small.numel() * 4 + sum(h.numel() * h.element_size() for v in h_rows.values()
                                     for h in v) +
           sum(h.numel() * h.element_size() for h in h_dout.values()) +
           (h_null.numel() * h_null.element_size() if cfg.delta else 0))
    d2h = host_out[0].numel() * 4
    K = args.e2e_steps or max(2, min(args.steps, 6))
    h2d_stream = torch.cuda.Stream()
    ev_small = [torch.cuda.Event() for _ in range(2)]
    ev_t = [{t: torch.cuda.Event() for t in h_rows} for _ in range(2)]
    ev_d = [{s: torch.cuda.Event() for s in sites} for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]

    def issue_copies(b):
        M = mbs[b]
        with torch.cuda.stream(h2d_stream):
            h2d_stream.wait_event(done[b])       # the step that last used this set is done
            M.small_in.copy_(h_small, non_blocking=True)
            if cfg.delta:
                M.null.copy_(h_null, non_blocking=True)
            ev_small[b].record(h2d_stream)
            for t in range(last + 1):
                for dst, src in zip(dev_rows(M, t), h_rows[t]):
                    dst.copy_(src, non_blocking=True)
                ev_t[b][t].record(h2d_stream)
            for s in reversed(sites):
                M.dout[s].copy_(h_dout[s], non_blocking=True)
                ev_d[b][s].record(h2d_stream)

    def compute(b):
        M = mbs[b]

        def on_site(kind, t):
            if kind == "fwd_begin":
                stream.wait_event(ev_t[b][t])
            elif kind == "bwd_begin":
                stream.wait_event(ev_d[b][t])

        stream.wait_event(ev_small[b])
        M.forward(stream, on_site=on_site)
        M.backward(stream, on_site=on_site)
        done[b].record(stream)
        # the step's result (one packed buffer) follows the step on its own
        # stream: a read-back queued on a separate copy stream behind this
        # step's end held up the next step's input copies
        host_out[b].copy_(M.small_out, non_blocking=True)

    def run(k_steps):
        # the input copies are queued a step ahead of the compute that
        # frees their buffers: when the host runs ahead of the GPU, a launch
        # call blocks until the queue drains, and copies queued only after
        # that call came too late for the next step
        h2d_stream.wait_stream(stream)
        issue_copies(0)
        if k_steps > 1:
            issue_copies(1)
        for k in range(k_steps):
            compute(k % 2)
            if k + 2 < k_steps:
                issue_copies(k % 2)              # step k + 2 reuses step k's buffers
        stream.wait_stream(h2d_stream)

    with torch.cuda.stream(stream):
        run(2)                                   # warm-up: both buffer sets
    torch.cuda.synchronize()
    # the host link alone: one step's input copies with nothing else running,
    # three times, the median kept (the host's memory and links are shared
    # with other jobs on the machine, so the end-to-end figure is read
    # against this)
    probes = []
    for _ in range(3):
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(h2d_stream):
            c0.record(h2d_stream)
        issue_copies(0)
        with torch.cuda.stream(h2d_stream):
            c1.record(h2d_stream)
        torch.cuda.synchronize()
        probes.append(h2d / (c0.elapsed_time(c1) * 1e-3) / 1e9)
    h2d_gbs_alone = sorted(probes)[1]
    if world > 1:
        dist.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        run(K)
        t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / K
    if world > 1:
        (ms,) = max_over_ranks([ms], device=f"cuda:{local}")
    del mbs[1]
    # the copies alone at the probed rate; a probe slower than the loop itself
    # saw (the step moved the same bytes faster) is no bound, so none is given
    copy_ms = h2d / (h2d_gbs_alone * 1e9) * 1e3
    return {"value": world * mb.cfg.T / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "steps": K, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "h2d_gbs_alone": h2d_gbs_alone, "h2d_gbs_probes": probes,
            "copy_bound_ms": copy_ms if copy_ms <= ms else None,
            "copies": "H2D on its own stream, double-buffered: the next step's inputs stream "
                      "in while the current step computes; D2H of each step's packed dq/dg "
                      "after the step"}


def multi_read(args):
    """One JSON line: Q queries over one row list (the workload's largest site)
    in one ar_route_fwd_multi launch, timed with CUDA events on its stream
    (inputs larger than L2), against the same Q reads one site at a time."""
    import torch

    import synth
    from depth_wise_attention_ar_gb300 import binding, workload

    torch.cuda.set_device(0)
    cfg = config_of(args, workload)
    H = args.heads or cfg.H
    Q = args.multi_read
    plan = workload.make_plan(cfg)
    rows = max((plan.sites[s] for s in plan.run_sites), key=len)
    inputs = synth.DeviceInputs(seed=3)
    bank = binding.Bank(cfg.T, cfg.d, cfg.r, max(rows) + 1, cfg.dtype, device="cuda")
    for j in range(max(rows) + 1):
        bank.append(inputs.output(j, cfg.T, cfg.d, cfg.dtype))
    qs = [inputs.query(k, cfg.r) for k in range(Q)]
    outs = [torch.empty((cfg.T, cfg.d), dtype=bank.torch_dtype, device="cuda") for _ in range(Q)]
    lses = [torch.empty((cfg.T, H), dtype=torch.float32, device="cuda") for _ in range(Q)]
    stream = torch.cuda.Stream()

    def multi():
        bank.route_fwd_multi(rows, H, qs, None, outs, lses, stream=stream)

    def singles():
        for k in range(Q):
            binding.ar_route_fwd(bank.handle, rows, H, qs[k], None, outs[k], lses[k], k, stream)

    def timed(fn):
        with torch.cuda.stream(stream):
            for _ in range(max(3, args.warmup)):
                fn()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            ev[0].record(stream)
            for _ in range(args.steps):
                fn()
            ev[1].record(stream)
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1]) / args.steps

    ms_multi, ms_single = timed(multi), timed(singles)
    if binding.ar_device_error() != 0:
        raise RuntimeError("device error word set")
    b = 2 if cfg.dtype == "bf16" else 4
    nbytes = cfg.T * (len(rows) * (cfg.d * b + 4) + Q * (cfg.d * b + 4 * H))
    hbm, kind = peaks()
    gbs = nbytes / (ms_multi * 1e-3) / 1e9
    print(json.dumps({"metric": "multi-query read (ar_route_fwd_multi), ms per launch",
                      "value": ms_multi, "unit": "ms", "higher_is_better": False,
                      "config": {"workload": f"{cfg.name}-shaped rows", "T": cfg.T, "d": cfg.d,
                                 "r": cfg.r, "H": H, "rows": len(rows), "queries": Q},
                      "single_reads_ms": ms_single,
                      "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                                   "frac": gbs / hbm, "bytes_per_launch": nbytes,
                                   "peak_source": kind}}), flush=True)


def reference_arm(args, rank, world):
    """The oracle as the reference implementation, on the host cores."""
    if rank != 0:
        return
    sys.path.insert(0, ROOT)
    from depth_wise_attention_ar_gb300 import workload
    cfg = config_of(args, workload)
    H = args.heads or cfg.H
    # each of the W + K runs is one token sample, sized so that the whole run
    # stays within a few minutes
    per_run = min(args.cpu_seconds, 150.0 / max(1, args.steps + args.warmup))
    cb, dt, Ts = cpu_baseline(cfg, H, per_run, steps=max(1, args.steps), warmup=args.warmup)
    from oracle import schedule
    oplan = schedule.block_plan(cfg.M, cfg.NB)
    run = list(cfg.sites) if cfg.sites is not None else list(range(len(oplan["sites"])))
    line = {
        "metric": METRIC,
        "value": cb["value"],
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": dt * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded numpy Philox)",
        "config": line_config(cfg, H, world, oplan["sites"], run),
        "tokens_per_step": Ts,
        "impl": "reference",
        "cpu_baseline": cb,
        "e2e": {"value": cb["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
