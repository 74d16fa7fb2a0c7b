"""Benchmark of one MoE dispatch + combine step on one GPU (N replicas under torchrun).

A step is the whole hot path over one batch of synthetic input already resident
in device memory: the dispatch layout (count, scan, slots), the dispatch
scatter (with the fused bf16 -> FP8-e4m3 cast on the DeepSeek-V3-shaped
workload) and the weighted combine. The metric is tokens/s (source tokens of
all logical ranks per second) and the HBM bandwidth each phase achieves.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle, timed on the host

Prints one JSON line (rank 0). Beside the contract keys it carries `phases`
(per-phase time, algorithmic bytes, GB/s and fraction of the measured copy
peak), `roofline` (the dominant kernel, with ncu DRAM traffic when the committed
capture matches the kernel's sources), `graph` (the same step replayed as one
CUDA graph), `fanout_copy` (a sequential one-read, many-write copy of the
dispatch's own bytes, register and bulk methods: a reference stream at the
dispatch's read:write mix), `e2e`
(the step through the ABI from pinned host buffers; `--host-link` times the
same copies alone, its bound) and `cpu_baseline` (the oracle on one host core).
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "dispatch+combine tokens/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
DEFAULT_WORKLOAD = "dsv3_fp8"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300's nominal HBM3e bandwidth: context beside the measured copy peak


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="native", choices=["native", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS))
    p.add_argument("--tokens", type=int, default=0,
                   help="override tokens per rank (small cases for profiling only)")
    p.add_argument("--compact", action="store_true",
                   help="packed receive rows: destinations back to back in R*T*min(K,R) rows")
    p.add_argument("--compact-window", action="store_true",
                   help="compact receive rows inside each destination's R*M-row window")
    p.add_argument("--align", type=int, default=0, help="expert_alignment of the expanded layout")
    p.add_argument("--zero-padding", action="store_true", help="zero the alignment padding rows")
    p.add_argument("--sf-pack", action="store_true",
                   help="packed power-of-two FP8 scales (4 exponent bytes per word)")
    p.add_argument("--copy-path", type=int, default=0, choices=[0, 1, 2],
                   help="unchanged rows: 0 automatic, 1 register copies, 2 bulk copies")
    p.add_argument("--precast", action="store_true",
                   help="x arrives already cast to fp8-e4m3 with its scales (FP8 receive only)")
    p.add_argument("--cached", action="store_true",
                   help="time dispatch + combine only, replaying a layout computed once")
    p.add_argument("--compare-sort", action="store_true",
                   help="time the deterministic dispatch against atomic slots + post-hoc sort")
    p.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay timing")
    p.add_argument("--host-link", action="store_true",
                   help="only time one step's host<->device copies (the end-to-end bound), nothing else")
    p.add_argument("--no-ceiling", action="store_true",
                   help="skip the one-read, many-write reference copy timed at the dispatch's byte counts")
    p.add_argument("--hbm-sweep", action="store_true",
                   help="only measure HBM bandwidth against the read:write mix (fan-out copies, torch copy/fill)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-baseline sample")
    return p.parse_args()


def workload(args):
    wl = W.WORKLOADS[args.workload]
    if args.tokens:
        wl = wl.replace(num_tokens=args.tokens, num_max_tokens_per_rank=max(args.tokens, 1))
    if args.compact:
        wl = wl.replace(compact=2)
    elif args.compact_window:
        wl = wl.replace(compact=1)
    if args.align:
        wl = wl.replace(expert_alignment=args.align)
    if args.zero_padding:
        wl = wl.replace(zero_padding=True)
    if args.sf_pack:
        wl = wl.replace(sf_pack=True)
    if args.precast:
        if wl.recv_dtype != "fp8":
            raise SystemExit("--precast needs a workload with an FP8 receive buffer")
        wl = wl.replace(x_dtype="fp8")
    return wl


def host_cpu() -> str:
    """CPU model and logical core count of this host, for the CPU-baseline line."""
    model = platform.processor() or platform.machine()
    try:
        for line in open("/proc/cpuinfo"):
            key = line.split(":")[0].strip().lower()
            if key in ("model name", "cpu part"):
                val = line.split(":", 1)[1].strip()
                model = val if key == "model name" else f"{platform.machine()}, CPU part {val}"
                break
    except OSError:
        pass
    return f"{model}, {os.cpu_count()} logical cores"


def describe(wl) -> str:
    lay = "expanded per-expert blocks" if wl.expand else (
        f"hybrid row form {wl.n_so}x{wl.n_su}" if wl.n_so > 1 else "direct row form")
    if wl.compact == 1:
        lay += ", compact receive rows (per-destination windows)"
    elif wl.compact == 2:
        lay += ", packed receive rows (destinations back to back)"
    if wl.expand and wl.expert_alignment > 1:
        lay += f", blocks aligned to {wl.expert_alignment}" + (" with zeroed padding" if wl.zero_padding else "")
    cast = {("bf16", "fp8"): "bf16 x cast to fp8-e4m3 inside dispatch (" + (
                "packed power-of-two scale per 128 columns" if wl.sf_pack else "fp32 scale per 128 columns") + ")",
            ("fp8", "fp8"): "pre-cast fp8-e4m3 x + fp32 scales",
            ("bf16", "bf16"): "bf16 rows"}[(wl.x_dtype, wl.recv_dtype)]
    return (f"{wl.name}: {wl.num_ranks} logical ranks x {wl.num_tokens} tokens, {wl.num_experts} experts "
            f"top-{wl.num_topk}, hidden {wl.hidden}, {lay}, {cast}, bf16 combine with fp32 weights, "
            f"routing {wl.routing}")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ---- algorithmic bytes (only what the method must move) ---------------------

def algorithmic_bytes(wl, ntpr, valid_lanes, tokens_with_lane, pad_rows=0):
    """Bytes per launch of each phase. ntpr: total deduplicated rows; valid_lanes:
    lanes with an expert; tokens_with_lane: source tokens with >= 1 valid lane;
    pad_rows: alignment padding rows dispatch zeroes (expanded, zero padding)."""
    R, T, K, H = wl.num_ranks, wl.num_tokens, wl.num_topk, wl.hidden
    G = H // 128
    n_tok = R * T
    eb_in = 1 if wl.x_dtype == "fp8" else 2
    eb_out = 1 if wl.recv_dtype == "fp8" else 2
    hid_rows = valid_lanes if wl.expand else ntpr
    layout = n_tok * K * 8 + n_tok * K * 4 + n_tok * R + 4 * R * (R + wl.num_experts) * 2
    if wl.expand:
        layout += n_tok * K * 4
    SW = ((G + 3) // 4 if wl.sf_pack else G) * 4                  # scale bytes per row
    dispatch = (tokens_with_lane * H * eb_in                       # x read once per routed token
                + (tokens_with_lane * SW if wl.x_dtype == "fp8" else 0)
                + hid_rows * H * eb_out                            # hidden rows written
                + (hid_rows * SW if wl.recv_dtype == "fp8" else 0)
                + pad_rows * (H * eb_out + (SW if wl.recv_dtype == "fp8" else 0))  # zeroed padding
                + ntpr * (K * 8 + K * 4 + (2 + K) * 4)             # sidecar rows
                + n_tok * K * (8 + 4 + 4))                         # topk_idx, weights, slots read
    dispatch_read = (tokens_with_lane * H * eb_in + (tokens_with_lane * SW if wl.x_dtype == "fp8" else 0)
                     + n_tok * K * (8 + 4 + 4))
    combine = (hid_rows * H * 2                                    # each expert-output row once
               + n_tok * H * 2                                     # out written
               + n_tok * K * (8 + 4 + 4))
    return {"layout": layout, "dispatch": dispatch, "combine": combine, "dispatch_read": dispatch_read}


def run_config(wl, args, world, ntpr):
    """The `config` object of the JSON line; both arms print the same one."""
    return {"workload": describe(wl) + (" (cached: layout replayed, not timed)" if args.cached else ""),
            "tokens_per_step": wl.num_ranks * wl.num_tokens, "dedup_rows": ntpr,
            "l2": "inputs larger than L2 between steps (no flush)",
            "copy_path": {0: "automatic", 1: "register copies", 2: "bulk copies"}[args.copy_path],
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def receive_bytes(recv, y, identity):
    """Device bytes of the receive tensors (and of the expert outputs y when they
    are a separate buffer): what the receive layout costs in memory."""
    n = sum(t.numel() * t.element_size() for t in (recv.recv_x, recv.recv_sf, recv.recv_topk_idx,
                                                     recv.recv_topk_weights, recv.recv_src_metadata)
            if t is not None)
    return {"recv_buffer_bytes": n, "recv_x_rows": recv.recv_x.shape[0],
            "expert_output_bytes": 0 if identity else y.numel() * y.element_size()}


# ---- clocks ----------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.25)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---- the native arm ---------------------------------------------------------

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v, device="cuda"):
    """Maximum of a per-rank value over all ranks (the slowest rank's time)."""
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, units_per_rank, total_ms, steps):
    """Units all ranks processed per second, timed by the slowest rank."""
    return world * units_per_rank / (total_ms * 1e-3 / steps)


def native(args):
    import combine_ep_get_02_gb300 as ep

    world, rank, local = dist_setup(args)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = workload(args)
    cfg = ep.config_of(wl, copy_path=args.copy_path)
    R, T, K, H = wl.num_ranks, wl.num_tokens, wl.num_topk, wl.hidden

    # inputs: seeded, generated on the host, then resident in device memory
    idx_h, w_h = W.routing(wl)
    x_h, sf_h = W.hidden(wl)
    idx, w, x = idx_h.to(dev), w_h.to(dev), x_h.to(dev)
    sf = None if sf_h is None else sf_h.to(dev)
    ws = ep.alloc_workspace(cfg, dev)
    lay = ep.alloc_layout(cfg, dev)
    recv = ep.alloc_recv(cfg, dev)
    rows = ep.ep_recv_rows(cfg)
    identity = wl.y_kind == "identity" and wl.recv_dtype == "bf16"
    y = recv.recv_x if identity else W.expert_outputs(wl, rows, device=str(dev))
    out = torch.empty(R, T, H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]

    def step(e=None):
        if e: e[0].record(stream)
        if not args.cached:
            ep.ep_get_dispatch_layout(cfg, idx, lay, ws, stream)
        if e: e[1].record(stream)
        ep.ep_dispatch(cfg, lay, x, sf, idx, w, recv, ws, stream)
        if e: e[2].record(stream)
        ep.ep_combine(cfg, lay, y, idx, w, out, ws, stream)
        if e: e[3].record(stream)

    if args.cached:  # the stored layout every timed step replays
        ep.ep_get_dispatch_layout(cfg, idx, lay, ws, stream)
    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize(dev)
    st = ep.ep_check_error(ws, stream)
    if st != ep.EP_OK:
        raise RuntimeError(f"device status {ep.ep_status_string(st)}")

    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize(dev)
        t_start.record(stream)
        for i in range(args.steps):
            step()
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
    total_ms = t_start.elapsed_time(t_end)
    total_ms = max_over_ranks(world, total_ms)
    ms_per_step = total_ms / args.steps
    # per-phase times: the same steps again, an event between the phases (which
    # also keeps each kernel from being placed while the one before it drains,
    # so every phase carries its launch; launch_floor_us is that cost alone)
    for i in range(args.steps):
        step(ev[i])
    torch.cuda.synchronize(dev)
    phase_ms = {name: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in ev)
                for j, name in enumerate(("layout", "dispatch", "combine"))}
    phase_med = {name: statistics.median(e[j].elapsed_time(e[j + 1]) for e in ev)
                 for j, name in enumerate(("layout", "dispatch", "combine"))}
    floor_us = launch_floor_us(stream, dev, args.steps)
    # each phase alone, replayed from a CUDA graph (no event or host launch between calls)
    replay = {}
    if not args.no_graph:
        if not args.cached:
            replay["layout"] = replay_us(lambda s: ep.ep_get_dispatch_layout(cfg, idx, lay, ws, s), stream, dev, 20)
        replay["dispatch"] = replay_us(lambda s: ep.ep_dispatch(cfg, lay, x, sf, idx, w, recv, ws, s), stream, dev, 10)
        replay["combine"] = replay_us(lambda s: ep.ep_combine(cfg, lay, y, idx, w, out, ws, s), stream, dev, 10)

    # algorithmic bytes from this layout's counts
    ntpr = int(lay.num_tokens_per_rank.sum().item())
    valid = idx_h >= 0
    valid_lanes = int(valid.sum().item())
    tokens_with_lane = int(valid.any(-1).sum().item())
    pad_rows = (int(lay.exp_region[-1].item()) - valid_lanes) if (wl.expand and wl.zero_padding) else 0
    abytes = algorithmic_bytes(wl, ntpr, valid_lanes, tokens_with_lane, pad_rows)
    peak, peak_kind = peaks()
    gbs = {k: abytes[k] / (phase_ms[k] * 1e-3) / 1e9 for k in phase_ms}
    dominant = max(("dispatch", "combine"), key=lambda k: phase_ms[k])
    dominant_kernel = "combine_kernel" if dominant == "combine" else dispatch_kernel_name(wl, args.copy_path)

    ceiling = None
    if not args.no_ceiling:
        ceiling = fanout_reference(ep, wl, abytes["dispatch_read"], abytes["dispatch"] - abytes["dispatch_read"],
                                   gbs["dispatch"], dev, stream, args)
    graph = None
    if not args.no_graph and not args.cached:
        graph = graph_replay(ep, cfg, idx, lay, ws, x, sf, w, recv, y, out, stream, dev, args, world, R * T)

    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(ep, cfg, wl, idx_h, w_h, x_h, sf_h, lay, recv, y, identity, ws, stream, dev,
                         args, world)

    line = {
        "metric": METRIC,
        "value": whole_job_rate(world, R * T, total_ms, args.steps),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("bf16 x -> fp8-e4m3 recv, fp32 combine accumulate"
                  if wl.recv_dtype == "fp8" and wl.x_dtype == "bf16" else
                  f"{wl.x_dtype} x -> {wl.recv_dtype} recv, fp32 combine accumulate"),
        "data": "synthetic (seeded routing and activations)",
        "config": run_config(wl, args, world, ntpr),
        "memory": receive_bytes(recv, y, identity),
        "phases": {
            k: {"us": phase_ms[k] * 1e3, "us_median": phase_med[k] * 1e3, "algorithmic_bytes": abytes[k],
                "gbs": gbs[k], "frac_of_peak": gbs[k] / peak, "frac_of_nominal": gbs[k] / NOMINAL_HBM_GBS}
            for k in ("layout", "dispatch", "combine")},
        "launch_floor_us": floor_us,
        "layout_replay_us": replay.get("layout"),
        "phase_replay": {k: {"us": v, "gbs": abytes[k] / (v * 1e-6) / 1e9, "frac_of_peak": abytes[k] / (v * 1e-6) / 1e9 / peak}
                         for k, v in replay.items()},
        "roofline": {"kernel": dominant_kernel, "bound": "hbm", "achieved": gbs[dominant],
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": gbs[dominant] / peak, "traffic": ncu_traffic(dominant_kernel, wl, R * T),
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": gbs[dominant] / NOMINAL_HBM_GBS},
        "clocks": clocks.summary(),
        "gpu_launches": args.steps * launches_per_step(wl, args.cached),
    }
    if e2e is not None:
        line["e2e"] = e2e
    if graph is not None:
        line["graph"] = graph
    if ceiling is not None:
        line["fanout_copy"] = ceiling
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, idx_h, w_h, x_h, sf_h, y, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def fanout_reference(ep, wl, read_b, write_b, dispatch_gbs, dev, stream, args):
    """Time the diagnostic fan-out copy (each row read once, written to a run of
    consecutive rows) moving the dispatch's read and write bytes, with register
    stores and with bulk copies: a plain one-read, many-write stream at the
    dispatch's read:write mix, reported beside it (not a bound: the dispatch's
    scattered rows can run faster than its sequential runs)."""
    row_bytes = wl.hidden * (1 if wl.x_dtype == "fp8" else 2)
    rows = max(1, round(read_b / row_bytes))
    den = 1024
    num = max(1, round(write_b / max(read_b, 1) * den))
    n_dst = rows * num // den
    gen = torch.Generator(device=dev).manual_seed(1)
    src = torch.randint(0, 256, (rows * row_bytes,), dtype=torch.uint8, device=dev, generator=gen)
    dst = torch.empty(n_dst * row_bytes, dtype=torch.uint8, device=dev)
    moved = rows * row_bytes + n_dst * row_bytes
    res = {"kernel": "fanout_copy", "read_bytes": rows * row_bytes, "write_bytes": n_dst * row_bytes}
    for method, name in ((0, "registers"), (1, "bulk")):
        if method == 1 and row_bytes > 16384:
            continue
        for _ in range(max(args.warmup, 3)):
            ep.ep_diag_copy_fanout(src, dst, rows, row_bytes, num, den, 0, method, stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            ep.ep_diag_copy_fanout(src, dst, rows, row_bytes, num, den, 0, method, stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) * 1e3 / args.steps
        res[name] = {"us": us, "gbs": moved / (us * 1e-6) / 1e9}
    del src, dst
    res["gbs"] = max(v["gbs"] for k, v in res.items() if k in ("registers", "bulk"))
    res["dispatch_over_fanout"] = dispatch_gbs / res["gbs"]
    return res


def graph_replay(ep, cfg, idx, lay, ws, x, sf, w, recv, y, out, stream, dev, args, world, units):
    """The same step captured once as a CUDA graph (its launches with no host work
    between them) and replayed: steps per second without launch gaps."""
    cs = torch.cuda.Stream(dev)
    cs.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cs), torch.cuda.graph(g, stream=cs):
        ep.ep_get_dispatch_layout(cfg, idx, lay, ws, cs)
        ep.ep_dispatch(cfg, lay, x, sf, idx, w, recv, ws, cs)
        ep.ep_combine(cfg, lay, y, idx, w, out, ws, cs)
    for _ in range(max(args.warmup, 1)):
        g.replay()
    torch.cuda.synchronize(dev)
    barrier(world)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(world, a.elapsed_time(b))
    return {"ms_per_step": ms / args.steps, "value": whole_job_rate(world, units, ms, args.steps),
            "unit": "tokens/s"}


def dispatch_kernel_name(wl, copy_path):
    """The dispatch kernel the library runs for this workload: the fused cast and
    small or register-copy inputs take dispatch_kernel, unchanged rows of at
    least 32 MiB (or copy path 2) the bulk-copy kernel."""
    unchanged = not (wl.x_dtype == "bf16" and wl.recv_dtype == "fp8")
    in_bytes = wl.num_ranks * wl.num_tokens * wl.hidden * (1 if wl.x_dtype == "fp8" else 2)
    bulk = unchanged and (copy_path == 2 or (copy_path == 0 and in_bytes >= 32 << 20))
    return "dispatch_bulk_kernel" if bulk else "dispatch_kernel"


def launch_floor_us(stream, dev, steps):
    """Event-bracketed time of an empty launch (a one-element tensor fill): the
    fixed cost inside every per-phase figure. The GPU is first held busy
    (torch.cuda._sleep) while all the launches are queued, so the figure is the
    device's own gap, not the host's launch rate."""
    t = torch.zeros(1, device=dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(5_000_000)  # a few ms of device time
        for a, b in evs:
            a.record(stream)
            t.fill_(1.0)
            b.record(stream)
    torch.cuda.synchronize(dev)
    return statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3


def replay_us(fn, stream, dev, n):
    """n calls of fn(stream) captured in one CUDA graph and replayed: the time per
    call without host launches or events between calls."""
    cs = torch.cuda.Stream(dev)
    cs.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cs), torch.cuda.graph(g, stream=cs):
        for _ in range(n):
            fn(cs)
    g.replay()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(5):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize(dev)
    return a.elapsed_time(b) * 1e3 / (5 * n)


def launches_per_step(wl, cached=False):
    """Kernels of this library one step launches: the layout (one kernel, three
    when expanded), dispatch and combine."""
    layout = 0 if cached else (3 if wl.expand else 1)
    return layout + (2 if wl.num_tokens > 0 else 0)


def end_to_end(ep, cfg, wl, idx_h, w_h, x_h, sf_h, lay, recv, y, identity, ws, stream, dev, args,
               world):
    """The same step through the public API from pinned host buffers: every step
    copies its inputs host->device and its output device->host inside the timed
    region. Copies run on their own streams, double-buffered, so step i+1's
    inputs and step i-1's output move while step i computes."""
    R, T, H = wl.num_ranks, wl.num_tokens, wl.hidden
    hx = x_h.pin_memory()
    hidx = idx_h.pin_memory()
    hw = w_h.pin_memory()
    hsf = None if sf_h is None else sf_h.pin_memory()
    nb = 2
    hout = [torch.empty(R, T, H, dtype=torch.bfloat16).pin_memory() for _ in range(nb)]
    dx = [torch.empty_like(hx, device=dev) for _ in range(nb)]
    didx = [torch.empty_like(hidx, device=dev) for _ in range(nb)]
    dw = [torch.empty_like(hw, device=dev) for _ in range(nb)]
    dsf = [None if hsf is None else torch.empty_like(hsf, device=dev) for _ in range(nb)]
    dout = [torch.empty(R, T, H, dtype=torch.bfloat16, device=dev) for _ in range(nb)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_done = [ev() for _ in range(nb)]
    comp_done = [ev() for _ in range(nb)]
    out_done = [ev() for _ in range(nb)]
    steps = max(40, args.steps)  # a job long enough that pipeline fill and drain stay small

    def run(n):
        for i in range(n):
            b = i % nb
            if i >= nb:
                s_in.wait_event(comp_done[b])      # step i-2 no longer reads buffer b
            with torch.cuda.stream(s_in):
                dx[b].copy_(hx, non_blocking=True)
                didx[b].copy_(hidx, non_blocking=True)
                dw[b].copy_(hw, non_blocking=True)
                if dsf[b] is not None:
                    dsf[b].copy_(hsf, non_blocking=True)
                in_done[b].record(s_in)
            stream.wait_event(in_done[b])
            if i >= nb:
                stream.wait_event(out_done[b])     # step i-2's output has left dout[b]
            ep.ep_get_dispatch_layout(cfg, didx[b], lay, ws, stream)
            ep.ep_dispatch(cfg, lay, dx[b], dsf[b], didx[b], dw[b], recv, ws, stream)
            ep.ep_combine(cfg, lay, recv.recv_x if identity else y, didx[b], dw[b], dout[b], ws, stream)
            comp_done[b].record(stream)
            s_out.wait_event(comp_done[b])
            with torch.cuda.stream(s_out):
                hout[b].copy_(dout[b], non_blocking=True)
                out_done[b].record(s_out)
        stream.wait_stream(s_out)

    run(2)
    torch.cuda.synchronize(dev)
    barrier(world)
    a = torch.cuda.Event(enable_timing=True)
    b_ = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    s_in.wait_stream(stream)
    run(steps)
    b_.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(world, a.elapsed_time(b_)) / steps
    h2d = hx.numel() * hx.element_size() + hidx.numel() * 8 + hw.numel() * 4 + \
        (0 if hsf is None else hsf.numel() * 4)
    d2h = hout[0].numel() * 2

    return {"value": whole_job_rate(world, R * T, ms * steps, steps), "unit": "tokens/s",
            "ms_per_step": ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps,
            "pipeline": "double-buffered host copies on two copy streams, overlapped with the kernels"}


def transfer_only_ms(hx, hidx, hw, hsf, dx, didx, dw, dsf, hout, dout, stream, dev, reps=5,
                     inputs=True, output=True):
    """One step's input copied in and/or its output copied back (at the same
    time when both), with no kernels: the host link's bound on the end-to-end
    step."""
    t_in, t_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def once():
        t_in.wait_stream(stream)
        t_out.wait_stream(stream)
        if inputs:
            with torch.cuda.stream(t_in):
                dx.copy_(hx, non_blocking=True)
                didx.copy_(hidx, non_blocking=True)
                dw.copy_(hw, non_blocking=True)
                if dsf is not None:
                    dsf.copy_(hsf, non_blocking=True)
        if output:
            with torch.cuda.stream(t_out):
                hout.copy_(dout, non_blocking=True)
        stream.wait_stream(t_in)
        stream.wait_stream(t_out)

    once()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        once()
    b.record(stream)
    torch.cuda.synchronize(dev)
    return a.elapsed_time(b) / reps


def host_link(args):
    """The host-link bound of the end-to-end step, in a process that does nothing
    else: one step's inputs in and output back (pinned host buffers), alone and
    at the same time."""
    dev = torch.device("cuda", 0)
    wl = workload(args)
    R, T, H = wl.num_ranks, wl.num_tokens, wl.hidden
    idx_h, w_h = W.routing(wl)
    x_h, sf_h = W.hidden(wl)
    hx, hidx, hw = x_h.pin_memory(), idx_h.pin_memory(), w_h.pin_memory()
    hsf = None if sf_h is None else sf_h.pin_memory()
    dx, didx, dw = (torch.empty_like(t, device=dev) for t in (hx, hidx, hw))
    dsf = None if hsf is None else torch.empty_like(hsf, device=dev)
    hout = torch.empty(R, T, H, dtype=torch.bfloat16).pin_memory()
    dout = torch.zeros(R, T, H, dtype=torch.bfloat16, device=dev)
    st = torch.cuda.current_stream(dev)
    f = lambda i, o: transfer_only_ms(hx, hidx, hw, hsf, dx, didx, dw, dsf, hout, dout, st, dev, inputs=i, output=o)
    h2d = hx.numel() * hx.element_size() + hidx.numel() * 8 + hw.numel() * 4 + (0 if hsf is None else hsf.numel() * 4)
    print(json.dumps({"mode": "host_link", "workload": describe(wl), "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": hout.numel() * 2, "h2d_ms": f(True, False), "d2h_ms": f(False, True),
                      "both_ms": f(True, True), "zero_copy_gbs": zero_copy_rates(dev, st)}), flush=True)


def zero_copy_rates(dev, st, nbytes=1 << 30):
    """The same link driven by kernels instead of copy engines: the fan-out
    diagnostic (1:1, register and bulk methods) reading pinned host memory into
    device memory, writing device memory into pinned host memory, and both at
    once on two streams."""
    import combine_ep_get_02_gb300 as ep
    row = 14336
    rows = nbytes // row
    h_in = torch.empty(rows * row, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(rows * row, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(rows * row, dtype=torch.uint8, device=dev)
    d_out = torch.zeros(rows * row, dtype=torch.uint8, device=dev)
    s0, s1 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn, reps=5):
        fn()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(reps):
            fn()
        b.record(st)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) * 1e-3 / reps

    def both(method):
        s0.wait_stream(st)
        s1.wait_stream(st)
        ep.ep_diag_copy_fanout(h_in, d_in, rows, row, 1, 1, 0, method, s0)
        ep.ep_diag_copy_fanout(d_out, h_out, rows, row, 1, 1, 0, method, s1)
        st.wait_stream(s0)
        st.wait_stream(s1)

    out = {}
    for method, name in ((0, "registers"), (1, "bulk")):
        out[name] = {
            "read_host": rows * row / timed(lambda: ep.ep_diag_copy_fanout(h_in, d_in, rows, row, 1, 1, 0, method, st)) / 1e9,
            "write_host": rows * row / timed(lambda: ep.ep_diag_copy_fanout(d_out, h_out, rows, row, 1, 1, 0, method, st)) / 1e9,
            "both": 2 * rows * row / timed(lambda: both(method)) / 1e9}
    return out


def ncu_traffic(kernel, wl, n_tok):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it was
    taken on the kernel's current sources (its unit and the headers it includes);
    scaled by source tokens when the capture ran a smaller case. None when there
    is no matching capture."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    try:
        from combine_ep_get_02_gb300 import _build
        src = _build.source_hash(kernel)
        for line in open(path):
            f = line.split()
            if len(f) == 6 and f[0] == kernel and f[1] == wl.name and f[5] == src:
                bytes_, tokens = float(f[2]) + float(f[3]), float(f[4])
                return bytes_ * n_tok / tokens
    except Exception:
        return None
    return None


# ---- the CPU oracle (baseline leg and reference arm) --------------------------

def cpu_sample(wl, idx_h, w_h, x_h, sf_h, y_dev, n_tokens, seed=0):
    """Oracle time per source token over a bounded sample: the layout of the whole
    input (its cost spread over all tokens) + dispatch and combine of n_tokens
    tokens drawn with a seeded generator."""
    import oracle
    R, T, K = wl.num_ranks, wl.num_tokens, wl.num_topk
    t0 = time.perf_counter()
    st, olay = oracle.layout(wl, idx_h)
    t_layout = time.perf_counter() - t0
    rng = np.random.default_rng(seed)
    toks = rng.choice(R * T, size=min(n_tokens, R * T), replace=False)
    idx_np = idx_h.numpy().reshape(R * T, K)
    w_np = w_h.numpy().reshape(R * T, K)
    xv = x_h.reshape(R * T, -1)
    xv = xv.view(torch.int16).numpy().view(np.uint16) if xv.dtype == torch.bfloat16 else xv.numpy()
    sfv = None if sf_h is None else sf_h.reshape(R * T, -1).numpy()
    lane_rows = oracle.global_rows(wl, olay, idx_h).reshape(R * T, K)[toks]
    uniq, inv = np.unique(lane_rows[lane_rows >= 0], return_inverse=True)
    compact = np.full(lane_rows.shape, -1, np.int64)
    compact[lane_rows >= 0] = inv
    ys = y_dev.index_select(0, torch.from_numpy(uniq).to(y_dev.device)).cpu()
    ys = ys.view(torch.int16).numpy().view(np.uint16)
    t0 = time.perf_counter()
    for tok in toks:
        s, t = divmod(int(tok), T)
        oracle.dispatch_token(wl, olay, s, t, xv[tok], None if sfv is None else sfv[tok],
                              idx_np[tok], w_np[tok])
    t_disp = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.combine_gathered(compact, ys, w_np[toks])
    t_comb = time.perf_counter() - t0
    per_token = t_layout / (R * T) + (t_disp + t_comb) / len(toks)
    return per_token, len(toks), t_layout, t_disp, t_comb


def cpu_baseline(wl, idx_h, w_h, x_h, sf_h, y_dev, seconds):
    # calibrate the sample so the whole measurement takes about `seconds`
    per, n, *_ = cpu_sample(wl, idx_h, w_h, x_h, sf_h, y_dev, 64, seed=1)
    n = int(max(64, min(wl.num_ranks * wl.num_tokens, seconds / per)))
    per, n, tl, td, tc = cpu_sample(wl, idx_h, w_h, x_h, sf_h, y_dev, n)
    return {"value": 1.0 / per, "unit": "tokens/s", "cores": 1, "kind": "oracle", "host": host_cpu(),
            "sample": (f"full layout of {wl.num_ranks * wl.num_tokens} tokens ({tl:.2f} s) + dispatch "
                       f"and combine of {n} seeded random source tokens ({td:.1f} s + {tc:.1f} s), "
                       f"single-threaded C++ oracle, scaled to tokens/s")}


REF_TOKENS_PER_STEP = 1024


def reference(args):
    """The oracle, as it stands, timed on the host's cores. A step is a bounded
    sample of the workload: the layout of every token plus dispatch and combine
    of REF_TOKENS_PER_STEP seeded random source tokens; `ms_per_step` is the
    measured time of that sampled work, and `value` extrapolates it to the whole
    workload (tokens/s of the full job at the sampled per-token cost)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = workload(args)
    idx_h, w_h = W.routing(wl)
    x_h, sf_h = W.hidden(wl)
    R, T = wl.num_ranks, wl.num_tokens
    import oracle
    st, olay = oracle.layout(wl, idx_h)  # the config's dedup row count (not timed)
    ntpr = int(olay["num_tokens_per_rank"].sum())
    # expert outputs for the sampled tokens: drawn on the host for the rows they read
    gen = torch.Generator().manual_seed(wl.seed * 1_000_003 + 1)

    class _LazyRows:  # y rows on demand: same shape of access as a device buffer
        device = "cpu"

        def index_select(self, dim, ix):
            return torch.randn(ix.numel(), wl.hidden, generator=gen).to(torch.bfloat16)

    n_tok = min(REF_TOKENS_PER_STEP, R * T)
    step_s, per_token = [], []
    for i in range(args.warmup + args.steps):
        per, n, t_layout, t_disp, t_comb = cpu_sample(wl, idx_h, w_h, x_h, sf_h, _LazyRows(), n_tok, seed=i)
        if i >= args.warmup:
            step_s.append(t_layout + t_disp + t_comb)
            per_token.append(per)
    value = 1.0 / statistics.mean(per_token)
    sample = (f"per step: layout of all {R * T} tokens + dispatch and combine of {n_tok} seeded random "
              f"source tokens of {describe(wl)}; ms_per_step is that sampled work's measured time, value "
              f"extrapolates it to all {R * T} tokens; single-threaded C++ oracle")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": statistics.mean(step_s) * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp32 oracle arithmetic", "data": "synthetic (seeded routing and activations)",
            "config": run_config(wl, args, world, ntpr),
            "sampled_tokens_per_step": n_tok,
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "host": host_cpu(), "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def compare_sort(args):
    """PR #753's comparison on one GPU: layout + deterministic dispatch against
    atomic-slot dispatch + post-hoc sort (same rows, same sidecars)."""
    import combine_ep_get_02_gb300 as ep
    dev = torch.device("cuda", 0)
    wl = workload(args)
    cfg = ep.config_of(wl, copy_path=args.copy_path)
    idx_h, w_h = W.routing(wl)
    x_h, sf_h = W.hidden(wl)
    idx, w, x = idx_h.to(dev), w_h.to(dev), x_h.to(dev)
    sf = None if sf_h is None else sf_h.to(dev)
    ws = ep.alloc_workspace(cfg, dev)
    lay = ep.alloc_layout(cfg, dev)
    recv = ep.alloc_recv(cfg, dev, zero=True)
    racy = ep.alloc_recv(cfg, dev, zero=True)
    srt = ep.alloc_recv(cfg, dev, zero=True)
    counters = torch.zeros(wl.num_ranks, wl.num_ranks, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fns, steps):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(fns) + 1)] for _ in range(steps)]
        for _ in range(max(args.warmup, 1)):
            for f in fns:
                f()
        torch.cuda.synchronize(dev)
        for e in evs:
            e[0].record(stream)
            for j, f in enumerate(fns):
                f()
                e[j + 1].record(stream)
        torch.cuda.synchronize(dev)
        return [statistics.mean(e[j].elapsed_time(e[j + 1]) * 1e3 for e in evs) for j in range(len(fns))]

    det = timed([lambda: ep.ep_get_dispatch_layout(cfg, idx, lay, ws, stream),
                 lambda: ep.ep_dispatch(cfg, lay, x, sf, idx, w, recv, ws, stream)], args.steps)
    old = timed([lambda: ep.ep_dispatch_atomic(cfg, x, sf, idx, w, racy, counters, ws, stream),
                 lambda: ep.ep_deterministic_sort(cfg, racy, counters, srt, stream)], args.steps)
    same = all(torch.equal(getattr(recv, f).view(torch.uint8), getattr(srt, f).view(torch.uint8))
               for f in ("recv_x", "recv_topk_idx", "recv_topk_weights", "recv_src_metadata"))
    print(json.dumps({"mode": "sort_comparison", "workload": describe(wl), "steps": args.steps,
                      "deterministic_us": {"layout": det[0], "dispatch": det[1], "total": sum(det)},
                      "atomic_sort_us": {"atomic_dispatch": old[0], "sort": old[1], "total": sum(old)},
                      "speedup": sum(old) / sum(det), "identical_after_sort": same}), flush=True)


def hbm_sweep(args):
    """Device-memory bandwidth against the read share of the traffic, with CUDA
    events: the diagnostic fan-out copy (each row read once and written to a run
    of fan consecutive rows, register and bulk methods) from mostly reads (1:64)
    to mostly writes (64:1), beside torch's 1:1 copy and its fill (writes
    only). About 4 GiB moved per point, rows of 14,336 bytes (a 7168-wide bf16
    token)."""
    import combine_ep_get_02_gb300 as ep
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    st = torch.cuda.current_stream(dev)

    def timed(fn, reps=10):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(reps):
            fn()
        b.record(st)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) * 1e-3 / reps

    gib = 1 << 30
    buf = torch.empty(4 * gib, dtype=torch.uint8, device=dev)
    out = {"mode": "hbm_sweep", "unit": "GB/s",
           "torch_copy_1to1": 4 * gib / timed(lambda: buf[2 * gib:].copy_(buf[:2 * gib])) / 1e9,
           "torch_fill_write_only": 4 * gib / timed(lambda: buf.view(torch.bfloat16).fill_(1.0)) / 1e9,
           "fanout": []}
    del buf
    row = 14336
    for num, den in ((1, 64), (1, 16), (1, 4), (1, 2), (1, 1), (2, 1), (3, 1), (3481, 1024), (4, 1), (8, 1),
                     (16, 1), (64, 1)):
        rows = int(4 * gib / row / (1 + num / den))
        n_dst = rows * num // den
        src = torch.empty(rows * row, dtype=torch.uint8, device=dev).random_()
        dst = torch.empty(max(n_dst, 1) * row, dtype=torch.uint8, device=dev)
        point = {"reads_per_write": f"{den}:{num}", "read_share": rows / (rows + n_dst)}
        for method, name in ((0, "registers"), (1, "bulk")):
            t = timed(lambda: ep.ep_diag_copy_fanout(src, dst, rows, row, num, den, 0, method, st))
            point[name] = (rows + n_dst) * row / t / 1e9
        out["fanout"].append(point)
        del src, dst
        torch.cuda.empty_cache()
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        reference(args)
    elif args.compare_sort:
        compare_sort(args)
    elif args.host_link:
        host_link(args)
    elif args.hbm_sweep:
        hbm_sweep(args)
    else:
        native(args)


if __name__ == "__main__":
    main()
