"""Benchmark of the MoE dispatch/combine hot path on GB300.

One step = one pass of the whole path over the workload resident in HBM:
layout -> notify -> dispatch -> combine (identity experts: combine reads the
dispatch arena), all through the C ABI of libmoe.so on one stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line. ``value`` is tokens/s over all ranks (S tokens per step
per rank); the device-timed kernels give the roofline of the dominant kernel
against the measured HBM copy bandwidth. ``--impl reference`` times the CPU
oracle on a bounded sample of the same workload instead (host cores only).
With N > 1 (torchrun) every rank runs an independent replica on its own GPU
(the path's P ranks are partitions of one GPU's memory) and the time is the
maximum over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "dispatch+combine tokens/s and achieved HBM GB/s (% of ~8 TB/s) on 1 GB300"
UNIT = "tokens/s"
L2_BYTES = 129 * 1000 * 1000  # GB300 L2, used when the device does not report it
FALLBACK_HBM_GBS = 6800.0
CLOCK_FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
KERNEL_SOURCES = ("combine_moe_layout_02_gb300/csrc/dispatch.cu", "combine_moe_layout_02_gb300/csrc/combine.cu",
                  "combine_moe_layout_02_gb300/csrc/moe_device.cuh")


# --------------------------------------------------------------------------
# Algorithmic (minimum) bytes per launch.

def dispatch_bytes(S, P, K, H, R, quant):
    """Read x once, write each received row's payload + metadata, side arrays,
    read topk ids/weights and the send_head row of every token."""
    payload = H if quant else 2 * H
    meta = 16 if quant else 12          # (scale +) triple
    return 2 * S * H + R * (payload + meta) + R * 4 + R * K * 8 + S * K * 8 + S * P * 4


def combine_bytes(S, P, K, H, R):
    """Read every received row once, write out, read send_head and topk."""
    return R * 2 * H + S * 2 * H + S * P * 4 + S * K * 8


def dispatch_expert_bytes(S, K, H, R, quant):
    """Expert-major layout: read x once, write one slot per (token, k) with its
    triple, recv_src_idx and recv_weight; read topk ids, weights, slot rows."""
    payload = H if quant else 2 * H
    meta = 16 if quant else 12
    return 2 * S * H + R * (payload + meta) + R * 8 + S * K * 12


def combine_expert_bytes(S, K, H, R):
    """Expert-major layout: read every slot row once, write out, read topk ids,
    weights and slot rows."""
    return R * 2 * H + S * 2 * H + S * K * 12


# --------------------------------------------------------------------------
# Multi-rank helpers (also exercised on CPU with gloo).

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(elapsed_s: float, units: float, world: int):
    """Max of the ranks' times and sum of their units (no-op for one rank)."""
    if world <= 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# --------------------------------------------------------------------------
# Clocks during the timed region.

class ClockSampler:
    def __init__(self, uuid: str | None, period_ms: int = 50):
        self.uuid = uuid
        self.period_ms = period_ms
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
               f"-lms={self.period_ms}"]
        if self.uuid:
            cmd.insert(1, f"--id={self.uuid}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
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
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 10 and f[2].replace(".", "").isdigit():
                rows.append(f)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i] == "Active"})
        sm = [float(r[2]) for r in rows]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][3]),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[4]) for r in rows if r[4].replace(".", "").isdigit())}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def kernel_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_key(workload: str, T, layout: str):
    """Key of a traffic record: the named workload at its own token count, with
    ":expert" for the expert-major receive layout. None for any other token
    count, which no record covers."""
    from combine_moe_layout_02_gb300 import inputs

    if T is not None and T != inputs.WORKLOADS[workload]["T"]:
        return None
    return workload + (":expert" if layout == "expert" else "")


def recorded_traffic(key, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, when it was taken
    on the kernels as they are now."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if key is None or not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_hash") != kernel_hash():
        return None
    return d.get("per_launch_bytes", {}).get(key, {}).get(kernel)


# --------------------------------------------------------------------------
# CPU oracle on a bounded sample (reference arm and cpu_baseline).

def int8_stand_in(w, layout: str):
    """bf16 rows standing in for the expert outputs an int8 combine reads: one
    seeded N(0,1) row per received row of the workload (the path makes no bf16
    rows for int8 slots; the GPU arm uses such an arena too)."""
    import numpy as np

    import oracle
    from combine_moe_layout_02_gb300 import inputs

    lay = oracle.layout(w.P, w.E, w.topk_idx)
    nt = oracle.notify(w.P, w.E, w.C, w.expert_alignment, lay["num_tokens_per_rank"],
                       lay["num_tokens_per_expert"], lay["is_token_in_rank"])
    if layout == "expert":
        ex = oracle.notify_expert(w.P, w.E, w.topk_idx, nt["num_recv_tokens_per_expert"],
                                  nt["recv_expert_offset"])
        rows = int(ex["expert_part_base"][-1])
    else:
        rows = int(nt["part_row_base"][-1])
    return inputs.draw_hidden(max(rows, 1), w.H, np.random.default_rng(1))


def oracle_sample(name: str, T_sample: int, min_seconds: float, max_passes: int = 1000,
                  workload=None, layout: str = "rank", y_int8=None):
    """Time the oracle's full path on a bounded sample of the workload: the same
    shape with T_sample tokens per rank. Returns tokens/s, passes, seconds and
    a description of the sample."""
    import oracle
    from combine_moe_layout_02_gb300 import inputs

    w = workload if workload is not None else inputs.workload(name, T=T_sample)
    expert = layout == "expert"

    def front():
        lay = oracle.layout(w.P, w.E, w.topk_idx)
        nt = oracle.notify(w.P, w.E, w.C, w.expert_alignment, lay["num_tokens_per_rank"],
                           lay["num_tokens_per_expert"], lay["is_token_in_rank"])
        ex = (oracle.notify_expert(w.P, w.E, w.topk_idx, nt["num_recv_tokens_per_expert"],
                                   nt["recv_expert_offset"]) if expert else None)
        return nt, ex

    # int8 slots: combine reads bf16 expert outputs (int8_stand_in), drawn
    # outside the timed passes when the caller has not drawn them already.
    if w.quant and y_int8 is None:
        y_int8 = int8_stand_in(w, layout)
    passes, t_total = 0, 0.0
    while passes < max_passes and (passes == 0 or t_total < min_seconds):
        t0 = time.perf_counter()
        nt, ex = front()
        if expert:
            rows = int(ex["expert_part_base"][-1])
            dis = oracle.dispatch_expert(w.P, w.E, w.H, w.quant, w.x_bits, w.topk_idx, w.topk_weights,
                                         ex["slot_row"], ex["expert_part_base"], rows)
        else:
            rows = int(nt["part_row_base"][-1])
            dis = oracle.dispatch(w.P, w.E, w.H, w.quant, w.x_bits, w.topk_idx, w.topk_weights,
                                  nt["send_head"], nt["part_row_base"], rows)
        y, y_stride = (y_int8, 2 * w.H) if w.quant else (dis["arena"], oracle.slot_stride(w.H, 0))
        if expert:
            oracle.combine_expert(w.P, w.E, w.H, y, y_stride, ex["expert_part_base"], rows, ex["slot_row"],
                                  w.topk_idx, w.topk_weights)
        else:
            oracle.combine(w.P, w.E, w.H, y, y_stride, nt["part_row_base"], rows, nt["send_head"], w.topk_idx,
                           w.topk_weights)
        t_total += time.perf_counter() - t0
        passes += 1
    sample = (f"{name} ({layout} layout) with T={w.T} tokens per rank (S={w.S}, {passes} pass(es)); "
              "single-threaded oracle: layout+notify+dispatch+combine")
    oracle_sample.last = dict(S=w.S, P=w.P, K=w.K, H=w.H, quant=w.quant, rows=rows, layout=layout)
    return w.S * passes / t_total, passes, t_total, sample


def oracle_gbs(tokens_per_s):
    """Algorithmic GB/s of the last oracle sample (the bench's byte formulas)."""
    m = getattr(oracle_sample, "last", None)
    if not m:
        return None
    if m["layout"] == "expert":
        b = (dispatch_expert_bytes(m["S"], m["K"], m["H"], m["rows"], m["quant"])
             + combine_expert_bytes(m["S"], m["K"], m["H"], m["rows"]))
    else:
        b = (dispatch_bytes(m["S"], m["P"], m["K"], m["H"], m["rows"], m["quant"])
             + combine_bytes(m["S"], m["P"], m["K"], m["H"], m["rows"]))
    return b / m["S"] * tokens_per_s / 1e9


def host_info():
    """Cores and CPU model of the machine the oracle runs on."""
    info = {"nproc": os.cpu_count(), "machine": platform.machine()}
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                info["cpu"] = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    return info


def reference_tokens(args, budget_s: float = 120.0) -> int:
    """Tokens per rank of the oracle arm's sample: the workload's own T when
    the whole --warmup + --steps run fits the time budget on this host, else
    the largest T that does (speed taken from one calibration pass)."""
    from combine_moe_layout_02_gb300 import inputs

    if args.ref_tokens:
        return args.ref_tokens
    full_T = inputs.WORKLOADS[args.workload]["T"]
    T_cal = min(full_T, 64)
    tps, _, _, _ = oracle_sample(args.workload, T_cal, 0.0, max_passes=1, layout=args.layout)
    per_step = budget_s / (args.steps + args.warmup)
    P = inputs.WORKLOADS[args.workload]["P"]
    T = int(tps * per_step / P)
    return max(1, min(full_T, T))


def run_reference(args, world, rank):
    if rank != 0:
        return
    from combine_moe_layout_02_gb300 import inputs

    T_ref = reference_tokens(args)
    w = inputs.workload(args.workload, T=T_ref)
    y_int8 = int8_stand_in(w, args.layout) if w.quant else None  # drawn once, untimed
    for _ in range(args.warmup):
        oracle_sample(args.workload, T_ref, 0.0, max_passes=1, workload=w, layout=args.layout, y_int8=y_int8)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _, _, _, sample = oracle_sample(args.workload, T_ref, 0.0, max_passes=1, workload=w,
                                        layout=args.layout, y_int8=y_int8)
    elapsed = time.perf_counter() - t0
    value = w.S * args.steps / elapsed
    sample = sample.replace("1 pass(es)", f"{args.steps} timed steps of 1 pass")
    full = inputs.WORKLOADS[args.workload]["T"]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * elapsed / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": path_dtype(w.quant),
        "data": "synthetic",
        # The config of what was timed: the workload at T_ref tokens per rank
        # (the full workload when the run fits the time budget).
        "config": dict(workload_config(args.workload, T_ref), layout=args.layout,
                       fused=bool(args.fused), graph=bool(args.graph),
                       sample=("full workload" if T_ref == full else
                               f"T={T_ref} of the workload's {full} tokens per rank (time budget)")),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample, "GB_s": oracle_gbs(value), "host": host_info()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def path_dtype(quant: int) -> str:
    """What the path moves and computes in: bf16 rows (fp32 accumulation in
    combine), or int8 rows quantised in fp32 from bf16 with an fp32 scale."""
    return "int8" if quant else "bf16"


def workload_config(name, T=None):
    from combine_moe_layout_02_gb300 import inputs

    c = dict(inputs.WORKLOADS[name])
    if T is not None:
        c["T"] = T
    return {"workload": name, "P": c["P"], "E": c["E"], "S": c["P"] * c["T"], "H": c["H"],
            "K": c["K"], "routing": c["routing"], "quant": c["quant"],
            "num_channels": inputs.NUM_CHANNELS}


# --------------------------------------------------------------------------
# Our arm.

def host_link_ceiling(dev, x_host, idx_host, wts_host, out_host, out, reps: int = 5):
    """The host link's sustained rate for the step's copies alone: the inputs
    host->device (x, topk_idx, topk_weights from pinned memory), the output
    device->host, and both at once on two streams. Each timing repeats the
    copies until at least 256 MB have moved in each direction (a small step's
    copies alone are latency-bound); best of `reps`, wall clock with a device
    synchronisation on both sides; GB/s."""
    import torch

    dx, di, dw = torch.empty_like(x_host, device=dev), torch.empty_like(idx_host, device=dev), \
        torch.empty_like(wts_host, device=dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    b_in = x_host.numel() * 2 + idx_host.numel() * 4 + wts_host.numel() * 4
    b_out = out_host.numel() * 2
    n_in = max(1, -(-(256 << 20) // b_in))
    n_out = max(1, -(-(256 << 20) // b_out))

    def copy_in():
        with torch.cuda.stream(s_in):
            for _ in range(n_in):
                dx.copy_(x_host, non_blocking=True)
                di.copy_(idx_host, non_blocking=True)
                dw.copy_(wts_host, non_blocking=True)

    def copy_out():
        with torch.cuda.stream(s_out):
            for _ in range(n_out):
                out_host.copy_(out, non_blocking=True)

    def best(fn):
        t = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize(dev)
            t = min(t, time.perf_counter() - t0)
        return t

    t_in, t_out = best(copy_in), best(copy_out)
    t_both = best(lambda: (copy_in(), copy_out()))
    del dx, di, dw
    return {"h2d_gbs": n_in * b_in / t_in / 1e9, "d2h_gbs": n_out * b_out / t_out / 1e9,
            "concurrent_gbs": (n_in * b_in + n_out * b_out) / t_both / 1e9,
            "method": "the step's pinned copies repeated to >= 256 MB per direction, alone and on two "
                      "streams at once, best of 5, wall clock"}


def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    from combine_moe_layout_02_gb300 import inputs, moe

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = inputs.workload(args.workload, T=args.tokens_per_rank)
    shape = moe.make_shape(w.P, w.E, w.S, w.K, w.H, w.C, w.expert_alignment, w.quant)
    buf = moe.Buffers(shape, dev, side_arrays=args.layout == "rank",
                      arena_rows=1 if args.layout == "expert" else None)
    x_host = torch.from_numpy(w.x_bits.view(np.int16)).pin_memory()
    idx_host = torch.from_numpy(w.topk_idx).pin_memory()
    wts_host = torch.from_numpy(w.topk_weights).pin_memory()
    x = x_host.to(dev)
    idx = idx_host.to(dev)
    wts = wts_host.to(dev)
    out = torch.empty((w.S, w.H), dtype=torch.int16, device=dev)
    out_host = torch.empty((w.S, w.H), dtype=torch.int16).pin_memory()
    stream = torch.cuda.current_stream(dev)

    expert = args.layout == "expert"
    if expert:
        buf._expert_buffers()
    # int8 slots: combine reads bf16 expert outputs. The expert stage is not
    # part of the path, so one bf16 output arena (random rows, seeded) is
    # made once here and every step's combine reads it.
    y_out, y_stride = None, None
    if w.quant:
        # moe_run_host's arena (either layout) bounds the rows combine may read
        rows_alloc = max(moe.moe_max_recv_rows(shape), moe.moe_max_expert_rows(shape))
        gen = torch.Generator(device=dev).manual_seed(0)
        y_out = torch.empty((max(rows_alloc, 1), w.H), dtype=torch.bfloat16, device=dev)
        y_out.normal_(generator=gen)
        y_out = y_out.view(torch.int16)
        y_stride = 2 * w.H

    fused = args.fused

    def step(ev=None, st=None):
        st = stream if st is None else st
        if ev is not None:
            ev[0].record(st)
        if fused:
            # layout + notify + dispatch in one launch: timed as "dispatch"
            if ev is not None:
                ev[1].record(st)
            buf.dispatch_fused(x, idx, wts, st)
        else:
            buf.layout(idx, st)
            buf.notify(st)
            if expert:
                buf.notify_expert(idx, st)
            if ev is not None:
                ev[1].record(st)
            if expert:
                buf.dispatch_expert(x, idx, wts, st)
            else:
                buf.dispatch(x, idx, wts, st)
        if ev is not None:
            ev[2].record(st)
        if expert:
            buf.combine_expert(out, idx, wts, y=y_out, y_row_stride=y_stride, stream=st)
        else:
            buf.combine(out, idx, wts, y=y_out, y_row_stride=y_stride, stream=st)
        if ev is not None:
            ev[3].record(st)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if int(buf.err[0].item()) != 0:
        raise RuntimeError(f"device error {moe.status_string(int(buf.err[0].item()))}")
    R = int((buf.expert_part_base if expert else buf.part_row_base)[-1].item())

    # Working sets below twice the L2 would be served from L2 across steps:
    # then a buffer of twice the L2 is READ before every timed step, outside
    # that step's events. Reading (a sum over it) leaves L2 holding that
    # buffer's clean lines, so the step neither finds its data in L2 nor pays
    # for writing back the flush's own dirty lines.
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or L2_BYTES)
    footprint = 2 * x.numel() + R * buf.stride + 2 * out.numel() + (2 * y_out.numel() if y_out is not None else 0)
    flush_buf = torch.ones(2 * l2 // 8, dtype=torch.int64, device=dev) if footprint < 2 * l2 else None
    flush_sink = torch.zeros(1, dtype=torch.int64, device=dev)

    def flush():
        torch.sum(flush_buf, dim=0, keepdim=True, out=flush_sink)

    def run_steps(n, fn):
        """Device seconds of n calls of fn (summed per call when flushing)."""
        if flush_buf is None:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(n):
                fn()
            b.record(stream)
            torch.cuda.synchronize(dev)
            return a.elapsed_time(b) / 1e3
        pairs = []
        for i in range(n):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            pairs.append((a, b))
        torch.cuda.synchronize(dev)
        return sum(a.elapsed_time(b) for a, b in pairs) / 1e3

    # --- device-timed region: whole steps --------------------------------
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        if not uuid.startswith("GPU-"):
            uuid = "GPU-" + uuid
    except Exception:
        uuid = None
    timed_step = step
    if args.graph:
        # One step captured as a CUDA graph, replayed in the timed region: the
        # launches of a small step cost more host time than its kernels.
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(graph, stream=cap):
            step(st=torch.cuda.current_stream(dev))
        stream.wait_stream(cap)
        graph.replay()
        torch.cuda.synchronize(dev)
        if int(buf.err[0].item()) != 0:
            raise RuntimeError(f"device error {moe.status_string(int(buf.err[0].item()))}")
        timed_step = graph.replay
    with ClockSampler(uuid) as clocks:
        barrier(world)
        torch.cuda.synchronize(dev)
        elapsed_s = run_steps(args.steps, timed_step)
        barrier(world)
    clk = clocks.summary()
    max_s, units = aggregate(elapsed_s, float(w.S * args.steps), world)
    value = units / max_s

    # --- per-kernel timing (same stream, events between the calls) --------
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    for i, e in enumerate(evs):
        if flush_buf is not None:
            flush()
        step(e)
    torch.cuda.synchronize(dev)
    t_front_ev = statistics.mean(e[0].elapsed_time(e[1]) for e in evs) / 1e3
    t_disp = statistics.mean(e[1].elapsed_time(e[2]) for e in evs) / 1e3
    t_comb = statistics.mean(e[2].elapsed_time(e[3]) for e in evs) / 1e3
    med = [statistics.median(e[a].elapsed_time(e[a + 1]) for e in evs) * 1e3 for a in range(3)]

    # --- what layout + notify cost inside a step --------------------------
    # An event recorded between two kernels ends the programmatic overlap of
    # the second with the first, so the bracketed time above also holds the
    # launch gaps the events create. The cost a step pays is the difference
    # between whole steps and steps without layout and notify (dispatch and
    # combine reuse the handle of the last notify), timed the same way.
    def step_without_front(st=None):
        st = stream if st is None else st
        if fused:
            buf.dispatch_fused(x, idx, wts, st)
        elif expert:
            buf.dispatch_expert(x, idx, wts, st)
        else:
            buf.dispatch(x, idx, wts, st)
        if expert:
            buf.combine_expert(out, idx, wts, y=y_out, y_row_stride=y_stride, stream=st)
        else:
            buf.combine(out, idx, wts, y=y_out, y_row_stride=y_stride, stream=st)

    n_front = max(args.steps, 20)
    t_whole = run_steps(n_front, step)
    t_rest = run_steps(n_front, step_without_front)
    t_front = max(0.0, (t_whole - t_rest) / n_front)
    peak, peak_kind = measured_peaks()
    if expert:
        db = dispatch_expert_bytes(w.S, w.K, w.H, R, w.quant)
        cb = combine_expert_bytes(w.S, w.K, w.H, R)
    else:
        db = dispatch_bytes(w.S, w.P, w.K, w.H, R, w.quant)
        cb = combine_bytes(w.S, w.P, w.K, w.H, R)
    disp_gbs = db / t_disp / 1e9
    comb_gbs = cb / t_comb / 1e9
    dominant = "dispatch" if t_disp >= t_comb else "combine"
    ach = disp_gbs if dominant == "dispatch" else comb_gbs
    if dominant == "combine":
        kname = "combine_kernel"
    elif fused:
        kname = "fused_kernel"  # layout + notify + dispatch in one launch
    else:
        kname = "dispatch_int8_kernel" if w.quant else "dispatch_bf16_kernel"

    # --- end to end through the public API with host buffers -------------
    h2d = x_host.numel() * 2 + idx_host.numel() * 4 + wts_host.numel() * 4
    d2h = out_host.numel() * 2
    e2e_steps = max(6, min(args.steps, 40))
    # The serving call: moe_run_host streams the batches from pinned host
    # memory through the path, overlapping the copies of neighbouring batches
    # with compute (wall clock around the blocking call).
    e2e_method = "moe_run_host: pinned host batches, 3-stream copy/compute overlap, wall clock"
    ws_bytes = moe.moe_run_host_workspace_bytes(shape, e2e_steps)
    workspace = torch.empty((ws_bytes,), dtype=torch.uint8, device=dev)
    hx, hi, hw, ho = [x_host] * e2e_steps, [idx_host] * e2e_steps, [wts_host] * e2e_steps, [out_host] * e2e_steps
    run_kw = dict(y=y_out, y_row_stride=y_stride or 0, fused=fused, expert=expert)
    moe.moe_run_host(shape, hx[:2], hi[:2], hw[:2], ho[:2], workspace, **run_kw)  # warm-up
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    moe.moe_run_host(shape, hx, hi, hw, ho, workspace, **run_kw)
    e_elapsed = time.perf_counter() - t0
    barrier(world)
    del workspace
    e_max, e_units = aggregate(e_elapsed, float(w.S * e2e_steps), world)
    if int(buf.err[0].item()) != 0:
        raise RuntimeError(f"device error {moe.status_string(int(buf.err[0].item()))}")
    link = host_link_ceiling(dev, x_host, idx_host, wts_host, out_host, out)
    link["e2e_gbs"] = (h2d + d2h) * e2e_steps / e_max / 1e9
    link["e2e_frac_of_concurrent"] = link["e2e_gbs"] / link["concurrent_gbs"]

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, passes, secs, sample = oracle_sample(args.workload, args.cpu_tokens, args.cpu_seconds,
                                                  layout=args.layout)
        cpu = {"value": tps, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
               "GB_s": oracle_gbs(tps), "host": host_info()}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * max_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": path_dtype(w.quant), "data": "synthetic",
        "config": dict(workload_config(args.workload, args.tokens_per_rank), layout=args.layout,
                       fused=bool(args.fused), graph=bool(args.graph),
                       l2=("no flush: working set (x, receive arena, out) of "
                           f"{footprint / 1e6:.0f} MB is larger than twice the {l2 / 1e6:.0f} MB L2"
                           if flush_buf is None else
                           f"flushed: a {2 * l2 / 1e6:.0f} MB buffer is read before every timed step, "
                           f"outside its events (working set {footprint / 1e6:.0f} MB)")),
        # per step: layout (+ its error fold), notify, [notify_expert: 2,] dispatch, combine;
        # the fused path: prep + fused launch, combine
        "gpu_launches": (3 if args.fused else (7 if expert else 5)) * args.steps,
        "roofline": {"bound": "hbm", "kernel": kname, "achieved": ach, "peak": peak, "unit": "GB/s",
                     "frac": ach / peak, "peak_source": f"{peak_kind} copy bandwidth (hbm_gbs)",
                     "traffic": recorded_traffic(traffic_key(args.workload, args.tokens_per_rank, args.layout),
                                                 kname),
                     "algorithmic_bytes": db if dominant == "dispatch" else cb},
        "stages": {
            "layout_notify_us": 1e6 * t_front,
            "layout_notify_method": ("whole steps minus steps without layout and notify (the cost inside a "
                                     "step); layout_notify_event_us brackets the two calls with events"),
            "layout_notify_event_us": 1e6 * t_front_ev,
            "dispatch": {"us": 1e6 * t_disp, "GB_s": disp_gbs, "frac_of_peak": disp_gbs / peak,
                         "frac_of_8TBs": disp_gbs / 8000.0, "tokens_per_s": w.S / t_disp,
                         "bytes": db},
            "combine": {"us": 1e6 * t_comb, "GB_s": comb_gbs, "frac_of_peak": comb_gbs / peak,
                        "frac_of_8TBs": comb_gbs / 8000.0, "tokens_per_s": w.S / t_comb,
                        "bytes": cb},
            "recv_rows": R,
            "median_us": {"layout_notify": med[0], "dispatch": med[1], "combine": med[2]},
        },
        "clocks": clk,
        "e2e": {"value": e_units / e_max, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps, "method": e2e_method,
                "host_link": link},
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    from combine_moe_layout_02_gb300 import inputs

    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=inputs.BENCH_WORKLOAD, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--layout", choices=["rank", "expert"], default="rank",
                    help="receive layout: one row per (token, rank), or one per (token, k) grouped by expert")
    ap.add_argument("--graph", action="store_true",
                    help="capture one step as a CUDA graph and replay it in the timed region")
    ap.add_argument("--fused", action="store_true",
                    help="layout + notify + dispatch as one cooperative launch (small shapes)")
    ap.add_argument("--tokens-per-rank", type=int, default=None,
                    help="override T (a smaller case of the same workload, e.g. for profiling)")
    ap.add_argument("--ref-tokens", type=int, default=None,
                    help="tokens per rank of the oracle arm's sample (default: the workload's own T when the "
                         "run fits about two minutes, else the largest T that does)")
    ap.add_argument("--cpu-tokens", type=int, default=512,
                    help="tokens per rank of the GPU arm's cpu_baseline sample")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        if args.impl == "reference":
            if rank != 0:
                return
        else:
            import torch

            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
    try:
        if args.impl == "reference":
            run_reference(args, 1 if world > 1 else world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1 and args.impl != "reference":
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
