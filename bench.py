"""Throughput of exact attention forward + backward on GB300.

One step = fa_forward + fa_backward (its two launches after the forward: the
preprocess and the gradient kernel) over one batch of the Llama-shaped causal
workload B=2, H=32, n=m=4096, d=128 (bf16 inputs, seeded N(0,1)), i.e. the whole
hot path. The metric is fwd+bwd TFLOP/s counting 4*B*H*n*m*d per forward (halved
under causal masking) and 2.5x that per backward. `value` times the steps with
the inputs already on the device, replaying the step from a CUDA graph (--eager
launches it from the host instead); `e2e` times the same step through the C-ABI
host-buffer calls fa_session_submit / fa_session_sync (inputs copied in from
pinned host memory and every output copied back, each step, inside the timed
region).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own batch (independent heads, no
collective on the data path: weak scaling); the timed region is bracketed by
barriers and the max time over ranks is reported. Rank 0 prints one JSON line.

--impl reference times the fp64 CPU oracle (tests' ground truth, not a
product path) on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from exact_io_aware_27_gb300 import inputs as wl  # noqa: E402

METRIC = "attention fwd+bwd TFLOP/s (bf16, causal) and % of GB300 dense BF16 peak"
UNIT = "TFLOP/s"
WORKLOAD = wl.LLAMA_B2_H32_N4096_D128
L2_BYTES = 129 * 1024 * 1024


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_seed(w, rank: int) -> int:
    """Seed of rank `rank`'s batch: every rank draws its own independent heads."""
    return w.seed + 17 * rank


def max_over_ranks(x: float, device=None) -> float:
    """The maximum of `x` over all ranks (identity without a process group)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_value(flops_per_rank_step: float, world: int, ms_per_step: float) -> float:
    """Whole-job TFLOP/s: every rank's FLOPs over the slowest rank's time."""
    return flops_per_rank_step * world / (ms_per_step * 1e-3) / 1e12


def _traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu capture, or None
    if there is none or the kernel's sources changed since it was taken."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            entry = json.load(f)[kernel]
        digest = hashlib.sha256()
        for rel in entry["files"]:
            with open(os.path.join(ROOT, rel), "rb") as f:
                digest.update(f.read())
        return entry["bytes"] if digest.hexdigest()[:16] == entry["source_sha256"] else None
    except (OSError, KeyError, ValueError):
        return None


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        sus_mhz = (p.get("clocks_under_load") or {}).get("sm_mhz_median")
        return {"bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "sustained_sm_mhz": float(sus_mhz) if sus_mhz else None,
                "sm_max_mhz": float(p.get("sm_max_mhz", 2070.0)),
                "hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sustained_sm_mhz": None,
                "sm_max_mhz": 2070.0, "hbm_gbs": 6800.0, "source": "fallback"}


def tensor_peak(peaks, clk):
    """The bf16 dense peak that matches the clock the timed region ran at.

    The burst figure was measured at the maximum SM clock, the sustained one
    under the power cap at a lower clock. A run whose sampled median SM clock is
    within 3 % of the maximum is divided by the burst peak; one at (or within
    5 % of) the power-capped clock of the sustained measurement by the sustained
    peak; one in between by the burst peak scaled by median / maximum clock.
    Without clock samples the burst peak is used. Returns (peak, description).
    """
    burst, sus = peaks["bf16_tflops"], peaks["bf16_tflops_sustained"]
    src = peaks["source"]
    mhz = clk.get("sm_mhz") if clk else None
    mx = (clk.get("sm_max_mhz") if clk else None) or peaks["sm_max_mhz"]
    if not mhz or not mx:
        return burst, f"bf16 dense, burst ({src}; no clock samples)"
    if mhz >= 0.97 * mx:
        return burst, f"bf16 dense, burst ({src}; SM clock {mhz:.0f} of {mx:.0f} MHz)"
    cap = peaks.get("sustained_sm_mhz")
    if cap and mhz <= 1.05 * cap:
        return sus, f"bf16 dense, sustained ({src}; SM clock {mhz:.0f} MHz, power-capped level {cap:.0f})"
    scaled = max(sus, burst * mhz / mx)
    return scaled, f"bf16 dense, burst x {mhz:.0f}/{mx:.0f} MHz ({src})"


def visible_pairs(n: int, m: int, causal: bool) -> int:
    """(query, key) pairs with a visible score in one head: one exp each in the
    forward. Top-left causal: query q sees keys 0..min(q, m - 1)."""
    if not causal:
        return n * m
    full = min(n, m)  # queries q < m see q + 1 keys
    return full * (full + 1) // 2 + max(0, n - m) * m


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: torch.device):
        self.proc = None
        self.error = None
        target = str(device.index or 0)
        try:
            uuid = torch.cuda.get_device_properties(device).uuid
            target = "GPU-" + str(uuid)
        except Exception:
            pass
        self.target = target

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.target, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception as e:  # no nvidia-smi
            self.error = str(e)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "note": f"nvidia-smi unavailable: {self.error}"}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power = [], [], []
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "no samples"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


def _cpu_baseline(workload, heads: int):
    """The oracle, as it stands, on `heads` full heads of the workload (rank 0)."""
    import oracle
    orc = oracle.default()
    Q, K, V, dO = wl.workload_inputs(workload)
    flat = [t.reshape(workload.heads, -1, workload.d) for t in (Q, K, V, dO)]
    t0 = time.perf_counter()
    for h in range(heads):
        q, k, v, do = (t[h].double().numpy() for t in flat)
        orc.forward(q, k, v, workload.causal)
        orc.backward(q, k, v, do, workload.causal)
    dt = time.perf_counter() - t0
    flops = (workload.flops_fwd() + workload.flops_bwd()) * heads / workload.heads
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": orc.num_threads(),
            "kind": "oracle",
            "sample": f"{heads} of {workload.heads} heads ({workload.describe()}), full fp64 "
                      f"forward + backward, {dt:.1f} s"}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    import oracle
    orc = oracle.default()
    w = wl.WORKLOADS[getattr(args, "workload", WORKLOAD.name)]  # the arm's own workload
    Q, K, V, dO = wl.workload_inputs(w)
    flat = [t.reshape(w.heads, -1, w.d) for t in (Q, K, V, dO)]
    # Each step: forward + backward of sampled query / key rows of one head,
    # sized so that warm-up + timed steps stay within about two minutes.
    per_step = max(0.05, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    rows = w.n
    heads_cycle = wl.sample_indices(w.heads, w.heads, 5003)

    def step(i, r):
        h = heads_cycle[i % len(heads_cycle)]
        q, k, v, do = (t[h].double().numpy() for t in flat)
        if r >= w.n:
            orc.forward(q, k, v, w.causal)
            orc.backward(q, k, v, do, w.causal)
        else:
            idx = wl.sample_indices(w.n, r, 6000 + i)
            orc.forward_rows(q, k, v, idx, w.causal)
            orc.backward_rows(q, k, v, do, idx, idx, w.causal)

    # calibrate the sample size on the first warm-up step
    t0 = time.perf_counter()
    step(0, rows)
    t_full = time.perf_counter() - t0
    if t_full > per_step:
        rows = max(32, int(w.n * per_step / t_full))
    for i in range(1, args.warmup):
        step(i, rows)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i, rows)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    flops = (w.flops_fwd() + w.flops_bwd()) / w.heads * rows / w.n
    value = flops / dt / 1e12
    sample = (f"one head per step, {rows} of {w.n} query rows (and as many key rows) sampled, "
              f"fp64 oracle forward + backward; flops counted as that share of the head")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "shape": w.describe()},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": orc.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import exact_io_aware_27_gb300 as fa

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = wl.WORKLOADS[args.workload]
    B, H, n, m, d = w.B, w.H, w.n, w.m, w.d
    Q, K, V, dO = wl.attention_inputs(B, H, n, m, d, rank_seed(w, rank), w.qk_std)
    q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
    O = torch.empty_like(q)
    L = torch.empty((B, H, n), dtype=torch.float32, device=dev)
    dQ, dK, dV = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = fa.alloc_workspace(B, H, n, m, d, dev)
    stream = torch.cuda.current_stream(dev)

    # --l2-flush: a buffer larger than L2 is overwritten before every timed step, so
    # each step starts with cold caches; the step time is then the sum of the three
    # kernels' event times (the flush itself is not counted).
    flush_buf = (torch.empty(512 << 20, dtype=torch.uint8, device=dev)
                 if args.l2_flush else None)

    def step(ev=None):
        if flush_buf is not None:
            flush_buf.fill_(1)
        if ev is not None:
            ev[0].record(stream)
        fa.fa_forward(q, k, v, w.causal, O=O, L=L)
        if ev is not None:
            ev[1].record(stream)
        fa.fa_backward_preprocess(O, do, L, ws)
        if ev is not None:
            ev[2].record(stream)
        fa.fa_backward_grads(q, k, v, do, ws, causal=w.causal, dQ=dQ, dK=dK, dV=dV)
        if ev is not None:
            ev[3].record(stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if fa.fa_get_device_status() != 0:
        raise RuntimeError("device barrier timeout during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    graph = None
    if not args.eager:
        # The timed steps replay the step captured once in a CUDA graph (no host
        # launch overhead between kernels; every kernel still runs every step). The
        # per-kernel split comes from eager steps timed here with events.
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            step()
        stream.wait_stream(cap)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        graph.replay()
        torch.cuda.synchronize(dev)
        for i in range(min(args.steps, 100)):  # enough for the split, short of the power cap
            step(evs[i])
        torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev)
    clocks.start()
    time.sleep(0.2)
    barrier()
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    timed = evs if graph is None else evs[:min(args.steps, 100)]
    stage = [0.0] * 3
    for e in timed:
        for j in range(3):
            stage[j] += e[j].elapsed_time(e[j + 1])
    stage = [s / len(timed) for s in stage]
    elapsed_ms = max_over_ranks(elapsed_ms, dev)
    if fa.fa_get_device_status() != 0:
        raise RuntimeError("device barrier timeout during the timed region")

    in_bytes = (2 * n + 2 * m) * d * 2 * B * H
    if args.l2_flush:
        l2_note = "L2 flushed before every step (512 MiB written); step time = sum of the kernels"
    elif in_bytes > L2_BYTES:
        l2_note = f"inputs exceed L2 (Q,K,V,dO {in_bytes / 2**20:.0f} MiB per step > 129 MB)"
    else:
        l2_note = f"inputs fit in L2 ({in_bytes / 2**20:.0f} MiB), no flush between steps"
    ms_per_step = elapsed_ms / args.steps
    if args.l2_flush:
        ms_per_step = max_over_ranks(sum(stage), dev)
    flops_step = w.flops_fwd() + w.flops_bwd()
    value = weak_value(flops_step, world, ms_per_step)
    peaks = _peaks()
    peak, peak_kind = tensor_peak(peaks, clk)

    # Dominant kernel and its roofline.
    # Algorithmic FLOPs per kernel (the backward's 2.5x the forward all fall in
    # the gradient kernel). That kernel executes 3.5x: S^T, dP^T, dV, dK for
    # dK/dV (2.0) and S, dP, dQ for dQ (1.5, of which S and dP are the
    # recompute that replaces reductions into dQ in memory); reported apart.
    names = ["forward", "bwd_preprocess", "bwd_grads"]
    flops = [w.flops_fwd(), 0.0, w.flops_bwd()]
    top = max(range(3), key=lambda j: stage[j])
    if flops[top] > 0:
        ach = flops[top] / (stage[top] * 1e-3) / 1e12
        traffic = _traffic(names[top]) if w.name == WORKLOAD.name else None
        roof = {"kernel": names[top], "bound": "tensor", "achieved": ach, "peak": peak,
                "unit": "TFLOP/s", "frac": ach / peak, "traffic": traffic,
                "traffic_unit": "bytes per launch (ncu dram read + write)",
                "peak_kind": peak_kind,
                "frac_of_burst": ach / peaks["bf16_tflops"],
                "frac_of_sustained": ach / peaks["bf16_tflops_sustained"]}
    else:
        roof = {"kernel": names[top], "bound": "hbm", "achieved": None, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": None, "traffic": None}
    kernels = {}
    for j, nm in enumerate(names):
        entry = {"ms": stage[j]}
        if flops[j] > 0:
            entry["tflops"] = flops[j] / (stage[j] * 1e-3) / 1e12
        kernels[nm] = entry
    kernels["bwd_grads"]["tflops_executed"] = 3.5 * w.flops_fwd() / (stage[2] * 1e-3) / 1e12
    # The forward's second ceiling: exponentials (one per visible score) per SM
    # clock per SM, from the forward's event time and the sampled SM clock.
    n_exp = visible_pairs(n, m, w.causal) * B * H
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = clk.get("sm_mhz") or peaks["sm_max_mhz"]
    kernels["forward"]["exp"] = {
        "exps": n_exp, "per_s": n_exp / (stage[0] * 1e-3),
        "per_clk_per_sm": n_exp / (stage[0] * 1e-3 * mhz * 1e6 * sms),
        "sm_mhz": mhz, "sms": sms}
    bpe = 2
    pre_bytes = 2 * B * H * n * d * bpe + B * H * n * 4 * 3  # read O, dO, L; write -D, -L2
    kernels["bwd_preprocess"]["gbs"] = pre_bytes / (stage[1] * 1e-3) / 1e9

    e2e = None
    if not args.no_e2e:
        # End to end through the C-ABI host-buffer calls: pinned host inputs in,
        # forward + backward, every output back in host memory, each step. Each step
        # is submitted with fa_session_submit and the session pipelines the copies and
        # kernels over chunks of at most B*H/4 heads, continuing across steps (the
        # next step's copies in run while this step's copies out do);
        # fa_session_sync after the last step waits for all outputs.
        hq, hk, hv, hdo = (t.pin_memory() for t in (Q, K, V, dO))
        ho, hl = torch.empty_like(hq).pin_memory(), torch.empty((B, H, n), dtype=torch.float32).pin_memory()
        hdq, hdk, hdv = (torch.empty_like(t).pin_memory() for t in (hq, hk, hv))
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
        d2h = sum(t.numel() * t.element_size() for t in (ho, hl, hdq, hdk, hdv))
        chunk = max(1, -(-(B * H) // 4))
        sess = fa.Session(B, H, n, m, d, chunk)

        def e2e_step():
            sess.submit(hq, hk, hv, hdo, w.causal, O=ho, L=hl, dQ=hdq, dK=hdk, dV=hdv)

        e2e_steps = max(3, min(args.steps, 50))
        for _ in range(3):
            e2e_step()
        sess.sync()
        torch.cuda.synchronize(dev)
        barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        sess.sync()  # every step's outputs are in host memory
        e2e_ms = (time.perf_counter() - t0) * 1e3 / e2e_steps
        sess.close()
        barrier()
        e2e_ms = max_over_ranks(e2e_ms, dev)
        e2e_value = weak_value(flops_step, world, e2e_ms)
        e2e = {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "api": (f"fa_session_submit per step, fa_session_sync after the last; "
                       f"host buffers, chunks of at most {chunk} heads")}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = _cpu_baseline(w, args.cpu_heads)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.name, "shape": w.describe(), "global_batch": B * world,
                       "seq_len": n, "parallelism": f"independent heads x{world}",
                       "l2": l2_note,
                       "launch": "eager" if args.eager else "CUDA graph replay of the step"},
            "pct_of_peak": 100.0 * value / world / peak,
            "peak_kind": peak_kind,
            "pct_of_burst_peak": 100.0 * value / world / peaks["bf16_tflops"],
            "pct_of_sustained_peak": 100.0 * value / world / peaks["bf16_tflops_sustained"],
            "roofline": roof,
            "kernels": kernels,
            "e2e": e2e,
            "gpu_launches": 3 * args.steps,
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


SOFTMAX_ROWS, SOFTMAX_COLS, SOFTMAX_SEED = 32768, 4096, 1100


def run_online_softmax(args):
    """The standalone online-softmax statistics kernel on rows shaped like the
    benchmark's score rows (32768 rows of 4096 fp32, 512 MiB > L2): HBM bound."""
    import exact_io_aware_27_gb300 as fa

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    x = wl.score_rows(SOFTMAX_ROWS, SOFTMAX_COLS, SOFTMAX_SEED + rank).to(dev)
    m = torch.empty(SOFTMAX_ROWS, dtype=torch.float32, device=dev)
    l = torch.empty_like(m)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        fa.fa_online_softmax_stats(x, m, l)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev)
    clocks.start()
    time.sleep(0.2)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        fa.fa_online_softmax_stats(x, m, l)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), dev) / args.steps
    nbytes = SOFTMAX_ROWS * SOFTMAX_COLS * 4 + SOFTMAX_ROWS * 8
    value = nbytes * world / (ms * 1e-3) / 1e9
    peaks = _peaks()
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        orc = oracle.default()
        xs = x[:256].double().cpu().numpy()
        t0 = time.perf_counter()
        for r in range(xs.shape[0]):
            orc.online_softmax_stats(xs[r], SOFTMAX_COLS)
        dt = time.perf_counter() - t0
        cpu = {"value": xs.size * 4 / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"256 of {SOFTMAX_ROWS} rows, fp64, {dt:.2f} s"}
    line = {
        "metric": "online softmax statistics, GB/s of rows read (fp32)", "value": value,
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"score_rows_{SOFTMAX_ROWS}x{SOFTMAX_COLS}_f32",
                   "shape": f"{SOFTMAX_ROWS} rows x {SOFTMAX_COLS} fp32, N(0,1)*5, seed {SOFTMAX_SEED}",
                   "l2": "inputs exceed L2 (512 MiB)"},
        "roofline": {"kernel": "online_softmax_stats", "bound": "hbm", "achieved": value,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": value / peaks["hbm_gbs"],
                     "traffic": None},
        "e2e": None, "gpu_launches": args.steps, "clocks": clk, "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


IO_SIZES = (1024, 4096, 16384)
IO_QUERY_ROWS = 65536  # the batched rows: B*H*n query rows in total


def io_configs():
    """(label, B, H, n, d) of the IO comparison: one head at each n (the pages'
    per-head model) and a batch of heads holding IO_QUERY_ROWS query rows."""
    out = []
    for n in IO_SIZES:
        out.append((f"one_head_n{n}_d128", 1, 1, n, 128))
        out.append((f"h{IO_QUERY_ROWS // n}_n{n}_d128", 1, IO_QUERY_ROWS // n, n, 128))
    return out


def io_model_bytes(B, H, n, m, d):
    """Algorithmic memory traffic of one forward, non-causal, in bytes:
    standard = read Q, K, V; write S; read S; write P; read P; write O, L (the
    pages' 4 n m element accesses of S and P on top of the inputs and outputs);
    tiled = read Q, K, V; write O, L."""
    heads = B * H
    io = heads * ((2 * n + 2 * m) * d * 2 + n * 4)
    return {"standard": io + heads * 4 * n * m * 2, "tiled": io}


def run_io_compare(args):
    """The pages' IO comparison on the GPU: the materialised standard path
    (fa_standard_forward: S and P written to memory) against the tiled forward
    (fa_forward) on the same inputs, non-causal, d = 128. Times are CUDA-event
    medians with L2 flushed before every launch; memory is the peak the path
    allocates beyond its inputs. DRAM bytes per kernel come from ncu."""
    import exact_io_aware_27_gb300 as fa

    world, rank, local = _dist()
    if rank != 0:
        return 0
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    rows = []
    for label, B, H, n, d in io_configs():
        Q, K, V, _ = wl.attention_inputs(B, H, n, n, d, seed=9000 + n + H, qk_std=1.0)
        q, k, v = (t.to(dev) for t in (Q, K, V))
        res = {"config": label, "B": B, "H": H, "n": n, "m": n, "d": d,
               "model_bytes": io_model_bytes(B, H, n, n, d)}
        for path in ("standard", "tiled"):
            torch.cuda.synchronize(dev)
            base = torch.cuda.memory_allocated(dev)
            torch.cuda.reset_peak_memory_stats(dev)

            def call():
                if path == "standard":
                    return fa.fa_standard_forward(q, k, v, False)
                return fa.fa_forward(q, k, v, False)

            out = call()
            torch.cuda.synchronize(dev)
            peak = torch.cuda.max_memory_allocated(dev) - base
            out_bytes = B * H * n * (d * 2 + 4)  # O and L, which both paths return
            del out
            times = []
            for _ in range(max(3, args.warmup) + min(args.steps, 50)):
                flush.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                o = call()
                e1.record(stream)
                torch.cuda.synchronize(dev)
                times.append(e0.elapsed_time(e1))
                del o
            t = statistics.median(times[max(3, args.warmup):])
            res[path] = {"ms": t, "peak_alloc_bytes": peak, "extra_bytes": peak - out_bytes}
        res["time_ratio"] = res["standard"]["ms"] / res["tiled"]["ms"]
        rows.append(res)
        del q, k, v
        torch.cuda.empty_cache()
    if fa.fa_get_device_status() != 0:
        raise RuntimeError("device barrier timeout during the IO comparison")
    big = rows[-1]
    line = {
        "metric": "IO comparison: time of the materialised standard forward / the tiled forward",
        "value": big["time_ratio"], "unit": "x", "n_gpus": 1, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": big["tiled"]["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": big["config"], "l2": "L2 flushed (512 MiB written) before every launch",
                   "causal": False},
        "rows": rows, "e2e": None, "gpu_launches": 4 * len(rows) * (max(3, args.warmup) + args.steps + 1),
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(wl.WORKLOADS), default=WORKLOAD.name,
                    help="workload to time (default: the Llama-shaped causal one)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="launch every step from the host instead of replaying a CUDA graph")
    ap.add_argument("--l2-flush", action="store_true",
                    help="overwrite a buffer larger than L2 before every timed step")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end host-buffer loop (profiling runs)")
    ap.add_argument("--cpu-heads", type=int, default=4,
                    help="heads of the workload the oracle baseline times")
    ap.add_argument("--kernel", choices=["attention", "online_softmax", "io_compare"],
                    default="attention",
                    help="the attention step (default), the standalone online-softmax "
                         "statistics kernel, or the IO comparison of the materialised "
                         "standard forward against the tiled one")
    args = ap.parse_args()
    if args.kernel == "online_softmax":
        return run_online_softmax(args)
    if args.kernel == "io_compare":
        return run_io_compare(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
