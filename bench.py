#!/usr/bin/env python3
"""Throughput of the KDA forward + full backward on GB300.

One step = kda_fwd + kda_bwd (every kernel of the hot path) on the fixed
T=8192, H=96, K=V=128 workload (bf16 tokens, fp32 parameters and state), with
inputs resident in HBM. Metric: token*heads per second of fwd+bwd (also
TFLOP/s on the fixed algorithmic count of 421,888 flop per token*head).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

N > 1 runs under torchrun: every rank runs its own copy of the workload
(independent sequences and heads: weak scaling, no collective on the data
path); the time is the max over ranks. `--impl reference` times the fp64 CPU
oracle on the host cores, on a bounded sample of the same workload (rank 0).
Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FLOP_PER_TH = 421_888           # fwd 140,629 + bwd 281,259 per token*head (C = 64, d = 128)
# secondary count, reported beside the primary one: triangular products counted as full
# tiles, fwd 6d^2 + 10Cd + C^2/3 = 181,589 + bwd 12d^2 + 20Cd + 2C^2/3 = 363,179
FLOP_PER_TH_DENSE_TILE = 544_768
# algorithmic minimum of HBM bytes: fwd reads q, k, v, g_raw, beta_raw and writes o
# (1,282 B); bwd reads the same with dO and writes dq, dk, dv, dg_raw, dbeta_raw (2,308 B)
BYTES_PER_TH = 3_590
METRIC = "fwd+bwd tokens·heads/s and TFLOP/s (% of bf16 TC peak) at T=8192,H=96,K=V=128"
UNIT = "tokens*heads/s"
# kernels of one kda_fwd + kda_bwd (plain heads): chunk table (with the status clear and the
# provenance stamp), intra-chunk, forward scan; backward scan (with the stamp check), state
# products, WY, pair terms, parameter reduction
LAUNCHES_PER_STEP = 8
L2_FLUSH_BYTES = 512 << 20

# Per-kernel algorithmic traffic and MMA work per (chunk, head) tile: the
# tensors each kernel reads and writes once at its interface, and the flops
# of its products (triangular products counted at half size).
KB = 1024
KERNEL_MODEL = {
    # name: (bytes per tile, flops per tile)
    "fwd_intra": ((64 + 0.125) * KB + 320.5 * KB, 2.5e6),
    "fwd_scan": (256.5 * KB, 7.34e6),
    "bwd_scan": (224.5 * KB, 7.34e6),
    "bwd_state": (320.5 * KB, 6.82e6),
    "bwd_wy": (208.375 * KB, 5.24e6),
    "bwd_pair": (225.0 * KB, 2.62e6),
}

# DRAM traffic per tile (dram__bytes_read.sum + dram__bytes_write.sum, one ncu capture
# on T=4096 H=32, 2,048 tiles). Valid only for the kernel sources it was measured on:
# `sources` is a hash of csrc/, checked at run time.
MEASURED_TRAFFIC = {
    "sources": "dfbafb8bc21cad1e",
    "per_tile": {"fwd_intra": 366081, "fwd_scan": 244082, "bwd_scan": 211530, "bwd_state": 308172, "bwd_wy": 196808, "bwd_pair": 221721},
}


# files that do not build the kernels of the forward + backward step
_NOT_STEP_SOURCES = ("kda_decode.cu", "kda_diag.cu", "kda_noalloc.cu")


def _sources_hash():
    """Hash of the sources of the step's kernels: MEASURED_TRAFFIC holds for them only."""
    import glob
    import hashlib
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "kimi_delta_attention_15_gb300", "csrc", "*"))):
        if os.path.basename(f) in _NOT_STEP_SOURCES or not os.path.isfile(f):
            continue
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _workload(args):
    from kimi_delta_attention_15_gb300 import inputs as I
    if not args.workload:
        return I.WORKLOADS[I.HEADLINE]
    for w in I.WORKLOADS + I.EXTRA_WORKLOADS:
        if w.name == args.workload:
            return w
    raise SystemExit(f"unknown workload {args.workload}")


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region: sampling starts (and its
    first sample has arrived) before the region, every sample carries nvidia-smi's timestamp,
    and only the samples inside the region [mark_start, mark_end] count (the one nearest to it
    when the region is shorter than the sampling period)."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 50

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", str(self.PERIOD_MS)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            deadline = time.time() + 5.0
            while not self.rows and time.time() < deadline and self.proc.poll() is None:
                time.sleep(0.01)
        except Exception:
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    @staticmethod
    def _when(stamp):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y-%m-%d %H:%M:%S.%f"):
            try:
                return datetime.datetime.strptime(stamp, fmt).timestamp()
            except ValueError:
                pass
        return None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = [r for r in self.rows if len(r) >= 10 and r[2].replace(".", "").isdigit()]
        inside = rows
        if self.t0 is not None and self.t1 is not None and rows:
            stamped = [(self._when(r[0]), r) for r in rows]
            stamped = [(t, r) for t, r in stamped if t is not None]
            if stamped:
                inside = [r for t, r in stamped if self.t0 <= t <= self.t1]
                if not inside:   # region shorter than the period: the sample nearest to it
                    mid = 0.5 * (self.t0 + self.t1)
                    inside = [min(stamped, key=lambda tr: abs(tr[0] - mid))[1]]
        sm = [float(r[2]) for r in inside]
        mx = [float(r[3]) for r in inside if r[3].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            for i, nme in enumerate(names):
                if r[6 + i].lower().startswith("active"):
                    reasons.add(nme)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm), "period_ms": self.PERIOD_MS}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _init_dist(ws, backend):
    import torch.distributed as dist
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def reduce_max(value, ws, device=None):
    """Max of a float over ranks (identity at world size 1)."""
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_oracle_sample(inp, heads, nthreads):
    """Time the fp64 oracle (forward + backward) on `heads` heads of the workload."""
    import oracle
    sub = {}
    for k, v in inp.items():
        if k in ("q", "k", "v", "g_raw", "do"):
            sub[k] = v[:, :heads]
        elif k == "beta_raw":
            sub[k] = v[:, :heads]
        elif k in ("A_log", "dt_bias"):
            sub[k] = v[:heads]
        elif k in ("h0", "dhT"):
            sub[k] = None if v is None else v[:, :heads]
        else:
            sub[k] = v
    t0 = time.perf_counter()
    oracle.forward(sub, nthreads=nthreads)
    oracle.backward(sub, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return dt, sub["q"].shape[0] * heads


def run_reference(args, ws, rank):
    if rank != 0:
        return
    from kimi_delta_attention_15_gb300 import inputs as I
    import oracle
    w = _workload(args)
    inp = I.make_inputs(w)
    cores = oracle.default_threads()
    heads = max(1, min(w.H, cores))
    oracle.build()
    for _ in range(args.warmup):
        cpu_oracle_sample(inp, heads, cores)
    total, units = 0.0, 0
    for _ in range(args.steps):
        dt, n = cpu_oracle_sample(inp, heads, cores)
        total += dt
        units += n
    value = units / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "T": w.T, "H": w.H, "K": 128, "V": 128, "global_batch": 1,
                       "seq_len": w.T, "parallelism": "host threads"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{heads} of {w.H} heads x {w.T} tokens, fwd+bwd, per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_gb300(args, ws, rank, local):
    import torch
    from kimi_delta_attention_15_gb300 import inputs as I, ops

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = _init_dist(ws, "nccl")
    w = _workload(args)
    inp = I.make_inputs(w)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    cu = d["cu_seqlens"] if w.packed else None
    shape = ops.make_shape(w.T, w.H, w.N)
    wsp = ops.alloc_workspace(shape, dev)
    o = torch.empty_like(d["v"])
    hT = torch.empty(w.N, w.H, 128, 128, device=dev)
    grads = dict(dq=torch.empty_like(d["q"]), dk=torch.empty_like(d["k"]), dv=torch.empty_like(d["v"]),
                 dg_raw=torch.empty_like(d["g_raw"]), dbeta_raw=torch.empty_like(d["beta_raw"]),
                 dA_log=torch.empty_like(d["A_log"]), ddt_bias=torch.empty_like(d["dt_bias"]),
                 dh0=torch.empty(w.N, w.H, 128, 128, device=dev))
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        ops.fwd(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"], h0=d["h0"],
                cu_seqlens=cu, workspace=wsp, o=o, hT=hT)
        ops.bwd(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"], d["do"], wsp,
                cu_seqlens=cu, dhT=d["dhT"], grads=grads)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if ops.device_status(wsp) != 0:
        raise RuntimeError("device status after warm-up: %d" % ops.device_status(wsp))

    timer = ops.KernelTimer()

    def timed_region():
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        per_kernel = {k: 0.0 for k in ops.KERNEL_SLOTS}
        clocks = ClockSampler(local)
        if ws > 1:
            dist.barrier()
        clocks.start()
        torch.cuda.synchronize()
        clocks.mark_start()
        for i in range(args.steps):
            flush.zero_()                      # evict L2 between steps
            starts[i].record(stream)
            with timer:
                step()
            ends[i].record(stream)
            ends[i].synchronize()
            for k, v in timer.times_ms().items():
                per_kernel[k] += v
        torch.cuda.synchronize()
        clocks.mark_end()
        if ws > 1:
            dist.barrier()
        return starts, ends, per_kernel, clocks.stop()

    def clocks_rejected(c):
        """thermal or hardware slowdown, or SM clocks well below their maximum with no reason
        reported (a clock lock left by someone else): the measurement is taken once more"""
        if not c or c.get("sm_mhz") is None or not c.get("sm_max_mhz"):
            return False
        bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
        return bool(bad & set(c["reasons"])) or (c["sm_mhz"] < 0.9 * c["sm_max_mhz"] and not c["reasons"])

    starts, ends, per_kernel, clk = timed_region()
    if ws == 1 and clocks_rejected(clk):
        first = clk
        starts, ends, per_kernel, clk = timed_region()
        clk = dict(clk, remeasured_after=first)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = reduce_max(sum(step_ms), ws, dev)
    ms_per_step = total_ms / args.steps
    value = ws * w.token_heads / (ms_per_step * 1e-3)
    tflops = ws * w.token_heads * FLOP_PER_TH / (ms_per_step * 1e-3) / 1e12
    hbm, bf16, bf16s, peak_src = _peaks()

    # dominant kernel and its roofline
    kms = {k: v / args.steps for k, v in per_kernel.items()}
    dom = max(KERNEL_MODEL, key=lambda k: kms[k])
    tiles = sum((L + 63) // 64 for L in w.lengths) * w.H
    bytes_tile, flops_tile = KERNEL_MODEL[dom]
    t_s = kms[dom] * 1e-3
    gbs = bytes_tile * tiles / t_s / 1e9
    tfl = flops_tile * tiles / t_s / 1e12
    hbm_frac, tc_frac = gbs / hbm, tfl / bf16
    bound = "hbm" if hbm_frac >= tc_frac else "tensor"
    roof = ({"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": hbm_frac}
            if bound == "hbm" else
            {"bound": "tensor", "achieved": tfl, "peak": bf16, "unit": "TFLOP/s", "frac": tc_frac})
    traffic = None
    if _sources_hash() == MEASURED_TRAFFIC["sources"] and dom in MEASURED_TRAFFIC["per_tile"]:
        traffic = MEASURED_TRAFFIC["per_tile"][dom] * tiles   # bytes per launch, scaled by tiles
    roof.update({"kernel": dom, "traffic": traffic, "algorithmic_bytes": bytes_tile * tiles,
                 "peak_source": peak_src,
                 "kernel_ms": {k: round(v, 4) for k, v in kms.items()}})

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 io, tf32 mma (bf16 mma for the cross terms of fp32-accurate products), fp32 accum/state", "data": "synthetic",
            "config": {"workload": w.name, "T": w.T, "H": w.H, "K": 128, "V": 128, "global_batch": 1,
                       "seq_len": w.T, "parallelism": f"replicas{ws}" if ws > 1 else "single",
                       "l2": "flushed (512 MiB write) before every timed step"},
            "tflops": tflops, "pct_bf16_peak": tflops / bf16,
            "tflops_dense_tile": tflops * FLOP_PER_TH_DENSE_TILE / FLOP_PER_TH,
            "gbs": value * BYTES_PER_TH / 1e9, "pct_hbm_peak": value * BYTES_PER_TH / 1e9 / hbm,
            "fwd_ms": sum(v for k, v in kms.items() if k.startswith("fwd")),
            "bwd_ms": sum(v for k, v in kms.items() if k.startswith("bwd")),
            "roofline": roof, "clocks": clk, "gpu_launches": LAUNCHES_PER_STEP * args.steps}

    # end to end through the public API with pinned host buffers
    if not args.no_e2e:
        line["e2e"] = e2e(args, inp, dev, w)
    if args.decode_requests > 0:
        line["decode"] = decode_bench(dev, hbm, n_req=args.decode_requests)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        cores = oracle.default_threads()
        heads = max(1, min(w.H, cores))
        dt, n = cpu_oracle_sample(inp, heads, cores)
        line["cpu_baseline"] = {"value": n / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": f"{heads} of {w.H} heads x {w.T} tokens, fwd+bwd, {dt:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def e2e(args, inp, dev, w):
    """Same metric with host buffers: every step copies all of its inputs from pinned
    host memory to the device, runs kda_fwd + kda_bwd, and copies the output and every
    gradient back, all inside the timed region. Reported two ways:
      pipelined (the `value`): inputs of step n+1 go up on one copy stream and results
        of step n-1 come down on another while the kernels of step n run (two device
        input buffers), as a training loop streaming batches from the host would;
      serial: copy in, compute, copy out, one after the other on one stream."""
    import torch
    from kimi_delta_attention_15_gb300 import ops
    names = ("q", "k", "v", "g_raw", "beta_raw", "A_log", "dt_bias", "do")
    host = {k: inp[k].pin_memory() for k in names}
    dvs = [{k: torch.empty_like(host[k], device=dev) for k in names} for _ in range(2)]
    cu = inp["cu_seqlens"].to(dev) if w.packed else None
    shape = ops.make_shape(w.T, w.H, w.N)
    wsp = ops.alloc_workspace(shape, dev)
    out_host = {"o": torch.empty_like(host["v"]).pin_memory()}
    for k in ("q", "k", "v", "g_raw", "beta_raw", "A_log", "dt_bias"):
        out_host["d" + k] = torch.empty_like(host[k]).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in out_host.values())
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()

    def compute(dv):
        o, _, _ = ops.fwd(dv["q"], dv["k"], dv["v"], dv["g_raw"], dv["beta_raw"], dv["A_log"], dv["dt_bias"],
                          cu_seqlens=cu, workspace=wsp, want_hT=False)
        g = ops.bwd(dv["q"], dv["k"], dv["v"], dv["g_raw"], dv["beta_raw"], dv["A_log"], dv["dt_bias"], dv["do"],
                    wsp, cu_seqlens=cu, want_dh0=False)
        res = {"o": o}
        res.update({"d" + k: g["d" + k] for k in ("q", "k", "v", "g_raw", "beta_raw", "A_log", "dt_bias")})
        return res

    def copy_down(res):
        for k, t in res.items():
            t.record_stream(down)
            out_host[k].copy_(t, non_blocking=True)

    def serial_step():
        dv = dvs[0]
        for k in names:
            dv[k].copy_(host[k], non_blocking=True)
        res = compute(dv)
        for k, t in res.items():
            out_host[k].copy_(t, non_blocking=True)

    def pipelined(nsteps):
        free = [torch.cuda.Event(), torch.cuda.Event()]   # compute done reading buffer b
        for ev in free:
            ev.record(comp)
        ready = [torch.cuda.Event(), torch.cuda.Event()]  # inputs of buffer b on the device

        def upload(i):
            b = i % 2
            up.wait_event(free[b])
            with torch.cuda.stream(up):
                for k in names:
                    dvs[b][k].copy_(host[k], non_blocking=True)
                ready[b].record(up)

        upload(0)
        for i in range(nsteps):
            b = i % 2
            if i + 1 < nsteps:
                upload(i + 1)
            comp.wait_event(ready[b])
            res = compute(dvs[b])
            free[b].record(comp)
            done = torch.cuda.Event()
            done.record(comp)
            down.wait_event(done)
            with torch.cuda.stream(down):
                copy_down(res)
        comp.wait_stream(down)

    def timed(fn):
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(comp)
        up.wait_stream(comp)
        down.wait_stream(comp)
        fn()
        e.record(comp)
        e.synchronize()
        return s.elapsed_time(e) / args.steps

    for _ in range(max(1, args.warmup)):
        serial_step()
    pipelined(max(2, args.warmup))
    ms_serial = timed(lambda: [serial_step() for _ in range(args.steps)])
    ms = timed(lambda: pipelined(args.steps))
    return {"value": w.token_heads / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "mode": "pipelined: step n+1 inputs up and step n-1 results down overlap step n kernels",
            "serial": {"value": w.token_heads / (ms_serial * 1e-3), "ms_per_step": ms_serial}}


def decode_bench(dev, hbm_peak, n_req=256, H=96, steps=20):
    """One decode step (kda_decode) for n_req requests x H heads: each (request, head)
    reads and writes its 64 KB fp32 state once, 3.2 GB in all, more than L2, so the
    step streams from HBM. Times `steps` consecutive steps with CUDA events."""
    import torch
    from kimi_delta_attention_15_gb300 import ops
    g = torch.Generator(device="cpu").manual_seed(20261202)
    tok = lambda: torch.randn(n_req, H, 128, generator=g).to(torch.bfloat16).to(dev)
    q, k, v, g_raw = tok(), tok(), tok(), tok()
    beta_raw = torch.randn(n_req, H, generator=g).to(torch.bfloat16).to(dev)
    A_log = torch.log(torch.rand(H, generator=g) * 15 + 1).to(dev)
    dt_bias = (0.1 * torch.randn(H, 128, generator=g)).to(dev)
    state = (0.1 * torch.randn(n_req, H, 128, 128, generator=g)).to(dev)
    o = torch.empty_like(v)
    for _ in range(3):
        ops.decode(q, k, v, g_raw, beta_raw, A_log, dt_bias, state, o=o)
    torch.cuda.synchronize()
    s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record()
    for _ in range(steps):
        ops.decode(q, k, v, g_raw, beta_raw, A_log, dt_bias, state, o=o)
    e0.record()
    e0.synchronize()
    ms = s0.elapsed_time(e0) / steps
    units = n_req * H
    bytes_step = units * (2 * 128 * 128 * 4 + 5 * 128 * 2 + 2)   # state in + out, q k v g o rows, beta
    gbs = bytes_step / (ms * 1e-3) / 1e9
    return {"workload": f"decode_{n_req}req_H{H}", "ms_per_step": ms,
            "tokens_heads_per_s": units / (ms * 1e-3), "bound": "hbm", "achieved_gbs": gbs,
            "peak_gbs": hbm_peak, "frac": gbs / hbm_peak, "bytes_per_step": bytes_step}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default=None,
                    help="name of a workload in kimi_delta_attention_15_gb300.inputs (default: the T=8192, H=96 one)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-requests", type=int, default=256,
                    help="requests in the decode measurement (x 96 heads; 0 skips it)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = _dist()
    if args.impl == "reference":
        if ws > 1:
            _init_dist(ws, "gloo")
        run_reference(args, ws, rank)
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    run_gb300(args, ws, rank, local)


if __name__ == "__main__":
    main()
