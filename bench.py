"""Benchmark: packed varlen bf16 attention, forward + backward, on the
windowed workload (8 segments, cu_seqlens_q = [0, 4032, ..., 35280], 17580 kv
rows per segment, H=56, D=128), as TFLOP/s:

    forward  4 * sum_b Sq_b * Sk_b * H * D   per step
    backward 2.5 x the forward count

One step = varlen_attn_fwd then varlen_attn_bwd over one batch of synthetic
inputs (seeded N(0,1) bf16) resident in HBM.  Inputs (q 0.5 GB, k and v 2 GB
each) are larger than L2, so no flush is needed between iterations.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs a batch of the same shape (its own seed) on its
own GPU, with no collective on the data path: weak scaling.  Rank 0 prints one
JSON line.  ``--impl reference`` times the fp64 CPU oracle (the only other
implementation of this operation here) on a bounded sample of the same
workload.
"""
from __future__ import annotations

import argparse
import json
import os
import pathlib
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np
import torch

from packed_variable_length_varlen_gb300 import sharding
from packed_variable_length_varlen_gb300 import workloads as W

METRIC = "varlen attention TFLOP/s (fwd, bwd) bf16 H=56 D=128; % of GB300 bf16 TC peak"
BWD_MAIN_DRAM_BYTES_PER_HEAD = {("windowed", 128): (874.832640e6 + 671.547392e6) / 8}


def _window(args):
    return tuple(args.window) if getattr(args, "window", None) else (-1, -1)


def _metric(args) -> str:
    mask = []
    if getattr(args, "causal", False):
        mask.append("causal")
    if _window(args) != (-1, -1):
        mask.append("window(%d,%d)" % _window(args))
    return METRIC.replace("bf16", "bf16 " + " ".join(mask), 1) if mask else METRIC


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.loads(pathlib.Path(p).read_text())
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons for one GPU."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.uuid = None
        try:
            self.uuid = str(torch.cuda.get_device_properties(device).uuid)
            if not self.uuid.startswith("GPU-"):
                self.uuid = "GPU-" + self.uuid
        except Exception:
            pass
        self.proc = None
        self.lines = []

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits", "-lms", "200"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(local)
    return ws, rank, local


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x: float, ws: int) -> float:
    return x if ws == 1 else sharding.max_over_ranks(x)


# ------------------------------------------------------------------ CPU side

def prep_roofline(total_q: int, num_heads: int, head_dim: int, prep_ms: float, hbm_gbs: float,
                  zero_accumulator: bool = True) -> dict:
    """HBM roofline of the backward preprocess: per (q row, head) it reads O
    and dO (2 D bf16) and LSE, writes delta and lse2 (the algorithmic bytes,
    4 D + 12), and, on the default path, zeroes the fp32 dQ accumulator
    (4 D more, reported as moved bytes, not algorithmic)."""
    pairs = float(total_q) * num_heads
    alg = pairs * (4 * head_dim + 12)
    moved = alg + (pairs * 4 * head_dim if zero_accumulator else 0.0)
    sec = prep_ms * 1e-3
    return {"kernel": "varlen_bwd_prep_kernel", "bound": "hbm", "unit": "GB/s", "peak": hbm_gbs,
            "achieved": alg / sec / 1e9, "frac": alg / sec / 1e9 / hbm_gbs,
            "moved_gbs": moved / sec / 1e9, "moved_frac": moved / sec / 1e9 / hbm_gbs,
            "algorithmic_bytes": alg, "moved_bytes": moved}


def _parse_cpulist(text: str):
    cpus = set()
    for part in text.strip().split(","):
        if not part:
            continue
        a, _, b = part.partition("-")
        cpus.update(range(int(a), int(b or a) + 1))
    return cpus


def _bind_near_gpu(dev_index: int):
    """Restricts this process to the CPUs the kernel lists as local to the
    GPU (its PCI device's local_cpulist), intersected with the CPUs it may
    use, so that pinned host buffers allocated afterwards sit in the memory
    next to that GPU.  Returns (previous affinity, description) or None when
    the topology is not readable."""
    try:
        p = torch.cuda.get_device_properties(dev_index)
        bdf = "%04x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        with open("/sys/bus/pci/devices/%s/local_cpulist" % bdf) as f:
            local = _parse_cpulist(f.read())
        before = os.sched_getaffinity(0)
        use = local & before
        if not use or use == before:
            return before, "unchanged (%d CPUs)" % len(before)
        os.sched_setaffinity(0, use)
        return before, "%d of %d CPUs local to %s" % (len(use), len(before), bdf)
    except (OSError, AttributeError, ValueError):
        return None


def _cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), e.g. an x86
    'model name' or an Arm 'Neoverse-V2'."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def _copy_rates(dev_t: torch.Tensor, host_in: torch.Tensor, host_out: torch.Tensor, stream) -> dict:
    """Pinned host <-> device copy bandwidth in GB/s, measured with CUDA
    events: host_in -> dev_t alone, dev_t -> host_out alone, and both at once
    on two streams (into a second device buffer), best of three each."""
    dev = dev_t.device
    nbytes = dev_t.numel() * dev_t.element_size()
    other = torch.empty_like(dev_t)
    s2 = torch.cuda.Stream(dev)

    def timed(fn):
        best = None
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        return best

    def both():
        s2.wait_stream(stream)
        with torch.cuda.stream(s2):
            other.copy_(host_in, non_blocking=True)
        host_out.copy_(dev_t, non_blocking=True)
        stream.wait_stream(s2)

    with torch.cuda.stream(stream):
        h2d = timed(lambda: dev_t.copy_(host_in, non_blocking=True))
        d2h = timed(lambda: host_out.copy_(dev_t, non_blocking=True))
        conc = timed(both)
    return {"bytes": int(nbytes), "h2d_gbs": nbytes / h2d / 1e6, "d2h_gbs": nbytes / d2h / 1e6,
            "concurrent_each_gbs": nbytes / conc / 1e6}


def _oracle_rate(w: W.Workload, target_s: float, seed: int = 0, causal: bool = False, window=(-1, -1)):
    """Times the oracle (forward + query-side backward) on sampled (row, head)
    pairs of the workload.  Credits each pair with its share of the step's
    algorithmic flops: 4*n*D (forward) + 10*n*D (backward), n = the keys the
    row sees (Sk, or fewer under a mask)."""
    import oracle
    inp = W.make_inputs(w, seed)
    pb = oracle.Problem(inp.q, inp.k, inp.v, inp.cu_q, inp.cu_k, w.softmax_scale, dout=inp.dout, causal=causal,
                        window=window)
    rng = np.random.default_rng(5)
    seg_k = {b: w.cu_k[b + 1] - w.cu_k[b] for b in range(w.batch)}

    def sample(n):
        rows = rng.integers(0, w.total_q, size=n).astype(np.int64)
        heads = rng.integers(0, w.num_heads, size=n).astype(np.int32)
        return rows, heads

    def flops(rows):
        b = np.searchsorted(np.asarray(w.cu_q), rows, side="right") - 1
        sk = np.array([seg_k[int(x)] for x in b], dtype=np.int64)
        sq = np.array([w.cu_q[int(x) + 1] - w.cu_q[int(x)] for x in b], dtype=np.int64)
        n = W.row_keys(rows - np.asarray(w.cu_q)[b], sq, sk, causal, window)
        return float((14.0 * n * w.head_dim).sum())

    def run(n):
        rows, heads = sample(n)
        t0 = time.perf_counter()
        pb.fwd(rows, heads)
        pb.bwd_q(rows, heads)
        return time.perf_counter() - t0, flops(rows), n

    # calibrate on a probe large enough that fixed per-call costs do not dominate
    probe = 256
    t, f, n = run(probe)
    n = int(max(probe, min(200000, probe * target_s / max(t, 1e-3))))
    return run, n, oracle.num_threads()


def reference_arm(args, w, ws, rank):
    """The oracle, as it stands, on the host cores: each step one bounded
    sample of the workload."""
    if rank != 0:
        return
    run, n, cores = _oracle_rate(w, target_s=max(2.0, 150.0 / max(args.steps + args.warmup, 1)),
                                 causal=args.causal, window=_window(args))
    for _ in range(args.warmup):
        run(n)
    tot_t = tot_f = 0.0
    for _ in range(args.steps):
        t, f, _ = run(n)
        tot_t += t
        tot_f += f
    val = tot_f / tot_t / 1e12
    sample = "oracle fwd + dQ backward on %d random (row, head) pairs of the %s workload per step" % (n, w.name)
    line = {"impl": "reference", "metric": _metric(args), "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "sample": sample},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "cpu_model": _cpu_model(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU side

def ours(args, w, ws, rank, local):
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    dev = torch.device("cuda", local)
    full_flops = None
    if args.shard == "heads":
        # one problem split by heads: every rank draws the same inputs and
        # runs its head range as views t[:, h0:h1] (no copies, no collective)
        h0, h1 = sharding.head_range(w.num_heads, ws, rank)
        if h1 == h0:
            raise SystemExit("--shard heads needs at most num_heads ranks")
        full_flops = (w.fwd_flops(args.causal, _window(args)), w.bwd_flops(args.causal, _window(args)))
        cpu = W.make_inputs(w, seed=0)
        for n in ("q", "k", "v", "dout"):
            setattr(cpu, n, getattr(cpu, n)[:, h0:h1])
        w = w.with_(num_heads=h1 - h0)
        args.no_e2e = True
    else:
        cpu = W.make_inputs(w, seed=rank)  # each rank's own batch of the same shape
    d = cpu.to(dev)
    H, D = w.num_heads, w.head_dim
    out = torch.empty_like(d.q)
    lse = torch.empty(H, w.total_q, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(d.q), torch.empty_like(d.k), torch.empty_like(d.v)
    ws_bytes = va.varlen_attn_bwd_workspace_size(w.batch, w.total_q, H, D)
    wsp = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    scale = w.softmax_scale
    stream = torch.cuda.current_stream(dev)

    if args.dense:
        sq_, sk_ = w.seqlens_q(), w.seqlens_k()
        if len(set(sq_)) != 1 or len(set(sk_)) != 1:
            raise SystemExit("--dense needs a workload with equal segment lengths (e.g. --workload dense)")
        if _window(args) != (-1, -1) or args.deterministic:
            raise SystemExit("--dense takes neither --window nor --deterministic (the dense entry points carry "
                             "the causal flag only)")
        Sq, Sk = sq_[0], sk_[0]
        ws_bytes = va.varlen_attn_bwd_dense_workspace_size(w.batch, Sq, H, D)
        wsp = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)

        def as4(t, S):  # the [batch, S, H, D] view of a packed [batch*S, H, D] tensor
            return t.as_strided((w.batch, S, H, D), (S * t.stride(0), t.stride(0), t.stride(1), 1), t.storage_offset())

    def run_fwd(x, o, l):
        if args.dense:
            st = va.varlen_attn_fwd_dense(as4(x.q, Sq), as4(x.k, Sk), as4(x.v, Sk), w.batch, Sq, Sk, H, D, scale,
                                          args.causal, as4(o, Sq), l, stream)
        else:
            st = va.varlen_attn_fwd(x.q, x.k, x.v, x.cu_q, x.cu_k, w.batch, w.total_q, w.total_k, H, D, w.max_q(),
                                    w.max_k(), scale, o, l, stream, causal=args.causal, window=_window(args))
        assert st == 0, va.varlen_attn_status_string(st)

    def run_bwd(x, o, l, gq, gk, gv):
        if args.dense:
            st = va.varlen_attn_bwd_dense(as4(x.q, Sq), as4(x.k, Sk), as4(x.v, Sk), as4(o, Sq), as4(x.dout, Sq),
                                          l, w.batch, Sq, Sk, H, D, scale, args.causal, as4(gq, Sq), as4(gk, Sk),
                                          as4(gv, Sk), wsp, ws_bytes, stream)
        else:
            st = va.varlen_attn_bwd(x.q, x.k, x.v, o, x.dout, l, x.cu_q, x.cu_k, w.batch, w.total_q,
                                    w.total_k, H, D, w.max_q(), w.max_k(), scale, gq, gk, gv, wsp, ws_bytes, stream,
                                    causal=args.causal, window=_window(args), deterministic=args.deterministic)
        assert st == 0, va.varlen_attn_status_string(st)

    def fwd():
        run_fwd(d, out, lse)

    def bwd():
        run_bwd(d, out, lse, dq, dk, dv)

    # one untimed forward and backward, checked for device errors
    fwd()
    bwd()
    has_bwd = True
    torch.cuda.synchronize()
    assert va.varlen_attn_get_device_status(stream) == 0

    K, Wm = args.steps, args.warmup
    for _ in range(Wm):
        fwd()
        if has_bwd:
            bwd()
    torch.cuda.synchronize()
    assert va.varlen_attn_get_device_status(stream) == 0

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    # per-kernel events inside varlen_attn_bwd: before prep / after prep /
    # after main / after the dQ conversion
    pev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local) if rank == 0 else None
    _barrier(ws)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    e_start.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        if has_bwd:
            va.varlen_attn_debug_set_phase_events(pev[i])
            bwd()
        ev[i][2].record(stream)
    e_end.record(stream)
    torch.cuda.synchronize()
    _barrier(ws)
    clocks = sampler.stop() if sampler else None
    va.varlen_attn_debug_set_phase_events(None)
    status = va.varlen_attn_get_device_status(stream)
    assert status == 0, va.varlen_attn_status_string(status)

    ms_total = _max_over_ranks(e_start.elapsed_time(e_end), ws)
    t_fwd = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    t_bwd = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    f_fwd = w.fwd_flops(args.causal, _window(args))
    f_bwd = w.bwd_flops(args.causal, _window(args)) if has_bwd else 0.0
    step_flops = f_fwd + f_bwd
    value = ws * K * step_flops / (ms_total * 1e-3) / 1e12
    if full_flops is not None:  # a head split: all ranks together did the one problem's flops
        value = K * (full_flops[0] + (full_flops[1] if has_bwd else 0.0)) / (ms_total * 1e-3) / 1e12
    fwd_tflops = f_fwd / (statistics.mean(t_fwd) * 1e-3) / 1e12
    bwd_tflops = f_bwd / (statistics.mean(t_bwd) * 1e-3) / 1e12 if has_bwd else None

    # ---- end to end through the C ABI with host buffers (pinned)
    e2e = None
    if not args.no_e2e:
        bound = _bind_near_gpu(local)
        host = {n: getattr(cpu, n).pin_memory() if getattr(cpu, n)._base is None
                else getattr(cpu, n)._base.pin_memory() for n in ("q", "k", "v", "dout")}
        hcu_q, hcu_k = cpu.cu_q.pin_memory(), cpu.cu_k.pin_memory()
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        h_dq, h_dk, h_dv = (torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dk, dv))
        h2d_bytes = sum(t.numel() * t.element_size() for t in host.values()) + (0 if args.dense else 2 * hcu_q.numel() * 4)
        d2h_bytes = sum(t.numel() * t.element_size() for t in (h_out, h_lse)) + (
            sum(t.numel() * t.element_size() for t in (h_dq, h_dk, h_dv)) if has_bwd else 0)

        # Every step copies its own inputs in (pinned host -> device) and its
        # own results out (device -> pinned host).  The copies of step i+1's
        # inputs and of step i-1's results run on two copy streams while step
        # i computes, on double-buffered device inputs and outputs; events
        # order each buffer's reuse.
        copy_in = torch.cuda.Stream(dev)
        copy_out = torch.cuda.Stream(dev)
        sets = [d, cpu.to(dev)]
        outs = [(out, lse, dq, dk, dv), (torch.empty_like(out), torch.empty_like(lse), torch.empty_like(dq),
                                         torch.empty_like(dk), torch.empty_like(dv))]

        def h2d(i):
            x = sets[i % 2]
            for n, h in host.items():
                t = getattr(x, n)
                (t if t._base is None else t._base).copy_(h, non_blocking=True)
            if not args.dense:  # the dense entry points take no cu_seqlens
                x.cu_q.copy_(hcu_q, non_blocking=True)
                x.cu_k.copy_(hcu_k, non_blocking=True)

        def compute(i):
            x = sets[i % 2]
            o, l, gq, gk, gv = outs[i % 2]
            run_fwd(x, o, l)
            if has_bwd:
                run_bwd(x, o, l, gq, gk, gv)

        def d2h(i):
            o, l, gq, gk, gv = outs[i % 2]
            h_out.copy_(o, non_blocking=True)
            h_lse.copy_(l, non_blocking=True)
            if has_bwd:
                h_dq.copy_(gq, non_blocking=True)
                h_dk.copy_(gk, non_blocking=True)
                h_dv.copy_(gv, non_blocking=True)

        def e2e_run(n, start, end, spans=None):
            """n pipelined steps between start and end; with `spans`, timing
            events around every copy and every step's kernels are appended to
            it as (kind, begin, end)."""
            ev = lambda: torch.cuda.Event()
            in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

            def span(kind, s, fn):
                if spans is None:
                    fn()
                    return
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(s)
                fn()
                b.record(s)
                spans.append((kind, a, b))

            start.record(stream)
            copy_in.wait_event(start)
            copy_out.wait_event(start)
            with torch.cuda.stream(copy_in):
                span("h2d", copy_in, lambda: h2d(0))
                in_done[0].record(copy_in)
            for i in range(n):
                b = i % 2
                if i + 1 < n:  # inputs of step i+1, once step i-1 has finished reading that set
                    with torch.cuda.stream(copy_in):
                        if i >= 1:
                            copy_in.wait_event(comp_done[(i + 1) % 2])
                        span("h2d", copy_in, lambda: h2d(i + 1))
                        in_done[(i + 1) % 2].record(copy_in)
                stream.wait_event(in_done[b])
                if i >= 2:
                    stream.wait_event(out_done[b])  # step i-2's results have left this output set
                span("kernels", stream, lambda: compute(i))
                comp_done[b].record(stream)
                with torch.cuda.stream(copy_out):
                    copy_out.wait_event(comp_done[b])
                    span("d2h", copy_out, lambda: d2h(i))
                    out_done[b].record(copy_out)
            stream.wait_event(out_done[(n - 1) % 2])
            stream.wait_event(in_done[(n - 1) % 2])
            end.record(stream)

        # the copy rates of this machine, measured on the largest input (k)
        rates = _copy_rates(d.k if d.k._base is None else d.k._base, host["k"],
                            torch.empty(host["k"].shape, dtype=host["k"].dtype).pin_memory(), stream)
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2e_run(2, a, b_)
        torch.cuda.synchronize()
        _barrier(ws)
        ke = K  # the same K steps as the device-timed value; the first copy-in and last copy-out are not hidden
        spans = []
        e2e_run(ke, a, b_, spans)
        torch.cuda.synchronize()
        ms_e2e = _max_over_ranks(a.elapsed_time(b_), ws)
        # what each copy and each step's kernels took inside the pipeline (a
        # machine whose copies slow the kernels, or the other way round, shows here)
        in_pipe = {k: statistics.mean(x.elapsed_time(y) for kk, x, y in spans if kk == k)
                   for k in ("h2d", "kernels", "d2h")}
        # What the copies alone cost per step at the measured concurrent
        # rate: with the copies overlapped, a step takes about the larger of
        # this and the kernels' time.
        copy_ms = 1e3 * max(h2d_bytes, d2h_bytes) / (rates["concurrent_each_gbs"] * 1e9)
        kern_ms = ms_total / K
        e2e = {"value": ws * ke * step_flops / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d_bytes), "d2h_bytes_per_step": int(d2h_bytes), "ms_per_step": ms_e2e / ke,
               "pipeline": "step i+1 inputs in and step i-1 results out on two copy streams during step i",
               "copy_rates": rates, "copy_ms_per_step_at_concurrent_rate": copy_ms,
               "kernel_ms_per_step": kern_ms, "exposed_ms_per_step": ms_e2e / ke - kern_ms,
               "in_pipeline_ms": in_pipe,
               "bound": "copies" if copy_ms > kern_ms else "kernels",
               "host_cpus": bound[1] if bound else "topology not readable"}
        if bound:
            os.sched_setaffinity(0, bound[0])  # the CPU baseline below uses every core again

    peaks, src = _peaks()
    if rank != 0:
        return
    # roofline of the dominant kernel (the one launch that does the most flops)
    t_prep = t_main = t_post = None
    if has_bwd:
        t_prep = statistics.mean(pev[i][0].elapsed_time(pev[i][1]) for i in range(K))
        t_main = statistics.mean(pev[i][1].elapsed_time(pev[i][2]) for i in range(K))
        t_post = statistics.mean(pev[i][2].elapsed_time(pev[i][3]) for i in range(K))
        dom_name, dom_flops, dom_ms = "varlen_bwd_main_kernel", f_bwd, t_main
        if args.deterministic:
            # The main kernel runs four of the five products (S^T, dP^T, dV, dK);
            # the dQ kernel recomputes S and dP and runs dQ (three, 0.6 x the
            # backward's algorithmic flops).
            dom_flops = 0.8 * f_bwd
    else:
        dom_name, dom_flops, dom_ms = "varlen_fwd_kernel", f_fwd, statistics.mean(t_fwd)
    ach = dom_flops / (dom_ms * 1e-3) / 1e12
    # The kernels run at the maximum SM clock without power capping (see
    # "clocks"), so the burst cuBLAS figure is the denominator; the sustained
    # (power-capped) figure is reported beside it.
    peak = float(peaks.get("bf16_tflops"))
    sust = float(peaks.get("bf16_tflops_sustained", peak))
    # DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the backward main
    # kernel, from one ncu capture of the windowed workload at H=8 (kernel as of commit af71323).
    # Every head reads its own q, k, v, dout and writes its own dk, dv and dq rows, so the
    # traffic scales with the number of heads.  Reported only for that workload and head size.
    traffic = None
    if dom_name == "varlen_bwd_main_kernel" and not args.causal and _window(args) == (-1, -1) and (w.name, D) in BWD_MAIN_DRAM_BYTES_PER_HEAD:
        traffic = BWD_MAIN_DRAM_BYTES_PER_HEAD[(w.name, D)] * H
    roof = {"kernel": dom_name, "bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
            "frac": ach / peak, "peak_source": "%s bf16_tflops (burst)" % src,
            "frac_of_sustained": ach / sust, "traffic": traffic}

    cpu_base = None
    if not args.no_cpu_baseline and ws == 1:  # the CPU baseline is reported at N = 1 only
        run, n, cores = _oracle_rate(w, target_s=12.0, causal=args.causal, window=_window(args))
        t, f, n = run(n)
        cpu_base = {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": cores, "cpu_model": _cpu_model(),
                    "kind": "oracle",
                    "sample": "oracle fwd + dQ backward on %d random (row, head) pairs of the %s workload "
                              "(%.1f s); each pair credited with 14*Sk*D flops" % (n, w.name, t)}

    burst = float(peaks.get("bf16_tflops"))
    line = {
        "metric": _metric(args), "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": K, "warmup": Wm,
        "ms_per_step": ms_total / K, "higher_is_better": True,
        "scaling": "strong" if full_flops is not None else "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "batch_segments": w.batch, "total_q": w.total_q, "total_k": w.total_k,
                   "num_heads": H, "head_dim": D, "step": "fwd+bwd" if has_bwd else "fwd only (bwd missing)",
                   "causal": bool(args.causal), "window": list(_window(args)),
                   "deterministic_bwd": bool(args.deterministic), "entry": "dense batched" if args.dense else "packed varlen",
                   "l2": "inputs larger than L2 (k, v 2 GB each); no flush",
                   "parallelism": ("heads split over %d ranks (this rank %d heads)" % (ws, H) if full_flops is not None
                                   else ("replicas" if ws > 1 else "single GPU"))},
        "fwd_tflops": fwd_tflops, "bwd_tflops": bwd_tflops,
        "fwd_frac_of_burst_peak": fwd_tflops / burst,
        "bwd_frac_of_burst_peak": (bwd_tflops / burst) if bwd_tflops else None,
        "fwd_ms": statistics.mean(t_fwd), "bwd_ms": statistics.mean(t_bwd) if has_bwd else None,
        "bwd_kernel_ms": ({"prep": t_prep, "main": t_main, ("dq" if args.deterministic else "post"): t_post}
                          if has_bwd else None),
        "fwd_kernel_roofline": {"achieved": fwd_tflops, "peak": peak, "frac": fwd_tflops / peak,
                                "frac_of_sustained": fwd_tflops / sust},
        "prep_kernel_roofline": (prep_roofline(w.total_q, H, D, t_prep, float(peaks.get("hbm_gbs", 6800.0)),
                                               zero_accumulator=not args.deterministic) if has_bwd else None),
        "clocks": clocks, "e2e": e2e, "gpu_launches": K * (1 + (3 if has_bwd else 0)),
        "roofline": roof, "cpu_baseline": cpu_base,
    }
    print(json.dumps(line), flush=True)


def fp8_forward(args, w, ws, rank, local):
    """Times the E4M3 forward (quantisation passes included) alone: K calls
    after W warm-up calls, CUDA events on the launching stream, max over
    ranks; FLOPs at the bf16 forward count (over the visible pairs under
    --causal / --window)."""
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    if w.head_dim != 128:
        raise SystemExit("--fp8 times the E4M3 forward: head size 128")
    causal, window = bool(args.causal), _window(args)
    dev = torch.device("cuda", local)
    d = W.make_inputs(w, seed=rank, with_dout=False).to(dev)
    H = w.num_heads
    out = torch.empty_like(d.q)
    lse = torch.empty(H, w.total_q, dtype=torch.float32, device=dev)
    nbytes = va.varlen_attn_fwd_fp8_workspace_size(w.batch, w.total_q, w.total_k, H, 128)
    wsp = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    if args.dense:
        sq_, sk_ = w.seqlens_q(), w.seqlens_k()
        if len(set(sq_)) != 1 or len(set(sk_)) != 1 or window != (-1, -1):
            raise SystemExit("--fp8 --dense needs equal segment lengths (e.g. --workload dense) and no --window")
        Sq, Sk = sq_[0], sk_[0]

        def as4(t, S):  # the [batch, S, H, D] view of a packed [batch*S, H, D] tensor
            return t.as_strided((w.batch, S, H, 128), (S * t.stride(0), t.stride(0), t.stride(1), 1),
                                t.storage_offset())

    def run():
        if args.dense:
            st = va.varlen_attn_fwd_fp8_dense(as4(d.q, Sq), as4(d.k, Sk), as4(d.v, Sk), w.batch, Sq, Sk, H, 128,
                                              w.softmax_scale, causal, as4(out, Sq), lse, wsp, nbytes, stream)
        else:
            st = va.varlen_attn_fwd_fp8(d.q, d.k, d.v, d.cu_q, d.cu_k, w.batch, w.total_q, w.total_k, H, 128,
                                        w.max_q(), w.max_k(), w.softmax_scale, out, lse, wsp, nbytes, stream,
                                        causal=causal, window=window)
        assert st == 0, va.varlen_attn_status_string(st)

    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    assert va.varlen_attn_get_device_status(stream) == 0
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(ws)
    a.record(stream)
    for _ in range(args.steps):
        run()
    b.record(stream)
    torch.cuda.synchronize()
    ms = _max_over_ranks(a.elapsed_time(b), ws) / args.steps
    if rank == 0:
        mask = ("causal " if causal else "") + ("window(%d,%d) " % window if window != (-1, -1) else "")
        print(json.dumps({"metric": "E4M3 varlen attention forward TFLOP/s (%sbf16 FLOP count, quantisation "
                                    "included)" % mask,
                          "value": ws * w.fwd_flops(causal, window) / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                          "n_gpus": ws,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate)",
                          "data": "synthetic", "config": {"workload": w.name, "num_heads": H, "head_dim": 128,
                                                          "step": "fp8 fwd", "causal": causal, "window": list(window),
                                                          "entry": "dense batched" if args.dense else "packed varlen",
                                                          "l2": "inputs larger than L2 (k, v 2 GB each); no flush"},
                          "gpu_launches": 4 * args.steps}),
              flush=True)


def mma_rates(args):
    """Cycles per tcgen05 MMA (M = 128, K = 16, bf16 -> fp32) issued by one
    thread, for N = 64 / 128 / 256 and the three issue forms of
    varlen_attn_debug_mma_cycles (best of three runs of 4096 MMAs each)."""
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    dev = torch.device("cuda", 0)
    cyc = torch.zeros(1, dtype=torch.int64, device=dev)
    n = 4096
    res = {}
    for mode, name in ((0, "smem A, low-word descriptors"), (1, "TMEM A"), (2, "smem A, descriptors rebuilt per MMA"),
                       (5, "TMEM A, B MN-major"), (6, "TMEM A, four warps loading TMEM meanwhile"),
                       (7, "TMEM A, four warps storing to shared memory meanwhile")):
        for n_cols in ((64, 128) if mode == 5 else (128,) if mode >= 6 else (64, 128, 256)):
            best = None
            for _ in range(3):
                st = va.varlen_attn_debug_mma_cycles(n, n_cols, mode, cyc)
                assert st == 0, va.varlen_attn_status_string(st)
                torch.cuda.synchronize()
                assert va.varlen_attn_get_device_status() == 0
                v = int(cyc.item()) / n
                best = v if best is None else min(best, v)
            res["%s, N=%d" % (name, n_cols)] = {"cycles_per_mma": round(best, 2),
                                                "flops_per_cycle": round(2 * 128 * n_cols * 16 / best, 1)}
    for mode, name in ((3, "tcgen05.ld 32x32b.x32"), (4, "tcgen05.st 32x32b.x32")):
        best = None
        for _ in range(3):
            st = va.varlen_attn_debug_mma_cycles(n, 128, mode, cyc)
            assert st == 0, va.varlen_attn_status_string(st)
            torch.cuda.synchronize()
            assert va.varlen_attn_get_device_status() == 0
            v = int(cyc.item()) / n
            best = v if best is None else min(best, v)
        # four warps move 4 KB each per iteration
        res["%s, 4 warps, wait after each" % name] = {"cycles_per_iteration": round(best, 2),
                                                       "bytes_per_cycle": round(4 * 4096 / best, 1)}
    print(json.dumps({"probe": "tcgen05.mma issue rate, one CTA, one issuing thread; TMEM load/store rate",
                      "n_mma": n, "shape": "M=128, K=16, bf16 x bf16 -> fp32", "results": res}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="windowed", choices=sorted(W.WORKLOADS))
    ap.add_argument("--heads", type=int, default=None,
                    help="override the head count (small cases for profiling captures)")
    ap.add_argument("--causal", action="store_true",
                    help="time the causal entry points (FLOPs counted over visible pairs only)")
    ap.add_argument("--window", type=int, nargs=2, metavar=("LEFT", "RIGHT"), default=None,
                    help="time the sliding-window entry points with this band (a negative side is unbounded)")
    ap.add_argument("--deterministic", action="store_true",
                    help="time the deterministic backward (dQ without atomics, a second q-major kernel)")
    ap.add_argument("--dense", action="store_true",
                    help="drive the dense batched entry points (needs equal segment lengths, e.g. --workload dense)")
    ap.add_argument("--mma-rates", action="store_true",
                    help="print cycles per tcgen05 MMA for N = 64/128/256 and three issue forms (one CTA)")
    ap.add_argument("--fp8", action="store_true",
                    help="time the E4M3 forward alone (head size 128; with --causal / --window its banded form, "
                         "with --dense the dense batched entry point; quantisation included)")
    ap.add_argument("--shard", choices=["replicas", "heads"], default="replicas",
                    help="under torchrun: every rank a batch of its own (replicas, weak scaling) or one problem "
                         "split by heads across the ranks (strong scaling); no collective on the data path either way")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3  # timing rule: at least three warm-up steps
    w = W.get(args.workload)
    if args.heads is not None and args.heads != w.num_heads:
        w = w.with_(num_heads=args.heads, name="%s_h%d" % (w.name, args.heads))
    if args.impl == "reference":
        ws = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        reference_arm(args, w, ws, rank)
        return
    ws, rank, local = _dist()
    if args.mma_rates:
        if rank == 0:
            mma_rates(args)
        return
    if args.fp8:
        fp8_forward(args, w, ws, rank, local)
    else:
        ours(args, w, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
