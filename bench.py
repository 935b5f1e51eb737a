#!/usr/bin/env python
"""Throughput of the NAtS-L hybrid attention layer forward on GB300.

One step = one full layer forward (score + select, compaction, softmax
branch, Gated DeltaNet prep + scan with commit / rollback, RMSNorm + gated
merge) over one batch of the 1.3B-scale workload: B=4, H=16, L=8192,
d_k=d_v=128, chunk 64, bf16, 25 % softmax chunks chosen by the score layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

With N > 1 it runs under torchrun, one rank per GPU: every rank processes its
own batch (independent (b, h) units, no collective on the data path; weak
scaling) and rank 0 prints one JSON line with the max-over-ranks time.
`--impl reference` times the fp64 CPU oracle on a bounded sample of the same
workload on the host cores (rank 0 only).
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "hybrid-attn fwd tokens/s on 1 GB300 and % of tensor-core roofline (L=8192)"
WORKLOAD = "l8192"
WORKLOAD_DESC = ("NAtS-L layer forward, 1.3B-scale: B=4 H=16 L=8192 d_k=d_v=128 chunk=64, bf16 Q/K/V "
                 "~N(0,1) with unit keys, fp32 g/beta, 25% softmax chunks chosen by the score layer")
C = 64


def set_workload(name):
    """Another bf16 workload of the generator for the device-timed step."""
    global WORKLOAD, WORKLOAD_DESC
    import gen

    cfg = gen.CONFIGS[name]
    if cfg["dtype"] != "bf16":
        raise SystemExit(f"--workload {name}: the timed step is the bf16 path")
    WORKLOAD = name
    WORKLOAD_DESC = (f"NAtS-L layer forward, workload {name}: B={cfg['B']} H={cfg['H']} L={cfg['L']} "
                     f"d_k=d_v={cfg['d']} chunk=64, bf16 Q/K/V ~N(0,1) with unit keys, fp32 g/beta, "
                     f"selection pattern {cfg['pattern']!r}")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("native", "reference"), default="native")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-x-path", action="store_true", help="skip the layer-with-projections measurement")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode-step measurement")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward-pass measurement")
    ap.add_argument("--no-nha", action="store_true", help="skip the Native Hybrid Attention measurement")
    ap.add_argument("--no-select", action="store_true", help="skip the score-layer (nats_select) measurement")
    ap.add_argument("--decode-context", type=int, default=8192,
                    help="context length before the timed decode steps (a multiple of 64)")
    ap.add_argument("--workload", default="l8192",
                    help="layer workload of the device-timed step (default: the 8192-token one); others, e.g. "
                         "'long' (1 x 32 x 65536, 12.5 %% softmax chunks), are extra data points")
    return ap.parse_args()


# ---------------------------------------------------------------- peaks ----

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# GB300 nominal dense rates (context for the measured-peak fractions):
# bf16 tensor 2.25 PFLOP/s, HBM3e 7.9 TB/s.
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 7900.0


# ------------------------------------------------------- algorithmic work ----

def algorithmic_work(sel, B, H, L, d, in_bytes):
    """FLOPs of the dense contractions the method computes, from the actual selection.

    softmax: 4 d per (query, visible key) pair; pairs of chunk c =
      C^2 * nprev[c] + C (C + 1) / 2.
    Gated DeltaNet per chunk: 5 C^2 d (QK^T, KK^T, T.bV, T.bgK, P.Delta with
      triangular halves) + 6 C d^2 (W S^T, Q S^T, Delta^T K).
    """
    import numpy as np

    soft = (sel == 0).astype(np.int64)
    nprev = np.cumsum(soft, axis=-1) - soft
    N = sel.shape[-1]
    pairs = C * C * int(nprev.sum()) + B * H * N * C * (C + 1) // 2
    f_soft = 4 * d * pairs
    f_gdn = B * H * N * (5 * C * C * d + 6 * C * d * d)
    return {"flops_softmax": float(f_soft), "flops_gdn": float(f_gdn),
            "flops_total": float(f_soft + f_gdn), "bytes_io": float(in_bytes),
            "softmax_fraction": float(soft.mean())}


def kernel_work(B, H, L, d, flops_softmax):
    """Algorithmic work per launch of each stage, with the bound it is held to.

    softmax: 4 d FLOP per visible (query, key) pair (tensor-bound).  The
    others are HBM-bound; their bytes are the unique I/O the stage has to
    move (bf16 activations, fp32 g, beta, G, gate, o_l):
      gdn_prep per chunk: read Q, K, V, g, beta; write W, U^T (bf16 C x d
        each), P (bf16 C x C), gate and G;
      gdn_scan per chunk: read W, U^T, Q, K, P, G; write o_l (bf16 C x d);
      merge per row: read o_l (bf16), gate, out (bf16); write out;
      score per chunk: read Q, K (only when a separate score pass runs).
    The softmax kernel and the scan run concurrently on two streams, so
    their CUDA-event durations overlap and each includes time spent sharing
    the GPU with the other."""
    N = L // C
    chunks, rows = B * H * N, B * H * L
    prep = 3 * C * d * 2 + 2 * C * 4 + 2 * C * d * 2 + C * C * 2 + 2 * C * 4
    scan = 4 * C * d * 2 + C * C * 2 + C * 4 + C * d * 2
    return {
        "softmax": ("tensor", float(flops_softmax), "softmax_tc.cu"),
        "gdn_prep": ("hbm", float(chunks * prep), "gdn_prep_tc.cu" if d == 128 else "gdn_prep_mma.cu"),
        "gdn_scan": ("hbm", float(chunks * scan), "gdn_scan_tc.cu"),
        "merge": ("hbm", float(rows * (d * 2 + 4 + 2 * d * 2)), "merge.cu"),
        "score": ("hbm", float(chunks * 2 * C * d * 2), "select.cu"),
    }


def rooflines(work, stage_ms, pk):
    """Per-stage roofline objects (achieved = algorithmic work / CUDA-event time)."""
    out = {}
    for name, (bound, amount, src) in work.items():
        if name not in stage_ms:
            continue
        ms = stage_ms[name]
        if bound == "tensor":
            achieved, peak, unit = amount / (ms / 1e3) / 1e12, pk["bf16_tflops_sustained"], "TFLOP/s"
            peak_src, per = f"{pk['source']} bf16 sustained", {"flops_per_launch": amount}
        else:
            achieved, peak, unit = amount / (ms / 1e3) / 1e9, pk["hbm_gbs"], "GB/s"
            peak_src, per = f"{pk['source']} HBM copy", {"bytes_per_launch": amount}
        nominal = NOMINAL_BF16_TFLOPS if bound == "tensor" else NOMINAL_HBM_GBS
        out[name] = {"kernel": name, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "peak_source": peak_src, "frac_of_nominal": achieved / nominal,
                     "traffic": recorded_traffic(os.path.join(ROOT, "linear_attention_nats_gb300", "csrc", src)),
                     "ms_per_launch": ms, **per}
    return out


# --------------------------------------------------------------- clocks ----

class _NvmlSampler:
    """SM clock and clock-event reasons of one GPU, read through NVML (the
    driver's management library, read-only queries) every `period` seconds
    on a background thread: enough samples inside a timed region of tens of
    milliseconds.  Raises OSError where NVML cannot be loaded."""

    # clock-event reason bits (nvml.h)
    BITS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}

    def __init__(self, dev_index, period=0.002):
        import threading

        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        bus = None
        try:
            import torch

            pr = torch.cuda.get_device_properties(dev_index)
            bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
        except Exception:  # noqa: BLE001 (older torch: no PCI ids)
            bus = None
        rc = lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(self.h)) if bus else 1
        if rc != 0 and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(dev_index), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle")
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint(0)
        lib.nvmlDeviceGetMaxClockInfo(self.h, ctypes.c_int(1), ctypes.byref(mx))  # NVML_CLOCK_SM
        self.max_mhz = float(mx.value)
        self.rows = []
        self.period = period
        self.stop_ev = threading.Event()
        self.th = threading.Thread(target=self._run, daemon=True)
        self.th.start()

    def _run(self):
        mhz, bits = ctypes.c_uint(0), ctypes.c_ulonglong(0)
        while not self.stop_ev.is_set():
            if self.lib.nvmlDeviceGetClockInfo(self.h, ctypes.c_int(1), ctypes.byref(mhz)) == 0 and \
                    self.reasons_fn(self.h, ctypes.byref(bits)) == 0:
                self.rows.append((float(mhz.value), int(bits.value)))
            time.sleep(self.period)

    def stop(self):
        self.stop_ev.set()
        self.th.join(timeout=5)
        self.lib.nvmlShutdown()
        if not self.rows:
            return None
        reasons = sorted({name for _, b in self.rows for bit, name in self.BITS.items() if b & bit})
        return {"sm_mhz": statistics.median(r[0] for r in self.rows), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.rows), "source": "nvml, every 2 ms"}


class Clocks:
    """Clock record of a timed region: NVML sampled on a thread where the
    library loads, else nvidia-smi every 100 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, enabled=True):
        self.proc = None
        self.nvml = None
        self.path = os.path.join("/tmp", f"nats_clocks_{os.getpid()}.csv")
        if not enabled:
            return
        try:
            self.nvml = _NvmlSampler(gpu_index)
            return
        except (OSError, AttributeError):
            self.nvml = None
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(gpu_index)], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.nvml is not None:
            return self.nvml.stop()
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "source": "nvidia-smi, every 100 ms"}


# ------------------------------------------------------------ traffic ----

def recorded_traffic(kernel_src, workload=None):
    """DRAM bytes per launch of a kernel from the committed ncu summaries, valid
    only while the kernel's source file is unchanged (hash match)."""
    workload = workload or WORKLOAD
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    h = hashlib.sha256(open(kernel_src, "rb").read()).hexdigest()[:16]
    for line in open(path):
        kv = dict(x.split("=", 1) for x in line.split() if "=" in x)
        if kv.get("src") == os.path.basename(kernel_src) and kv.get("sha") == h and kv.get("workload") == workload:
            return float(kv["dram_bytes_per_launch"])
    return None


# ------------------------------------------------------------- oracle ----

def oracle_sample(inp, n_heads, threads):
    """Wall time of the oracle on the first n_heads (b, h) heads, all rows."""
    import oracle

    oracle.build()
    heads = list(range(n_heads))
    t0 = time.perf_counter()
    r = oracle.forward_inputs(inp, heads=heads, outputs=("out",), threads=threads)
    dt = time.perf_counter() - t0
    return dt, r["threads"]


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------- ranks ----

def rank_seed(seed, rank):
    """Every rank draws its own batch: the (b, h) units are independent, so the
    ranks share nothing on the data path (weak scaling)."""
    return seed + 1000 * rank


def max_over_ranks(x, dist, device):
    """The slowest rank's value (the job ends when its last rank does)."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank, world, ms_per_step):
    """Whole-job tokens/s: every rank's tokens over the max-over-ranks step time."""
    return tokens_per_rank * world / (ms_per_step / 1e3)


# -------------------------------------------------------------- arms ----

def run_reference(args, rank):
    """The oracle on the host cores: each step is n heads (one per core) of the workload."""
    if rank != 0:
        return None
    import gen

    inp = gen.config_inputs(WORKLOAD)
    cores = cpu_cores()
    n = min(cores, inp.B * inp.H)
    for _ in range(args.warmup):
        oracle_sample(inp, n, cores)
    times = []
    used = cores
    for _ in range(args.steps):
        dt, used = oracle_sample(inp, n, cores)
        times.append(dt)
    total = sum(times)
    tokens_per_step = n * inp.L / inp.H  # n of the B*H (b, h) head-rows of L tokens
    value = tokens_per_step * args.steps / total
    sample = f"{n} of {inp.B * inp.H} (b,h) heads, all {inp.L} rows, per step"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_native(args, rank, world, local_rank):
    import numpy as np
    import torch

    import gen
    import linear_attention_nats_gb300 as nats
    from linear_attention_nats_gb300 import _native

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    cfg = dict(gen.CONFIGS[WORKLOAD])
    cfg["seed"] = rank_seed(cfg["seed"], rank)
    inp = gen.make_inputs(name=WORKLOAD, **cfg)
    B, H, L, d = inp.B, inp.H, inp.L, inp.d
    N = L // C

    host = {}
    for n in ("q", "k", "v"):
        host[n] = torch.from_numpy(getattr(inp, n)).to(torch.bfloat16)  # exact: values are bf16
    for n in ("g", "beta", "w_s", "b_s", "w_g", "b_g"):
        host[n] = torch.from_numpy(np.ascontiguousarray(getattr(inp, n)))
    dv = {n: t.to(dev) for n, t in host.items()}
    out = torch.empty_like(dv["q"])
    sel = torch.empty((B, H, N), dtype=torch.uint8, device=dev)
    dm = nats.dims(B, H, L, d, nats.NATS_BF16)
    ws_bytes = int(_native.lib.nats_workspace_size(ctypes.byref(dm)))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    P = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None

    def call(tensors, prof=None, out_t=None):
        # on the current stream (a graph capture makes its own stream current)
        code = _native.lib.nats_hybrid_fwd_profiled(
            ctypes.byref(dm), P(tensors["q"]), P(tensors["k"]), P(tensors["v"]), P(tensors["g"]),
            P(tensors["beta"]), P(tensors["w_s"]), P(tensors["b_s"]), P(tensors["w_g"]), P(tensors["b_g"]),
            None, None, None, P(out if out_t is None else out_t), P(sel), None, None, None, P(ws),
            ctypes.c_size_t(ws_bytes),
            ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream),
            ctypes.byref(prof) if prof is not None else None)
        if code != 0:
            raise _native.NatsError(code, "nats_hybrid_fwd_profiled")

    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(max(args.warmup, 0)):
        call(dv)
    torch.cuda.synchronize()
    sel_h = sel.cpu().numpy()
    in_bytes = sum(t.numel() * t.element_size() for n, t in dv.items() if n in ("q", "k", "v", "g", "beta")) \
        + out.numel() * out.element_size()
    work = algorithmic_work(sel_h, B, H, L, d, in_bytes)

    # ---- device-resident timed region: K back-to-back steps, as one CUDA
    # graph (captured once, outside the timed region: every step's kernels,
    # each on the step's full work, replayed back to back without host
    # launch gaps; inputs larger than L2) ----
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(args.steps):
            call(dv)
    torch.cuda.synchronize()
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = Clocks(local_rank, enabled=not args.no_clocks and rank == 0)
    barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    graph.replay()
    t_stop.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = t_start.elapsed_time(t_stop)
    del graph
    # ---- the same K steps called one by one with per-stage events (stage
    # times and launch counts; the events themselves add ~15 us a step, so
    # this pass is not the headline) ----
    stage_ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in _native.STAGES] for _ in range(args.steps)]
    for row in stage_ev:  # materialise the event handles
        for a, b in row:
            a.record(stream)
            b.record(stream)
    profs = []
    for row in stage_ev:
        p = _native.Profile()
        for i, (a, b) in enumerate(row):
            p.start[i] = a.cuda_event
            p.stop[i] = b.cuda_event
        profs.append(p)
    torch.cuda.synchronize()
    for i in range(args.steps):
        call(dv, profs[i])
    torch.cuda.synchronize()
    launches = sum(p.launches for p in profs)  # the kernels the graph replays in the timed region
    stage_ms = {}
    for si, name in enumerate(_native.STAGES):
        if profs[0].stage_launches[si] == 0:  # the path does not run this stage
            continue
        vals = [row[si][0].elapsed_time(row[si][1]) for row in stage_ev]
        stage_ms[name] = sum(vals) / len(vals)
    ms = max_over_ranks(ms, dist, dev)
    ms_step = ms / args.steps
    tokens = B * L * world
    value = job_throughput(B * L, world, ms_step)

    # ---- end to end: pinned host buffers in, result out, copies timed ----
    # Every step copies its own inputs from pinned host memory and reads its
    # output back.  As in an input pipeline, the copy of step i + 1's inputs
    # (copy stream) overlaps step i's layer (compute stream), and step i's
    # output read (third stream) overlaps step i + 1; two staging sets.
    e2e = None
    if not args.no_e2e:
        pin = {n: t.pin_memory() for n, t in host.items()}
        out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in pin.values())
        d2h = out_h[0].numel() * out_h[0].element_size()
        staged = [{n: torch.empty_like(t) for n, t in dv.items()} for _ in range(2)]
        outs = [torch.empty_like(out) for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev = lambda: torch.cuda.Event()

        def run_e2e(n_steps):
            h2d_done = [ev() for _ in range(n_steps)]
            comp_done = [ev() for _ in range(n_steps)]
            d2h_done = [ev() for _ in range(n_steps)]
            for i in range(n_steps):
                j = i & 1
                with torch.cuda.stream(s_in):  # inputs of step i (set j free once step i - 2 ran)
                    if i >= 2:
                        s_in.wait_event(comp_done[i - 2])
                    for n in pin:
                        staged[j][n].copy_(pin[n], non_blocking=True)
                    h2d_done[i].record(s_in)
                stream.wait_event(h2d_done[i])
                if i >= 2:
                    stream.wait_event(d2h_done[i - 2])  # output set j has been read back
                call(staged[j], out_t=outs[j])
                comp_done[i].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(comp_done[i])
                    out_h[j].copy_(outs[j], non_blocking=True)
                    d2h_done[i].record(s_out)
            return d2h_done[-1]

        run_e2e(3)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        e0.record(s_in)
        s_in.wait_event(e0)
        last = run_e2e(args.steps)
        s_out.wait_event(last)
        e1.record(s_out)
        torch.cuda.synchronize()
        barrier()
        ems = e0.elapsed_time(e1)
        ems = max_over_ranks(ems, dist, dev)
        # the host link alone: one step's input copies with an output read
        # back at the same time and nothing else, the floor of an e2e step
        link_ms = float("inf")
        for _ in range(3):
            l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            l0.record(s_in)
            s_out.wait_event(l0)
            with torch.cuda.stream(s_in):
                for n in pin:
                    staged[0][n].copy_(pin[n], non_blocking=True)
            with torch.cuda.stream(s_out):
                out_h[0].copy_(outs[0], non_blocking=True)
                o_done = ev()
                o_done.record(s_out)
            s_in.wait_event(o_done)
            l1.record(s_in)
            torch.cuda.synchronize()
            link_ms = min(link_ms, l0.elapsed_time(l1))
        link_ms = max_over_ranks(link_ms, dist, dev)
        e2e_ms = ems / args.steps
        e2e = {"value": tokens / (e2e_ms / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "pipeline": "step i + 1's input copy and step i - 1's output read overlap step i's layer",
               "host_link": {"ms_per_step": link_ms, "h2d_gbs": h2d / (link_ms / 1e3) / 1e9,
                             "frac": link_ms / e2e_ms,
                             "what": "the step's input copies and an output read-back alone (no layer): "
                                     "the floor of an e2e step on this host link"}}
        launches_e2e = None  # noqa: F841 (counted in gpu_launches only for the device-timed region)

    pk = peaks()
    peak_tc = pk["bf16_tflops_sustained"]
    per_kernel = rooflines(kernel_work(B, H, L, d, work["flops_softmax"]), stage_ms, pk)
    dominant = max(per_kernel, key=lambda k: per_kernel[k]["ms_per_launch"])
    roofline = per_kernel[dominant]
    layer_tflops = work["flops_total"] / (ms_step / 1e3) / 1e12 / world
    res = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC, "global_batch": B * world, "seq_len": L,
                   "parallelism": f"replicas x{world} ((b,h) units per rank, no collective)",
                   "l2": f"inputs larger than L2: Q/K/V {3 * B * H * L * d * 2 / 2**20:.0f} MiB + workspace per step, "
                         "no explicit flush",
                   "timed": f"{args.steps} steps of nats_hybrid_fwd captured once in a CUDA graph and replayed (every "
                            "kernel of every step); stage times from the same steps called one by one with events",
                   "softmax_fraction": work["softmax_fraction"]},
        "roofline": roofline,
        "kernel_rooflines": per_kernel,
        "layer_roofline": {"bound": "tensor", "achieved": layer_tflops, "peak": peak_tc,
                           "unit": "TFLOP/s", "frac": layer_tflops / peak_tc,
                           "frac_of_burst": layer_tflops / pk["bf16_tflops"],
                           "frac_of_nominal": layer_tflops / NOMINAL_BF16_TFLOPS,
                           "what": "the whole step (all kernels) against the bf16 tensor peak; `roofline` is the "
                                   "dominant kernel's",
                           "flops_per_step": work["flops_total"]},
        "stages_ms": stage_ms,
        "gpu_launches": launches,
        "e2e": e2e,
        "clocks": clk,
    }
    # ---- the layer with its projections (nats_hybrid_fwd_x), same shapes,
    # hidden = H d = 2048: tokens/s of the whole model layer ----
    if not args.no_x_path:
        res["x_path"] = run_x_path(args, rank, dev, stream, dist)
    if not args.no_decode:
        res["decode"] = run_decode(args, rank, dev, stream, dist)
    if not args.no_backward:
        res["backward"] = run_backward(args, dev, stream, dist, dv, B, H, L, d, work)
    if not args.no_nha:
        res["nha"] = run_nha(args, rank, dev, stream, dist)
    if not args.no_select:
        res["select"] = run_select(args, dev, stream, dist, dv, B, H, L, d)
    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1 only) ----
    if not args.no_cpu_baseline and world == 1 and rank == 0:
        cores = cpu_cores()
        n = min(2 * cores, B * H)
        dt, used = oracle_sample(inp, n, cores)
        res["cpu_baseline"] = {"value": n * L / H / dt, "unit": "tokens/s", "cores": used, "kind": "oracle",
                               "sample": f"{n} of {B * H} (b,h) heads of the workload, all {L} rows "
                                         f"({dt:.1f} s wall)"}
    return res


def run_x_path(args, rank, dev, stream, dist):
    """Times nats_hybrid_fwd_x: x [B, L, hidden] -> y, through the C ABI, inputs
    resident in HBM (K steps after warm-up, CUDA events, max over ranks)."""
    import numpy as np
    import torch

    import gen
    import linear_attention_nats_gb300 as nats
    from linear_attention_nats_gb300 import _native

    cfg = dict(gen.X_CONFIGS["x_l8192"])
    cfg["seed"] = rank_seed(cfg["seed"], rank)
    xi = gen.make_x_inputs(name="x_l8192", **cfg)

    def bf(a):
        return torch.from_numpy(gen.bf16_bits(np.ascontiguousarray(a, np.float32)).view(np.int16)).view(
            torch.bfloat16).to(dev)

    def f(a):
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)

    B, H, L, d, hidden = xi.B, xi.H, xi.L, xi.d, xi.hidden
    t = dict(x=bf(xi.x), w_qkv=bf(xi.w_qkv), w_ab=bf(xi.w_ab), w_o=bf(xi.w_o), b_a=f(xi.b_a),
             a_scale=f(xi.a_scale), b_b=f(xi.b_b), w_s=f(xi.w_s), b_s=f(xi.b_s), w_g=f(xi.w_g), b_g=f(xi.b_g))
    y = torch.empty((B, L, hidden), dtype=torch.bfloat16, device=dev)
    sel = torch.empty((B, H, L // 64), dtype=torch.uint8, device=dev)  # the chunks the score layer chose
    dm = nats.dims(B, H, L, d, nats.NATS_BF16)
    wsb = int(_native.lib.nats_x_workspace_size(ctypes.byref(dm), hidden))
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    P = lambda v: ctypes.c_void_p(v.data_ptr())

    def call(prof=None):
        code = _native.lib.nats_hybrid_fwd_x_profiled(
            ctypes.byref(dm), hidden, P(t["x"]), P(t["w_qkv"]), P(t["w_ab"]), P(t["b_a"]), P(t["a_scale"]),
            P(t["b_b"]), P(t["w_s"]), P(t["b_s"]), P(t["w_g"]), P(t["b_g"]), P(t["w_o"]), P(y), P(sel), P(ws),
            ctypes.c_size_t(wsb), ctypes.c_void_p(stream.cuda_stream),
            ctypes.byref(prof) if prof is not None else None)
        if code != 0:
            raise _native.NatsError(code, "nats_hybrid_fwd_x_profiled")

    for _ in range(max(args.warmup, 1)):
        call()
    torch.cuda.synchronize()
    # per-stage events of every timed step (the two projection GEMMs among them)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in _native.STAGES] for _ in range(args.steps)]
    profs = []
    for row in ev:
        p = _native.Profile()
        for i, (a0, a1) in enumerate(row):
            a0.record(stream)
            a1.record(stream)
            p.start[i] = a0.cuda_event
            p.stop[i] = a1.cuda_event
        profs.append(p)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(args.steps):
        call(profs[i])
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), dist, dev) / args.steps
    world = dist.get_world_size() if dist is not None else 1
    stage_ms = {}
    for si, name in enumerate(_native.STAGES):
        if profs[0].stage_launches[si] == 0:
            continue
        vals = [row[si][0].elapsed_time(row[si][1]) for row in ev]
        stage_ms[name] = sum(vals) / len(vals)
    f_in = 2.0 * B * L * hidden * (3 * H * d + 2 * H)
    f_out = 2.0 * B * L * H * d * hidden
    pk = peaks()
    peak = pk["bf16_tflops_sustained"]
    gemms = {}
    for name, fl in (("proj_in", f_in), ("proj_out", f_out)):
        if name in stage_ms:
            ach = fl / (stage_ms[name] / 1e3) / 1e12
            gemms[name] = {"kernel": "gemm_tc_kernel", "bound": "tensor", "achieved": ach, "peak": peak,
                           "unit": "TFLOP/s", "frac": ach / peak, "peak_source": f"{pk['source']} bf16 sustained",
                           "ms_per_launch": stage_ms[name], "flops_per_launch": fl,
                           "traffic": recorded_traffic(os.path.join(ROOT, "linear_attention_nats_gb300", "csrc",
                                                                    "gemm_tc.cu"), f"x_l8192_{name}")}
    dom = max(gemms, key=lambda k: gemms[k]["ms_per_launch"]) if gemms else None
    return {"what": "nats_hybrid_fwd_x: x -> q, k, v, g, beta (tcgen05 GEMM, head split + key norm + gates in "
                    "its epilogue), the layer, output projection (the same GEMM kernel)",
            "config": {"B": B, "H": H, "L": L, "d": d, "hidden": hidden,
                       # random projections and score weights with zero bias: the score layer's own
                       # choice, near half the chunks (the layer leg fixes 25 % by its inputs)
                       "softmax_chunk_frac": float((sel == 0).float().mean().item())},
            "value": job_throughput(B * L, world, ms), "unit": "tokens/s", "ms_per_step": ms,
            "stages_ms": stage_ms, "projection_gemm_flops_per_step": f_in + f_out,
            "roofline": gemms.get(dom), "gemm_rooflines": gemms}


def run_select(args, dev, stream, dist, dv, B, H, L, d):
    """Times nats_select (the Attention Score Layer alone: chunk mean pool of
    [q; k], the linear score, the argmax; score_kernel) on the layer
    workload's Q and K, inputs resident in HBM.  HBM-bound: it reads Q and K
    once (the bf16 layer forward takes its selection inside the chunk-factor
    kernel instead)."""
    import torch

    from linear_attention_nats_gb300 import _native

    N = L // C
    dm = _native.dims(B, H, L, d, _native.NATS_BF16)
    sel = torch.empty((B, H, N), dtype=torch.uint8, device=dev)
    P = lambda t: ctypes.c_void_p(t.data_ptr())

    def call():
        code = _native.lib.nats_select(ctypes.byref(dm), P(dv["q"]), P(dv["k"]), P(dv["w_s"]), P(dv["b_s"]), P(sel),
                                       None, ctypes.c_void_p(stream.cuda_stream))
        if code != 0:
            raise _native.NatsError(code, "nats_select")

    for _ in range(max(args.warmup, 1)):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), dist, dev) / args.steps
    nbytes = 2.0 * B * H * L * d * 2 + B * H * N
    pk = peaks()
    ach = nbytes / (ms / 1e3) / 1e9
    return {"what": "nats_select (score_kernel): mean pool + linear score + argmax per 64-token chunk",
            "ms_per_launch": ms,
            "roofline": {"kernel": "score_kernel", "bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"],
                         "unit": "GB/s", "frac": ach / pk["hbm_gbs"], "peak_source": f"{pk['source']} HBM copy",
                         "bytes_per_launch": nbytes,
                         "traffic": recorded_traffic(os.path.join(ROOT, "linear_attention_nats_gb300", "csrc",
                                                                  "select.cu"))}}


def nha_work(B, H, L, d, m, w):
    """Algorithmic FLOPs of the NHA layer (tensor-core work of its plain
    definition): per query 4 d per window key (q.k and p v) and, once a token
    has left the window, 4 d per slot (q.K~ and p V~); per token written into
    the slots 4 m d (the gated update of K~ and V~)."""
    import numpy as np

    t = np.arange(L)
    pairs = np.minimum(t + 1, max(w, 0)).sum() if w > 0 else 0
    n_slot = max(L - w, 0)
    attn = 4.0 * d * (pairs + m * n_slot)
    state = 4.0 * m * d * n_slot
    # the slot-memory stage is bound by HBM: per chunk the gate kernel reads
    # the log-gates (fp32 C x m) and writes E' (fp32), G' and Gamma (bf16)
    # and e^{A_r}, e^{A_63}; the scan reads K and V (bf16 C x d), Gamma and
    # e^{A_r}, e^{A_63} once per memory and writes S0''^T and V0''^T (bf16
    # d x m)
    C = 64
    chunks = B * H * (L // C) if w < L else 0
    gate_b = C * m * 4 + C * m * (4 + 2 + 2) + 2 * m * 4
    scan_b = 2 * C * d * 2 + 2 * (C * m * 2 + 2 * m * 4) + 2 * d * m * 2
    return {"attn": B * H * attn, "state": B * H * state, "state_bytes": float(chunks * (gate_b + scan_b))}


def run_nha(args, rank, dev, stream, dist):
    """Times nats_nha_fwd (Native Hybrid Attention: one softmax over 64 slots
    and a 512-token window) at the 1.3B-scale layer shape (B = 4, H = 16,
    L = 8192, d = 128), inputs resident in HBM, K steps after warm-up."""
    import numpy as np
    import torch

    import gen
    import linear_attention_nats_gb300 as nats
    from linear_attention_nats_gb300 import _native

    cfg = dict(gen.NHA_CONFIGS["nha_l8192"])
    cfg["seed"] = rank_seed(cfg["seed"], rank)
    inp = gen.make_nha_inputs(name="nha_l8192", **cfg)
    B, H, L, d, m, w = inp.B, inp.H, inp.L, inp.d, inp.m, inp.window

    def bf(a):
        return torch.from_numpy(gen.bf16_bits(np.ascontiguousarray(a, np.float32)).view(np.int16)).view(
            torch.bfloat16).to(dev)

    q, k, v = bf(inp.q), bf(inp.k), bf(inp.v)
    la = torch.from_numpy(np.ascontiguousarray(inp.log_alpha)).to(dev)
    out = torch.empty_like(q)
    dm = _native.nha_dims(B, H, L, d, m, w)
    wsb = int(_native.lib.nats_nha_workspace_size(ctypes.byref(dm)))
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    P = lambda t: ctypes.c_void_p(t.data_ptr())

    def call(prof=None):
        code = _native.lib.nats_nha_fwd_profiled(ctypes.byref(dm), P(q), P(k), P(v), P(la), P(out), P(ws),
                                                 ctypes.c_size_t(wsb), ctypes.c_void_p(stream.cuda_stream),
                                                 ctypes.byref(prof) if prof is not None else None)
        if code != 0:
            raise _native.NatsError(code, "nats_nha_fwd_profiled")

    for _ in range(max(args.warmup, 1)):
        call()
    torch.cuda.synchronize()
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(2)]
          for _ in range(args.steps)]
    profs = []
    for row in ev:
        p = _native.Profile()
        for i, (a0, a1) in enumerate(row):
            a0.record(stream)
            a1.record(stream)
            p.start[i] = a0.cuda_event
            p.stop[i] = a1.cuda_event
        profs.append(p)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(args.steps):
        call(profs[i])
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), dist, dev) / args.steps
    world = dist.get_world_size() if dist is not None else 1
    kms = {name: sum(row[i][0].elapsed_time(row[i][1]) for row in ev) / len(ev)
           for i, name in enumerate(("nha_state", "nha_attn")) if profs[0].stage_launches[i]}
    fl = nha_work(B, H, L, d, m, w)
    pk = peaks()
    peak = pk["bf16_tflops_sustained"]
    rl = {}
    src = os.path.join(ROOT, "linear_attention_nats_gb300", "csrc", "nha.cu")
    if "nha_attn" in kms:
        ach = fl["attn"] / (kms["nha_attn"] / 1e3) / 1e12
        rl["nha_attn"] = {"kernel": "nha_attn_kernel", "bound": "tensor", "achieved": ach, "peak": peak,
                          "unit": "TFLOP/s", "frac": ach / peak, "peak_source": f"{pk['source']} bf16 sustained",
                          "ms_per_launch": kms["nha_attn"], "flops_per_launch": fl["attn"],
                          "traffic": recorded_traffic(src, "nha_l8192_nha_attn")}
    if "nha_state" in kms:
        gbs = fl["state_bytes"] / (kms["nha_state"] / 1e3) / 1e9
        rl["nha_state"] = {"kernel": "nha_gate_kernel + nha_state_kernel", "bound": "hbm", "achieved": gbs,
                           "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": gbs / pk["hbm_gbs"],
                           "peak_source": f"{pk['source']} HBM copy", "ms_per_stage": kms["nha_state"],
                           "bytes_per_stage": fl["state_bytes"], "flops_per_stage": fl["state"],
                           "traffic": recorded_traffic(src, "nha_l8192_nha_state")}
    tot = fl["attn"] + fl["state"]
    return {"what": "nats_nha_fwd: Native Hybrid Attention (reading CONV-16), 64 slots + a 512-token window under "
                    "one softmax; chunk-parallel gate factors, the slot-memory scan (tcgen05 writes, two CTAs "
                    "per head), then the attention (tcgen05, persistent)",
            "config": {"B": B, "H": H, "L": L, "d": d, "slots": m, "window": w},
            "value": job_throughput(B * L, world, ms), "unit": "tokens/s", "ms_per_step": ms,
            "kernels_ms": kms, "flops_per_step": tot,
            "layer_roofline": {"bound": "tensor", "achieved": tot / (ms / 1e3) / 1e12, "peak": peak,
                               "unit": "TFLOP/s", "frac": tot / (ms / 1e3) / 1e12 / peak},
            "roofline": rl.get("nha_attn"), "kernel_rooflines": rl,
            "gpu_launches": sum(p.launches for p in profs)}


def run_backward(args, dev, stream, dist, dv, B, H, L, d, work):
    """Times nats_hybrid_bwd on the layer workload: the gradients of a seeded
    dout at the forward's selection, from the activations the CUDA forward
    saved (one forward outside the timed region, which also saves the softmax
    rows' log-sum-exp for a bf16 layer).  Its stages are timed with
    the library's own stage events (softmax_bwd on the caller's stream and
    gdn_bwd on the library's second stream run side by side, so their times
    overlap and the shares add up to more than one) and set against the
    roofline of their own kind of work:
      merge_bwd     HBM: per token it reads q, dout (bf16) and o_soft, o_lin
                    (fp32) and writes d o_soft (bf16), d o_lin, dq (fp32) and
                    delta: 22 d + 4 bytes;
      softmax_bwd   bf16 tensor (tcgen05): 10 d FLOP per visible (query,
                    key) pair (scores recomputed, dP, dq, dk, dv; the row
                    log-sum-exp comes from the forward), plus the compaction
                    of the softmax-chunk lists;
      gdn_bwd       bf16 / fp16 tensor: per chunk the forward's chunk factors
                    and scan that recompute the chunk start states (5 C^2 d +
                    6 C d^2 FLOP, the forward's count, on tcgen05), the
                    adjoint's chunk factors (2 x 4 C^2 d) and reverse scan
                    (2 x 3 C d^2; warp-level mma.sync, fp16 operands);
      gdn_products  HBM: the adjoint's per-chunk products in one kernel (on
                    tcgen05 for d = 128) read S0 and dS_C (fp32 d x d each),
                    q, k, v (bf16), dO (fp32), Linv and P (fp32 C x C),
                    update dq, dk, dv (fp32) and write dg, dbeta: 8 d^2 +
                    34 C d + 8 C^2 + 8 C bytes per chunk (its 2 (5 C d^2 +
                    10 C^2 d) FLOP are a few percent of the tensor peak).
    The headline roofline is the stage with the largest share of the time."""
    import torch

    import linear_attention_nats_gb300 as nats
    from linear_attention_nats_gb300 import _native

    t = dv
    tc_layer = t["q"].dtype == torch.bfloat16
    fwd = nats.hybrid_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_s"], t["b_s"], t["w_g"], t["b_g"],
                          return_sel=True, return_branches=True, return_lse=tc_layer, stream=stream)
    gen_ = torch.Generator(device="cpu").manual_seed(43)
    dout = torch.randn((B, H, L, d), generator=gen_).to(t["q"].dtype).to(dev)
    dm = nats.dims(B, H, L, d, 0 if t["q"].dtype == torch.bfloat16 else 1)
    ws = torch.empty(int(nats._native.lib.nats_bwd_workspace_size(ctypes.byref(dm))), dtype=torch.uint8, device=dev)
    ns = len(_native.BWD_STAGES)

    def step(prof=None):
        return nats.hybrid_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["w_g"], t["b_g"], fwd["sel"],
                               fwd["o_soft"], fwd["o_lin"], dout, workspace=ws, stream=stream, profile=prof,
                               lse=fwd.get("lse"))

    steps = max(1, min(args.steps, 3))
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    stage_ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(ns)]
                for _ in range(steps)]
    for row in stage_ev:  # materialise the event handles
        for a, b in row:
            a.record(stream)
            b.record(stream)
    profs = []
    for row in stage_ev:
        pr = _native.Profile()
        for i, (a, b) in enumerate(row):
            pr.start[i] = a.cuda_event
            pr.stop[i] = b.cuda_event
        profs.append(pr)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = Clocks(torch.cuda.current_device(), enabled=not args.no_clocks)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for i in range(steps):
            step(profs[i])
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), dist, dev) / steps
    world = dist.get_world_size() if dist is not None else 1
    stage_ms = {name: sum(r[i][0].elapsed_time(r[i][1]) for r in stage_ev) / steps
                for i, name in enumerate(_native.BWD_STAGES)}
    pk = peaks()
    tokens = B * H * L
    pairs = work["flops_softmax"] / (4 * d)
    Cc = 64
    chunks = B * H * (L // Cc)
    amounts = {"merge_bwd": ("hbm", (22 * d + 4) * tokens, stage_ms["merge_bwd"]),
               "softmax_bwd": ("tensor", 10 * d * pairs, stage_ms["softmax_bwd"]),
               "gdn_bwd": ("tensor", chunks * (5 * Cc * Cc * d + 6 * Cc * d * d + 2 * (4 * Cc * Cc * d + 3 * Cc * d * d)),
                           stage_ms["gdn_bwd"]),
               "gdn_products": ("hbm", chunks * (8 * d * d + 34 * Cc * d + 8 * Cc * Cc + 8 * Cc),
                                stage_ms["gdn_products"])}
    per = {}
    for name, (bound, amount, sms) in amounts.items():
        if bound == "hbm":
            ach, peak, unit, src = amount / (sms / 1e3) / 1e9, pk["hbm_gbs"], "GB/s", f"{pk['source']} HBM copy"
        else:
            ach, peak, unit = amount / (sms / 1e3) / 1e12, pk["bf16_tflops_sustained"], "TFLOP/s"
            src = f"{pk['source']} bf16 sustained" + (" (tcgen05)" if name == "softmax_bwd" else
                                                      " (tcgen05 recompute; fp16 mma.sync adjoint factors and scan)")
        per[name] = {"bound": bound, "ms": sms, "share": sms / ms if ms else None, "achieved": ach, "peak": peak,
                     "unit": unit, "frac": (ach / peak) if peak else None, "peak_source": src,
                     ("bytes_per_step" if bound == "hbm" else "flops_per_step"): amount}
    top = max(per, key=lambda n: per[n]["ms"])
    return {"what": "nats_hybrid_bwd: gradients of q, k, v, g, beta, W_g, b_g and the RMSNorm weights at the "
                    "forward's selection, same workload as the forward",
            "value": job_throughput(B * L, world, ms), "unit": "tokens/s", "ms_per_step": ms, "steps": steps,
            "launches_per_step": int(profs[0].launches), "stages_ms": stage_ms,
            "stages_overlap": "softmax_bwd (caller's stream) and gdn_bwd (second stream) run side by side",
            "stages": per, "clocks": clk,
            "roofline": {"kernel": top, **{k: per[top][k] for k in ("bound", "achieved", "peak", "unit", "frac",
                                                                   "peak_source")}}}


def run_decode(args, rank, dev, stream, dist):
    """Times nats_decode_step after a T-token context (--decode-context,
    default 8192; B = 4, H = 16, d = 128, bf16, 25 % of the context's chunks
    retained: T / 4 keys / values per head): K steps at positions following
    the warm-up steps, captured in
    a CUDA graph and replayed (device time, CUDA events, max over ranks), as
    a serving loop would run them; the same steps issued one call at a time
    from Python are reported beside it (host-bound).  The steps go through
    the states of four layers in turn, as a model's layers would, so that a
    step's state and keys (76 MB) are not in L2 from the step before (the
    four together, 304 MB, are larger than L2).  The states and the retained
    keys / values are seeded synthetic values of the right shapes."""
    import torch

    import linear_attention_nats_gb300 as nats

    B, H, d, NL = 4, 16, 128, 4
    t0 = args.decode_context
    kept = t0 // 4
    g_ = torch.Generator(device="cpu").manual_seed(rank_seed(41, rank))
    nw = max(args.warmup, NL)
    K = max(args.steps, 32)  # steps per timed region: the graph's launch spread over enough of them
    steps_all = nw + 2 * K
    cap = 64 * ((t0 + steps_all // NL) // 64 + 1)
    rn = lambda *shape: torch.randn(*shape, generator=g_)
    states = []
    # the retained keys / values are drawn once and copied into every layer's state
    kv_k = torch.nn.functional.normalize(rn(B, H, kept, d), dim=-1).to(torch.bfloat16).to(dev)
    kv_v = rn(B, H, kept, d).to(torch.bfloat16).to(dev)
    for _ in range(NL):
        st = nats.DecodeState(B, H, d, cap=cap, dtype=torch.bfloat16, device=dev)
        st.S.copy_(0.05 * rn(B, H, d, d))
        st.S0.copy_(st.S)
        st.kv_k[:, :, :kept].copy_(kv_k)
        st.kv_v[:, :, :kept].copy_(kv_v)
        st.n_kv.fill_(kept)
        states.append(st)
    del kv_k, kv_v
    q = rn(steps_all, B, H, d).to(torch.bfloat16).to(dev)
    k = torch.nn.functional.normalize(rn(steps_all, B, H, d), dim=-1).to(torch.bfloat16).to(dev)
    v = rn(steps_all, B, H, d).to(torch.bfloat16).to(dev)
    g = (-0.1 * torch.nn.functional.softplus(rn(steps_all, B, H))).to(dev)
    beta = torch.sigmoid(rn(steps_all, B, H)).to(dev)
    w_s = (0.02 * rn(H, 2, 2 * d)).to(dev)
    b_s = torch.zeros(H, 2).to(dev)
    w_g = (0.02 * rn(H, d)).to(dev)
    b_g = torch.zeros(H).to(dev)
    out = torch.empty((B, H, d), dtype=torch.bfloat16, device=dev)

    def step(i, s=None):  # step i: layer i % NL at position t0 + i // NL
        nats.decode_step(states[i % NL], t0 + i // NL, q[i], k[i], v[i], g[i], beta[i], w_s, b_s, w_g, b_g,
                         out=out, stream=s)

    with torch.cuda.stream(stream):
        for i in range(nw):
            step(i)
    torch.cuda.synchronize()
    # one call at a time from Python (host-bound)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record()
        for i in range(K):
            step(nw + i)
        e1.record()
    torch.cuda.synchronize()
    host_ms = e0.elapsed_time(e1) / K
    # the next K steps as one CUDA graph
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(K):
            step(nw + K + i)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), dist, dev) / K
    for st in states:
        st.check()  # no step gave up waiting for its copies
    world = dist.get_world_size() if dist is not None else 1
    # bytes a step has to move: the state (read + write), the retained and
    # current-chunk keys / values (read), the token in and out
    p_mean = (t0 % 64) + (nw + K + (K - 1) / 2.0) / NL
    nbytes = B * H * (2 * d * d * 4 + (kept + p_mean + 1) * d * 2 * 2 + 5 * d * 2)
    pk = peaks()
    gbs = nbytes / (ms / 1e3) / 1e9
    step_mb = B * H * (2 * d * d * 4 + (kept + 64) * d * 2 * 2) / 2**20
    return {"what": f"nats_decode_step: one token per (b, h) after a {t0}-token context, 25 % of its chunks "
                    f"retained ({kept} keys / values per head)",
            "config": {"B": B, "H": H, "d": d, "position": t0, "retained_per_head": kept, "layers_in_turn": NL,
                       "l2": f"four layers' states in turn: each step's {step_mb:.0f} MB was evicted by the other "
                             "three"},
            "value": job_throughput(B, world, ms), "unit": "tokens/s", "ms_per_step": ms, "steps": K,
            "host_loop_ms_per_step": host_ms,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"], "bytes_per_step": nbytes}}


def main():
    args = parse()
    if args.workload != WORKLOAD:
        set_workload(args.workload)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        res = run_reference(args, rank)
        print(json.dumps(res), flush=True)
        return 0
    import __graft_entry__

    __graft_entry__.build()
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_native(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
