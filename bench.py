#!/usr/bin/env python
"""PISA select+attend throughput on GB300.

Default workload (one GPU): prefill over N = 65536 tokens, B = 1, Hq = 16, Hkv = 2, d = 128,
leaf C = 64, K = 16, g = 2, Qtile = 4, bf16 N(0,1) inputs with 8 needle leaf blocks per KV
head. One step = pyramid build + pyramid Top-K selection + causal block-sparse attention
forward over the selection, on inputs already resident in HBM; tokens/s = B*N / step time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload prefill_64k|prefill_32k|prefill_4k|sweep|quality|decode|train]
                  [--sweep-n 4096,...]

Under torchrun each rank runs the same workload on its own GPU (independent problems, no
collective on the data path: weak scaling); the timed region is bracketed by barriers and
the slowest rank's time is reported. `--impl reference` times the fp64 CPU oracle on a
bounded sample of the same workload on the host cores (rank 0 only).
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
import time

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")   # the oracle legs run single-threaded
os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import pisa_synth as syn  # noqa: E402

WORKLOADS = {
    "prefill_64k": dict(B=1, N=65536, Hq=16, Hkv=2, d=128, C=64, K=16, g=2, qtile=4, needles=True),
    "prefill_4k": dict(B=1, N=4096, Hq=4, Hkv=1, d=64, C=64, K=8, g=2, qtile=1, needles=False),
    "prefill_32k": dict(B=1, N=32768, Hq=16, Hkv=2, d=128, C=64, K=16, g=2, qtile=4, needles=True),
    "sweep": dict(B=1, N=65536, Hq=32, Hkv=8, d=128, C=64, K=16, g=2, qtile=4, needles=True),
    "quality": dict(B=1, N=16384, Hq=16, Hkv=2, d=128, C=64, K=16, g=2, qtile=4, needles=True),
    "train": dict(B=4, N=16384, Hq=16, Hkv=4, d=128, C=64, K=16, g=2, qtile=4, needles=False),
    "decode": dict(B=32, N=131072, Hq=32, Hkv=8, d=128, C=64, K=16, g=2, qtile=1, needles=False),
    # the decode kernel at batch 4 (2 GB of cache): small enough for sectioned profiler captures
    "decode_small": dict(B=4, N=131072, Hq=32, Hkv=8, d=128, C=64, K=16, g=2, qtile=1, needles=False),
}
METRIC = "PISA select+attend tokens/s vs N (4K-256K) on 1 GB300; % of HBM/TC roofline"
L2_BYTES = 129 * 2 ** 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="prefill_64k", choices=sorted(WORKLOADS))
    ap.add_argument("--sweep-n", default="4096,16384,65536,131072,262144")
    ap.add_argument("--quality-n", default="4096,16384,65536")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="headline workload only")
    return ap.parse_args()


# ------------------------------------------------------------------ environment helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of the ranks' values: the slowest rank sets the whole job's time."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def rank_barrier(world: int) -> None:
    """All ranks meet, then this rank's GPU work drains (both sides of a timed region)."""
    if world > 1:
        torch.distributed.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: every rank's units over the (max-over-ranks) step time."""
    return units_per_rank * world / (ms / 1e3)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            out = {}
            for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                v = d.get(k)
                if isinstance(v, dict):
                    v = v.get("value")
                if v is not None:
                    out[k] = float(v)
            if "hbm_gbs" in out and "bf16_tflops" in out:
                out.setdefault("bf16_tflops_sustained", out["bf16_tflops"])
                return out, "measured"
        except Exception:  # malformed file: fall back, and say so
            pass
    return dict(FALLBACK_PEAKS), "fallback"


class _NvmlReader:
    """SM clock, its maximum and the active clock-event reasons of one GPU through the driver's
    NVML library (read-only queries; nothing is set)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, cuda_index: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        bus = None
        try:
            props = torch.cuda.get_device_properties(cuda_index)
            bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0".encode()
        except Exception:
            bus = None
        rc = self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(self.dev)) if bus else 1
        if rc != 0 and self.lib.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(self.dev)) != 0:
            raise OSError("no NVML handle")
        self.reason_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons")

    def read(self):
        c, m, r = self.ct.c_uint(), self.ct.c_uint(), self.ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.dev, 1, self.ct.byref(c)) != 0:
            return None
        self.lib.nvmlDeviceGetMaxClockInfo(self.dev, 1, self.ct.byref(m))
        self.reason_fn(self.dev, self.ct.byref(r))
        return float(c.value), float(m.value), [n for bit, n in self.REASONS.items() if r.value & bit]

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clocks and throttle reasons sampled during the timed region: every 10 ms through NVML
    from a host thread, or (without NVML) every 50 ms by nvidia-smi."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.nvml = None
        self.samples = []
        self.path = os.path.join("/tmp", f"pisa_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.nvml = _NvmlReader(self.index)
        except Exception:
            self.nvml = None
        if self.nvml is not None:
            import threading
            self.stop = threading.Event()

            def loop():
                while not self.stop.is_set():
                    x = self.nvml.read()
                    if x is not None:
                        self.samples.append(x)
                    self.stop.wait(0.01)

            self.thread = threading.Thread(target=loop, daemon=True)
            self.thread.start()
            return self
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.nvml is not None:
            self.stop.set()
            self.thread.join(timeout=5)
            self.nvml.close()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def wait_started(self, busy, timeout_s: float = 3.0):
        """Run untimed work (busy) until the sampler has taken its first sample, so that its
        samples cover the timed region that follows."""
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < timeout_s:
            if self.nvml is not None:
                if self.samples:
                    return
            elif self.proc is None:
                return
            else:
                try:
                    if os.path.getsize(self.path) > 0:
                        return
                except OSError:
                    pass
            busy()
            torch.cuda.synchronize()

    def summary(self):
        sm, mx, reasons = [], [], set()
        if self.nvml is not None:
            for c, m, r in self.samples:
                sm.append(c)
                mx.append(m)
                reasons.update(r)
        elif self.proc is not None and os.path.exists(self.path):
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    mx.append(float(f[2]))
                except ValueError:
                    continue
                for n, v in zip(names, f[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvml" if self.nvml is not None else "nvidia-smi"}


# Sources whose change invalidates a kernel's committed DRAM traffic figure: the kernel's own
# file, the headers it includes and the grouping that shapes its work items.
KERNEL_SOURCES = {
    "route_prefix": ["select.cu", "device.cuh", "tc.cuh"],
    "route": ["select.cu", "device.cuh", "pyramid.cu", "tc.cuh"],
    "leaf_score": ["leaf_tc.cu", "tiles.cuh", "tc.cuh", "tmap.cpp", "device.cuh", "group.cu", "group.h", "select.cu"],
    "attn_fwd_tc": ["attn_ws.cu", "tiles.cuh", "tc.cuh", "tmap.cpp", "device.cuh", "group.cu", "group.h", "attn.cu"],
    "attn_bwd": ["attn_bwd.cu", "attn_bwd_tc.cu", "tiles.cuh", "tc.cuh", "tmap.cpp", "device.cuh", "group.cu", "group.h"],
}


def source_hash(files=None) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "pyramid_top_selection_gb300", "csrc")
    for f in sorted(files if files is not None else os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, units_per_launch: float):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on these sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        e = d.get(kernel)
        if not e or e.get("source_hash") != source_hash(KERNEL_SOURCES.get(kernel)):
            return None
        return e["dram_bytes_per_unit"] * units_per_launch
    except Exception:
        return None


# ------------------------------------------------------------------ algorithmic work
def algorithmic(kernel, cfg, idx_host=None):
    """(bound, per-launch amount, unit, units processed, per-unit figure) of a kernel."""
    B, N, Hq, Hkv, d, C, K = (cfg[k] for k in ("B", "N", "Hq", "Hkv", "d", "C", "K"))
    G = Hq // Hkv
    n0 = -(-N // C)
    i = torch.arange(N, dtype=torch.float64)
    if kernel in ("build_leaves",):
        units = B * N * Hkv
        per = d * 2 + (n0 * 4 * d * (1 + 0.5 + 0.25 + 0.125)) / N
        return "hbm", units * per, "bytes", units, per
    if kernel == "route":
        sizes = [n0]
        while sizes[-1] > 1:
            sizes.append(-(-sizes[-1] // 2))
        lvl = sum(1 for l in range(1, len(sizes) - 1) if sizes[l] > K)   # levels that prune
        units = B * Hkv * N
        per = lvl * (2 * K) * 2 * G * 2 * d   # 2K candidates x 2 children x G heads x 2d flops
        return "tensor", units * per, "flops", units, per
    if kernel == "leaf_score":
        cands = torch.clamp(torch.floor(i / C) + 1, max=2 * K).sum().item()
        units = B * Hkv * cands
        per = G * C * 2 * d
        return "tensor", units * per, "flops", units, per
    if kernel == "attn_fwd_tc" and idx_host is not None:
        keys = selected_keys(idx_host, C, N)
        units = keys * G
        per = 4 * d
        return "tensor", units * per, "flops", units, per
    if kernel == "attn_lse_tc" and idx_host is not None:
        keys = selected_keys(idx_host, C, N)
        units = keys * G
        per = 2 * d
        return "tensor", units * per, "flops", units, per
    if kernel == "attn_rows":   # K block LSEs + K indices read, lse written
        units = B * N * Hq
        per = K * 4 + K * 4 / G + 4
        return "hbm", units * per, "bytes", units, per
    if kernel == "attn_out":    # fp32 accumulator read, bf16 O written
        units = B * N * Hq
        per = d * 4 + d * 2
        return "hbm", units * per, "bytes", units, per
    return None


def selected_keys(idx: torch.Tensor, C: int, N: int) -> float:
    """Number of (query, visible key) pairs inside the selection, over all KV heads."""
    B, Hkv, N_, K = idx.shape
    i = torch.arange(N_, dtype=torch.int64).view(1, 1, N_, 1)
    t = idx.to(torch.int64)
    start = t * C
    cnt = torch.clamp(torch.minimum(start + C, i + 1) - start, min=0)
    cnt = torch.where(t >= 0, cnt, torch.zeros_like(cnt))
    return float(cnt.sum().item())


# ------------------------------------------------------------------ our arm
def run_ours(args, cfg, rank, world, local):
    import pyramid_top_selection_gb300 as pisa
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    B, N, Hq, Hkv, d, C, K, g, qtile = (cfg[k] for k in ("B", "N", "Hq", "Hkv", "d", "C", "K", "g", "qtile"))
    Q, Kt, V = syn.make_prefill(B, N, Hq, Hkv, d, C=C, seed=0, needles=cfg["needles"], device=dev)
    shape = pisa.make_shape(B, N, Hq, Hkv, d, C, K, g, qtile)
    _, _, nodes = pisa.pyramid_layout(shape)
    pyr = torch.empty(B, Hkv, nodes, d, dtype=torch.float32, device=dev)
    idx = torch.empty(B, Hkv, N, K, dtype=torch.int32, device=dev)
    score = torch.empty(B, Hkv, N, K, dtype=torch.float32, device=dev)
    hl = torch.empty(B, Hq, N, K, dtype=torch.float32, device=dev)
    O = torch.empty_like(Q)
    lse = torch.empty(B, Hq, N, dtype=torch.float32, device=dev)
    ws_sel = pisa.workspace(shape, 0, dev)
    ws_att = pisa.workspace(shape, 2, dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def step(Qs, Ks, Vs):
        pisa.build_pyramid(Ks, shape, out=pyr)
        pisa.select(Qs, Ks, pyr, shape, ws=ws_sel, idx=idx, score=score, head_lse=hl)
        pisa.sparse_attn_fwd(Qs, Ks, Vs, idx, shape, ws=ws_att, out=O, lse=lse, head_lse=hl)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step(Q, Kt, V)
    stream = torch.cuda.current_stream(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    with ClockSampler(local) as clk:
        clk.wait_started(lambda: step(Q, Kt, V))
        for k in range(args.steps):
            flush.zero_()                        # L2 flush, outside the timed events
            ev[k][0].record(stream)
            step(Q, Kt, V)
            ev[k][1].record(stream)
        barrier()
    times = [a.elapsed_time(b) for a, b in ev]
    ms = sum(times) / len(times)
    ms = max_over_ranks(ms, world, dev)
    value = job_rate(B * N, world, ms)

    # per-kernel times (events around every launch, on the launch stream)
    pisa.profile_start()
    for k in range(args.steps):
        flush.zero_()
        step(Q, Kt, V)
    torch.cuda.synchronize()
    pisa.profile_stop()
    prof = pisa.profile_read()
    launches = sum(v[0] for v in prof.values())
    per_step_launches = launches / args.steps
    kernels = {k: {"launches": v[0], "avg_ms": v[1] / v[0], "share": 0.0} for k, v in prof.items()}
    tot = sum(v[1] for v in prof.values())
    for k, v in prof.items():
        kernels[k]["share"] = v[1] / tot if tot else 0.0
    dom = max(prof.items(), key=lambda kv: kv[1][1])[0]

    idx_host = idx.cpu()
    pk, psrc = peaks()
    roof = None
    alg = algorithmic(dom, cfg, idx_host)
    if alg is not None:
        bound, amount, unit, units, per = alg
        avg_s = kernels[dom]["avg_ms"] / 1e3
        if unit == "bytes":
            achieved = amount / avg_s / 1e9
            peak = pk["hbm_gbs"]
            u = "GB/s"
        else:
            achieved = amount / avg_s / 1e12
            peak = pk["bf16_tflops"]
            u = "TFLOP/s"
        roof = {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak, "unit": u,
                "frac": achieved / peak, "peak_source": psrc,
                "traffic": traffic_for(dom, units), "units_per_launch": units, "per_unit": per,
                "per_unit_kind": unit}

    # e2e through the public API with host buffers (pinned): every step copies its inputs in
    # and its results (O, idx, lse) out inside the timed region. The steps are software-
    # pipelined over three streams (step k+1's inputs travel while step k computes and step
    # k-1's results travel back), with two device buffer sets so no copy overwrites data in
    # use; one event pair brackets the whole run.
    e2e = None
    if not args.no_e2e:
        hQ, hK, hV = (x.cpu().pin_memory() for x in (Q, Kt, V))
        hO = torch.empty(O.shape, dtype=O.dtype, pin_memory=True)
        hidx = torch.empty(idx.shape, dtype=idx.dtype, pin_memory=True)
        hlse = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        din = [tuple(torch.empty_like(x) for x in (Q, Kt, V)) for _ in range(2)]
        dout = [tuple(torch.empty_like(x) for x in (O, idx, lse, score, hl)) for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def run_pipeline(n):
            ev_in = [torch.cuda.Event() for _ in range(n)]
            ev_done = [torch.cuda.Event() for _ in range(n)]
            ev_out = [torch.cuda.Event() for _ in range(n)]
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(s_in)
            for k in range(n):
                sl = k % 2
                with torch.cuda.stream(s_in):
                    if k >= 2:
                        s_in.wait_event(ev_done[k - 2])          # slot's inputs no longer read
                    for dst, src in zip(din[sl], (hQ, hK, hV)):
                        dst.copy_(src, non_blocking=True)
                    ev_in[k].record(s_in)
                stream.wait_event(ev_in[k])
                if k >= 2:
                    stream.wait_event(ev_out[k - 2])             # slot's results copied out
                o_, i_, l_, sc_, hl_ = dout[sl]
                pisa.build_pyramid(din[sl][1], shape, out=pyr)
                pisa.select(din[sl][0], din[sl][1], pyr, shape, ws=ws_sel, idx=i_, score=sc_, head_lse=hl_)
                pisa.sparse_attn_fwd(din[sl][0], din[sl][1], din[sl][2], i_, shape, ws=ws_att, out=o_, lse=l_,
                                     head_lse=hl_)
                ev_done[k].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_done[k])
                    for dst, src in zip((hO, hidx, hlse), (o_, i_, l_)):
                        dst.copy_(src, non_blocking=True)
                    ev_out[k].record(s_out)
            s_in.wait_stream(s_out)
            t1.record(s_in)
            t1.synchronize()
            return t0.elapsed_time(t1)

        run_pipeline(2)
        barrier()
        e_ms = run_pipeline(args.steps) / args.steps
        barrier()
        e_ms = max_over_ranks(e_ms, world, dev)
        h2d = sum(x.numel() * x.element_size() for x in (hQ, hK, hV))
        d2h = sum(x.numel() * x.element_size() for x in (hO, hidx, hlse))
        e2e = {"value": job_rate(B * N, world, e_ms), "unit": "tokens/s", "ms_per_step": e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "schedule": "3 streams: inputs of step k+1 in and results of step k-1 out while step k computes; "
                           "inputs larger than L2 (no flush)"}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, *(x.cpu().double().numpy() for x in (Q, Kt, V)), budget_s=12.0)

    # The other configurations, compact, in the same record (rank 0 only; each rank's GPU is
    # its own replica, so one rank's figures stand for all).
    configs = None
    if rank == 0 and not args.no_extras:
        configs = other_configs(dev, flush)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "ms_per_step_median": statistics.median(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16, 8 needle leaf blocks per KV head)",
            "config": {"workload": f"prefill select+attend, N={N}", "B": B, "N": N, "Hq": Hq, "Hkv": Hkv,
                       "d": d, "C": C, "K": K, "g": g, "qtile": qtile,
                       "l2": "flushed between timed steps (256 MiB write)",
                       "step": "build_pyramid + select + sparse_attn_fwd", "parallelism": f"replica x{world}"},
            "gpu_launches": int(round(per_step_launches * args.steps)),
            "kernels": kernels, "roofline": roof, "e2e": e2e, "cpu_baseline": cpu,
            "configs": configs,
        }
        if clk.summary() is not None:
            line["clocks"] = clk.summary()
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ oracle legs
def oracle_sample(cfg, Q, Kt, V, n_queries, seed=0):
    """Run the oracle's select + attention on a sample of queries (all KV heads)."""
    from oracle import pisa_oracle as po
    N, C, K = cfg["N"], cfg["C"], cfg["K"]
    g = torch.Generator().manual_seed(seed)
    qs = sorted(torch.randperm(N, generator=g)[:n_queries].tolist())
    t0 = time.perf_counter()
    ora = po.select(Q, Kt, C, K, queries=qs)
    po.sparse_attn_fwd(Q, Kt, V, ora["idx"], C, queries=qs)
    return time.perf_counter() - t0, qs


def oracle_setup_time(cfg, Kt):
    from oracle import pisa_oracle as po
    t0 = time.perf_counter()
    for b in range(cfg["B"]):
        for kv in range(cfg["Hkv"]):
            po.CausalKeySummaries(Kt[b, :, kv, :], cfg["C"])
    return time.perf_counter() - t0


def cpu_baseline(cfg, Q, Kt, V, budget_s=12.0):
    """The oracle as it stands, single-threaded on the host, on a bounded query sample.

    tokens/s = sampled queries / (their select+attend time + the per-head summary set-up
    time scaled by sample/N, i.e. amortised as over the full workload)."""
    n = 8
    setup = oracle_setup_time(cfg, Kt)
    t_run, _ = oracle_sample(cfg, Q, Kt, V, n)
    per_q = max(t_run - setup, 1e-6) / n
    n = max(8, min(cfg["N"], int((budget_s - setup) / per_q)))
    t_run, qs = oracle_sample(cfg, Q, Kt, V, n, seed=1)
    t_q = max(t_run - setup, 1e-9)
    value = n / (t_q + setup * n / cfg["N"])
    return {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} random queries of the N={cfg['N']} workload (all {cfg['Hkv']} KV heads), "
                      f"fp64 numpy, 1 thread; per-head summary set-up {setup:.2f}s amortised over N"}


def run_reference(args, cfg, rank, world):
    if rank != 0:
        return
    B, N, Hq, Hkv, d, C = (cfg[k] for k in ("B", "N", "Hq", "Hkv", "d", "C"))
    Q, Kt, V = (x.double().numpy() for x in syn.make_prefill(B, N, Hq, Hkv, d, C=C, seed=0,
                                                              needles=cfg["needles"]))
    setup = oracle_setup_time(cfg, Kt)
    n = 16
    for w in range(args.warmup):
        oracle_sample(cfg, Q, Kt, V, 2, seed=100 + w)
    times = []
    for k in range(args.steps):
        t, _ = oracle_sample(cfg, Q, Kt, V, n, seed=k)
        times.append(max(t - setup, 1e-9))
    per_step = sum(times) / len(times) + setup * n / N
    value = n / per_step
    cpu = {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
           "sample": f"{n} random queries per step of the N={N} workload (all {Hkv} KV heads), fp64 "
                     f"numpy, 1 thread; summary set-up {setup:.2f}s amortised over N"}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16, 8 needle leaf blocks per KV head)",
            "config": {"workload": f"prefill select+attend, N={N}", **{k: cfg[k] for k in
                       ("B", "N", "Hq", "Hkv", "d", "C", "K", "g", "qtile")}},
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ extra workloads
def exact_leaf_lse(Qg, Kk, q0, q1, C, scale):
    """Per-head exact leaf LSEs of queries q0..q1-1 of one KV head: [q, G, visible leaves] fp32,
    -inf where a leaf has no visible key (a plain dense reference for the quality measurement)."""
    nk = q1
    logits = scale * torch.einsum("igd,jd->igj", Qg[q0:q1].float(), Kk[:nk].float())
    i = torch.arange(q0, q1, device=Kk.device).view(-1, 1, 1)
    j = torch.arange(nk, device=Kk.device).view(1, 1, -1)
    logits = logits.masked_fill(j > i, float("-inf"))
    nl = -(-nk // C)
    pad = nl * C - nk
    if pad:
        logits = torch.nn.functional.pad(logits, (0, pad), value=float("-inf"))
    return torch.logsumexp(logits.view(q1 - q0, Qg.shape[1], nl, C), dim=-1)


def quality_stats(sels, Q, Kt, C, K, needles, QB=256):
    """Selection quality of every selection in `sels` (name -> idx [B,Hkv,N,K]) and of the exact
    top-K itself, against exhaustive exact leaf scores: recall of the exact top-K (queries with
    more than K visible leaves), recall of the planted needle leaves (queries aligned with the
    needle direction), and the mean share of each head's full causal softmax mass that falls
    inside the selected leaves."""
    B, N, Hq, d = Q.shape
    Hkv = Kt.shape[2]
    G = Hq // Hkv
    dev = Q.device
    scale = 1.0 / math.sqrt(d)
    acc = {k: dict(hit=0.0, units=0, needle=0.0, nunits=0, mass=0.0, munits=0) for k in list(sels) + ["exact"]}
    for b in range(B):
        for kv in range(Hkv):
            Qg = Q[b, :, kv * G:(kv + 1) * G, :]
            Kk = Kt[b, :, kv, :]
            u = syn.needle_direction(Q, Hkv, b, kv)
            nd = torch.tensor(needles[b][kv], device=dev)
            for q0 in range(0, N, QB):
                q1 = min(q0 + QB, N)
                ll = exact_leaf_lse(Qg, Kk, q0, q1, C, scale)                     # [q, G, nl]
                full = torch.logsumexp(ll, dim=-1, keepdim=True)                  # [q, G, 1]
                score = ll.sum(1)                                                 # [q, nl]
                nl = score.shape[1]
                vis = torch.arange(q0, q1, device=dev) // C + 1                   # visible leaves
                kk = min(K, nl)
                exact = torch.topk(score, kk, dim=-1).indices
                exact = exact.masked_fill(torch.arange(kk, device=dev).view(1, -1) >= vis.view(-1, 1), -1)
                aligned = (Qg[q0:q1].float() @ u).sum(-1) > 0
                vneed = (nd.view(1, -1) < vis.view(-1, 1))                        # [q, 8]
                prune = vis > K                                                   # rows where K < visible
                for name, a in acc.items():
                    sel = exact if name == "exact" else sels[name][b, kv, q0:q1].long()
                    hit = (sel.unsqueeze(-1) == exact.unsqueeze(1)) & (sel.unsqueeze(-1) >= 0)
                    a["hit"] += hit.any(-1).sum(-1)[prune].float().sum().item()
                    a["units"] += int(prune.sum().item()) * K
                    got = (nd.view(1, 1, -1) == sel.unsqueeze(-1)).any(1) & vneed      # [q, 8]
                    rows = aligned & vneed.any(-1)
                    a["needle"] += (got.sum(-1).float() / vneed.sum(-1).clamp_min(1))[rows].sum().item()
                    a["nunits"] += int(rows.sum().item())
                    g_ = sel.clamp_min(0).unsqueeze(1).expand(-1, G, -1)
                    m = torch.exp(torch.gather(ll, 2, g_) - full) * (sel >= 0).unsqueeze(1)
                    a["mass"] += m.sum(-1).sum().item()
                    a["munits"] += (q1 - q0) * G
    return {name: {"recall_exact_topk": a["hit"] / max(1, a["units"]),
                   "needle_recall_aligned": a["needle"] / max(1, a["nunits"]),
                   "attention_mass": a["mass"] / max(1, a["munits"])} for name, a in acc.items()}


QUALITY_NOTES = {"reference": "exhaustive exact leaf scores (dense fp32 logits on the GPU, per-head LSE per leaf "
                              "summed over the group)",
                 "recall_rows": "queries with more than K visible leaves",
                 "needle_rows": "queries with sum_h q.u > 0 and at least one visible needle leaf",
                 "mass": "mean over (query, head) of the full causal softmax mass inside the selected leaves"}


def quality_selections(Q, Kt, cfg):
    """The library's selections compared by the quality workload."""
    import pyramid_top_selection_gb300 as pisa
    B, N, Hq, d = Q.shape
    shape = pisa.make_shape(B, N, Hq, Kt.shape[2], d, cfg["C"], cfg["K"], cfg["g"], cfg["qtile"])
    pyr = pisa.build_pyramid(Kt, shape)
    return {"pyramid": pisa.select(Q, Kt, pyr, shape, want_score=False)[0],
            "pisa1_mean": pisa.select_mean(Q, Kt, pyr, shape, want_score=False)[0],
            "pisa2_meanvar": pisa.select_meanvar(Q, Kt, pyr, shape, want_score=False)[0],
            "flat": pisa.select_flat(Q, Kt, pyr, shape, want_score=False)[0]}


def run_quality(args, cfg, local):
    """Selection quality on the needle data (one JSON line per N)."""
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    for N in [int(x) for x in args.quality_n.split(",")]:
        c = dict(cfg, N=N)
        B, Hq, Hkv, d, C, K = c["B"], c["Hq"], c["Hkv"], c["d"], c["C"], c["K"]
        Q, Kt, _ = syn.make_prefill(B, N, Hq, Hkv, d, C=C, seed=0, needles=True, device=dev)
        needles = syn.needle_leaves(B, Hkv, -(-N // C), 3, device=dev)
        out = quality_stats(quality_selections(Q, Kt, c), Q, Kt, C, K, needles)
        print(json.dumps({"workload": "selection quality", "N": N, "B": B, "Hq": Hq, "Hkv": Hkv, "d": d, "C": C,
                          "K": K, "data": "synthetic (seeded N(0,1) bf16, 8 needle leaf blocks per KV head)",
                          **QUALITY_NOTES, **out}), flush=True)


def graph_of(fn, check=None):
    """fn() captured once in a CUDA graph (its buffers fixed) for replay in place of the eager
    calls, so that a launch-bound chain of small kernels runs without host launch gaps. None when
    the capture fails or a replay's `check` output differs from the eager run's (a selection is
    bit-exact from run to run)."""
    torch.cuda.synchronize()
    ref = check.clone() if check is not None else None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            fn()
        g.replay()
        torch.cuda.synchronize()
    except Exception:
        return None
    if ref is not None and not torch.equal(ref, check):
        return None
    return g


def sweep_point(args, cfg, N, dev, flush):
    """Pyramid selection, its PISA-1 ablation and the flat comparator at one N (selection only,
    median of L2-flushed runs), plus the pyramid build's achieved HBM bandwidth."""
    import pyramid_top_selection_gb300 as pisa
    c = dict(cfg, N=N)
    Q, Kt, _ = syn.make_prefill(c["B"], N, c["Hq"], c["Hkv"], c["d"], C=c["C"], seed=0, needles=True, device=dev)
    shape = pisa.make_shape(c["B"], N, c["Hq"], c["Hkv"], c["d"], c["C"], c["K"], c["g"], c["qtile"])
    _, _, nodes = pisa.pyramid_layout(shape)
    pyr = torch.empty(c["B"], c["Hkv"], nodes, c["d"], dtype=torch.float32, device=dev)
    idx = torch.empty(c["B"], c["Hkv"], N, c["K"], dtype=torch.int32, device=dev)
    ws_p, ws_f = pisa.workspace(shape, 0, dev), pisa.workspace(shape, 1, dev)

    launch = []

    def timed(fn, check):
        for _ in range(max(1, args.warmup)):
            fn()
        g = graph_of(fn, check)
        launch.append("cuda_graph" if g is not None else "eager")
        run = g.replay if g is not None else fn
        ts = []
        for _ in range(args.steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            run()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    out = {"build_ms": timed(lambda: pisa.build_pyramid(Kt, shape, out=pyr), pyr)}
    build_bytes = Kt.numel() * 2 + pyr.numel() * 4
    out["build_gbs"] = build_bytes / (out["build_ms"] / 1e3) / 1e9
    ws_v = pisa.workspace(shape, 5, dev)
    for name, fn, ws in (("pyramid", pisa.select, ws_p), ("pisa1_mean", pisa.select_mean, ws_p),
                         ("pisa2_meanvar", pisa.select_meanvar, ws_v), ("flat", pisa.select_flat, ws_f)):
        call = lambda: fn(Q, Kt, pyr, shape, ws=ws, want_score=False, idx=idx)   # noqa: E731
        out[name] = timed(call, idx)
        kern, _, _ = profile_kernels(pisa, call, max(1, args.steps), flush)
        out[name + "_kernels"] = {k: round(v["avg_ms"], 4) for k, v in kern.items()}
    pk, _ = peaks()
    line = {"workload": "selection sweep", "N": N, "B": c["B"], "Hq": c["Hq"], "Hkv": c["Hkv"], "d": c["d"],
            "K": c["K"], "pyramid_select_ms": out["pyramid"], "flat_select_ms": out["flat"],
            "flat_over_pyramid": out["flat"] / out["pyramid"],
            "pyramid_tokens_per_s": c["B"] * N / (out["pyramid"] / 1e3),
            "pyramid_kernels_ms": out["pyramid_kernels"], "flat_kernels_ms": out["flat_kernels"],
            "pisa1_mean_select_ms": out["pisa1_mean"], "pisa1_mean_kernels_ms": out["pisa1_mean_kernels"],
            "pisa2_meanvar_select_ms": out["pisa2_meanvar"], "pisa2_meanvar_kernels_ms": out["pisa2_meanvar_kernels"],
            "build_ms": out["build_ms"], "build_gbs": out["build_gbs"],
            "build_hbm_frac": out["build_gbs"] / pk["hbm_gbs"],
            "launch": launch[0] if len(set(launch)) == 1 else ",".join(launch)}
    del Q, Kt, pyr, idx, ws_p, ws_f, ws_v
    torch.cuda.empty_cache()
    return line


def run_sweep(args, cfg, local):
    """Pyramid selection vs the flat comparator over N (one JSON line per N)."""
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    for N in [int(x) for x in args.sweep_n.split(",")]:
        print(json.dumps(sweep_point(args, cfg, N, dev, flush)), flush=True)


def prefill_point(args, cfg, dev, flush):
    """Device step time of build + select + attend on one prefill configuration."""
    import pyramid_top_selection_gb300 as pisa
    B, N, Hq, Hkv, d, C, K, g, qtile = (cfg[k] for k in ("B", "N", "Hq", "Hkv", "d", "C", "K", "g", "qtile"))
    Q, Kt, V = syn.make_prefill(B, N, Hq, Hkv, d, C=C, seed=0, needles=cfg["needles"], device=dev)
    shape = pisa.make_shape(B, N, Hq, Hkv, d, C, K, g, qtile)
    _, _, nodes = pisa.pyramid_layout(shape)
    pyr = torch.empty(B, Hkv, nodes, d, dtype=torch.float32, device=dev)
    idx = torch.empty(B, Hkv, N, K, dtype=torch.int32, device=dev)
    hl = torch.empty(B, Hq, N, K, dtype=torch.float32, device=dev)
    O, lse = torch.empty_like(Q), torch.empty(B, Hq, N, dtype=torch.float32, device=dev)
    ws_sel, ws_att = pisa.workspace(shape, 0, dev), pisa.workspace(shape, 2, dev)

    def step():
        pisa.build_pyramid(Kt, shape, out=pyr)
        pisa.select(Q, Kt, pyr, shape, ws=ws_sel, want_score=False, idx=idx, head_lse=hl)
        pisa.sparse_attn_fwd(Q, Kt, V, idx, shape, ws=ws_att, out=O, lse=lse, head_lse=hl)

    for _ in range(args.warmup):
        step()
    g = graph_of(step, idx)
    run = g.replay if g is not None else step
    ts = []
    for _ in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        run()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    ms = sum(ts) / len(ts)
    kernels, _, _ = profile_kernels(pisa, step, args.steps, flush)
    return {"workload": f"prefill select+attend, N={N}", "tokens_per_s": B * N / (ms / 1e3), "ms_per_step": ms,
            "launch": "cuda_graph" if g is not None else "eager",
            "config": {k: cfg[k] for k in ("B", "N", "Hq", "Hkv", "d", "C", "K", "g", "qtile")},
            "kernels_ms": {k: round(v["avg_ms"], 4) for k, v in kernels.items()}}


def other_configs(dev, flush):
    """The other configurations, each measured briefly on this GPU, as compact sub-objects of
    the headline record: the 4K prefill, the headline shape's throughput at 4K-256K, the
    selection sweep (pyramid vs flat) at 16K-256K with the pyramid build's bandwidth, the
    batch-32 decode and the training step."""
    import types
    sub = types.SimpleNamespace(steps=5, warmup=3)
    t0 = time.perf_counter()
    out = {"prefill_4k": prefill_point(sub, WORKLOADS["prefill_4k"], dev, flush)}
    # the headline's select+attend throughput against N (4K-256K) on its own head shape
    curve = {}
    for N in (4096, 16384, 131072, 262144):
        pp = prefill_point(sub, dict(WORKLOADS["prefill_64k"], N=N), dev, flush)
        curve[f"N={N}"] = {"tokens_per_s": pp["tokens_per_s"], "ms_per_step": pp["ms_per_step"], "launch": pp["launch"]}
    out["prefill_vs_n"] = {"config": {k: WORKLOADS["prefill_64k"][k] for k in ("B", "Hq", "Hkv", "d", "C", "K", "g", "qtile")},
                           "note": "N=65536 is the headline line itself", **curve}
    sw = {}
    for N in (16384, 65536, 131072, 262144):
        p = sweep_point(sub, WORKLOADS["sweep"], N, dev, flush)
        e = {k: p[k] for k in ("pyramid_select_ms", "flat_select_ms", "flat_over_pyramid", "pisa1_mean_select_ms",
                               "pisa2_meanvar_select_ms", "build_ms", "build_gbs", "build_hbm_frac", "launch")}
        e["route_prefix_ms"] = p["pyramid_kernels_ms"].get("route_prefix")
        e["route_ms"] = p["pyramid_kernels_ms"].get("route")
        e["leaf_score_ms"] = p["pyramid_kernels_ms"].get("leaf_score")
        sw[f"N={N}"] = e
    out["selection_sweep"] = {"config": {k: WORKLOADS["sweep"][k] for k in ("B", "Hq", "Hkv", "d", "C", "K", "g")},
                              **sw}
    dl = run_decode(types.SimpleNamespace(steps=64, warmup=4), WORKLOADS["decode"], 0, 1, dev.index, emit=False)
    out["decode"] = {"tokens_per_s": dl["value"], "ms_per_step": dl["ms_per_step"], "hbm_gbs": dl["roofline"]["achieved"],
                     "hbm_frac": dl["roofline"]["frac"], "config": dl["config"]}
    tr = run_train(types.SimpleNamespace(steps=5, warmup=3), WORKLOADS["train"], 0, 1, dev.index, emit=False)
    out["train"] = {"tokens_per_s": tr["value"], "ms_per_step": tr["ms_per_step"],
                    "bwd_ms": tr["kernels"]["attn_bwd"]["avg_ms"], "bwd_tensor_tflops": tr["roofline"]["achieved"],
                    "bwd_tensor_frac": tr["roofline"]["frac"], "config": tr["config"]}
    qc = dict(WORKLOADS["quality"], N=4096)
    Q, Kt, _ = syn.make_prefill(qc["B"], qc["N"], qc["Hq"], qc["Hkv"], qc["d"], C=qc["C"], seed=0, needles=True,
                                device=dev)
    needles = syn.needle_leaves(qc["B"], qc["Hkv"], -(-qc["N"] // qc["C"]), 3, device=dev)
    out["selection_quality"] = {"config": {k: qc[k] for k in ("B", "N", "Hq", "Hkv", "d", "C", "K")},
                                **quality_stats(quality_selections(Q, Kt, qc), Q, Kt, qc["C"], qc["K"], needles),
                                **QUALITY_NOTES}
    out["seconds"] = time.perf_counter() - t0
    return out


# ------------------------------------------------------------------ decode and training
def profile_kernels(pisa, step, steps, flush=None):
    """Per-kernel CUDA-event times over `steps` calls of `step` (events on the launch stream)."""
    pisa.profile_start()
    for _ in range(steps):
        if flush is not None:
            flush.zero_()
        step()
    torch.cuda.synchronize()
    pisa.profile_stop()
    prof = pisa.profile_read()
    tot = sum(v[1] for v in prof.values()) or 1.0
    kernels = {k: {"launches": v[0], "avg_ms": v[1] / v[0], "share": v[1] / tot} for k, v in prof.items()}
    dom = max(prof.items(), key=lambda kv: kv[1][1])[0]
    return kernels, dom, sum(v[0] for v in prof.values())


def roofline_entry(kernel, bound, amount, unit_kind, avg_ms, units, per):
    pk, psrc = peaks()
    sec = avg_ms / 1e3
    if unit_kind == "bytes":
        achieved, peak, u = amount / sec / 1e9, pk["hbm_gbs"], "GB/s"
    else:
        achieved, peak, u = amount / sec / 1e12, pk["bf16_tflops"], "TFLOP/s"
    return {"kernel": kernel, "bound": bound, "achieved": achieved, "peak": peak, "unit": u,
            "frac": achieved / peak, "peak_source": psrc, "traffic": traffic_for(kernel, units),
            "units_per_launch": units, "per_unit": per, "per_unit_kind": unit_kind}


def run_decode(args, cfg, rank, world, local, emit=True):
    """Autoregressive decode: a batch of sequences with a long cache, one fused step per token."""
    import pyramid_top_selection_gb300 as pisa
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    B, L0, Hq, Hkv, d, C, K = (cfg[k] for k in ("B", "N", "Hq", "Hkv", "d", "C", "K"))
    total = 256                                      # steps the cache has room for
    Ncap = L0 + total
    steps = max(1, min(args.steps, total - args.warmup - 8))
    Kc = syn.randn_bf16((B, Ncap, Hkv, d), 1, dev)
    Vc = syn.randn_bf16((B, Ncap, Hkv, d), 2, dev)
    qs, ks, vs = syn.make_decode_stream(B, total, Hq, Hkv, d, seed=0, device=dev)
    shape = pisa.make_decode_shape(B, Ncap, Hq, Hkv, d, C, K)
    length = torch.full((B,), L0, dtype=torch.int32, device=dev)
    pyr = pisa.decode_build_pyramid(Kc, length, shape)
    pos = (L0 + torch.arange(total, device=dev, dtype=torch.int32)).view(total, 1).repeat(1, B).contiguous()
    o = torch.empty(B, Hq, d, dtype=torch.bfloat16, device=dev)
    idx = torch.empty(B, Hkv, K, dtype=torch.int32, device=dev)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    cur = [0]

    def step():
        t = cur[0]
        pisa.decode_step(shape, pos[t], Kc, Vc, pyr, qs[t], ks[t], vs[t], o=o, idx=idx, status=status)
        cur[0] += 1

    for _ in range(args.warmup):
        step()
    stream = torch.cuda.current_stream(dev)
    a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    rank_barrier(world)
    with ClockSampler(local) as clk:
        a.record(stream)
        for _ in range(steps):
            step()
        b_.record(stream)
        rank_barrier(world)
    ms = max_over_ranks(a.elapsed_time(b_) / steps, world, dev)
    prof_steps = min(8, total - cur[0])
    kernels, dom, launches = profile_kernels(pisa, step, prof_steps)
    assert int(status.sum()) == 0
    sizes = [-(-Ncap // C)]
    while sizes[-1] > 1:
        sizes.append(-(-sizes[-1] // 2))
    lv = sum(1 for l in range(1, len(sizes) - 1) if sizes[l] > K)
    per = (2 * K * C * d * 2 + K * C * d * 2 + lv * 2 * K * 2 * d * 4 + C * d * 2 + len(sizes) * 3 * d * 4)
    units = B * Hkv
    roof = roofline_entry("decode_step", "hbm", units * per, "bytes", kernels["decode_step"]["avg_ms"], units, per)
    line = None
    if rank == 0:
        line = {"workload": "decode", "metric": "decode tokens/s (one fused kernel per step)",
                "value": job_rate(B, world, ms), "unit": "tokens/s", "n_gpus": world, "steps": steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16",
                "config": {"B": B, "cache_tokens": L0, "Ncap": Ncap, "Hq": Hq, "Hkv": Hkv, "d": d, "C": C, "K": K,
                           "l2": "working set per step larger than L2 (no flush)"},
                "gpu_launches": steps, "kernels": kernels, "roofline": roof}
        if clk.summary() is not None:
            line["clocks"] = clk.summary()
        if emit:
            print(json.dumps(line), flush=True)
    return line


def run_train(args, cfg, rank, world, local, emit=True):
    """Training step: pyramid + selection (no gradient) + sparse attention forward and backward."""
    import pyramid_top_selection_gb300 as pisa
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    B, N, Hq, Hkv, d, C, K, g, qtile = (cfg[k] for k in ("B", "N", "Hq", "Hkv", "d", "C", "K", "g", "qtile"))
    Q, Kt, V = syn.make_prefill(B, N, Hq, Hkv, d, C=C, seed=0, needles=cfg["needles"], device=dev)
    dO = syn.make_grad_out(B, N, Hq, d, seed=0, device=dev)
    shape = pisa.make_shape(B, N, Hq, Hkv, d, C, K, g, qtile)
    _, _, nodes = pisa.pyramid_layout(shape)
    pyr = torch.empty(B, Hkv, nodes, d, dtype=torch.float32, device=dev)
    idx = torch.empty(B, Hkv, N, K, dtype=torch.int32, device=dev)
    hl = torch.empty(B, Hq, N, K, dtype=torch.float32, device=dev)
    O = torch.empty_like(Q)
    lse = torch.empty(B, Hq, N, dtype=torch.float32, device=dev)
    ws_sel, ws_f, ws_b = (pisa.workspace(shape, op, dev) for op in (0, 2, 3))
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def step():
        pisa.build_pyramid(Kt, shape, out=pyr)
        pisa.select(Q, Kt, pyr, shape, ws=ws_sel, want_score=False, idx=idx, head_lse=hl)
        pisa.sparse_attn_fwd(Q, Kt, V, idx, shape, ws=ws_f, out=O, lse=lse, head_lse=hl)
        pisa.sparse_attn_bwd(Q, Kt, V, O, lse, dO, idx, shape, ws=ws_b)

    for _ in range(args.warmup):
        step()
    stream = torch.cuda.current_stream(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    rank_barrier(world)
    with ClockSampler(local) as clk:
        for k in range(args.steps):
            flush.zero_()
            ev[k][0].record(stream)
            step()
            ev[k][1].record(stream)
        rank_barrier(world)
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev) / args.steps, world, dev)
    kernels, dom, launches = profile_kernels(pisa, step, args.steps, flush)
    keys = selected_keys(idx.cpu(), C, N)
    units = keys * (Hq // Hkv)
    roof = roofline_entry("attn_bwd", "tensor", units * 10 * d, "flops", kernels["attn_bwd"]["avg_ms"], units, 10 * d)
    line = None
    if rank == 0:
        line = {"workload": "train", "metric": "training tokens/s (select + sparse attention fwd + bwd)",
                "value": job_rate(B * N, world, ms), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16",
                "config": {k: cfg[k] for k in ("B", "N", "Hq", "Hkv", "d", "C", "K", "g", "qtile")},
                "gpu_launches": int(round(launches)), "kernels": kernels, "dominant": dom, "roofline": roof}
        if clk.summary() is not None:
            line["clocks"] = clk.summary()
        if emit:
            print(json.dumps(line), flush=True)
    return line


def main():
    args = parse()
    rank, world, local = dist_env()
    if world > 1 and args.impl == "ours":
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    cfg = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, cfg, rank, world)
        return
    if args.workload == "sweep":
        if rank == 0:
            run_sweep(args, cfg, local)
        return
    if args.workload == "quality":
        if rank == 0:
            run_quality(args, cfg, local)
        return
    if args.workload in ("decode", "decode_small"):
        run_decode(args, cfg, rank, world, local)
    elif args.workload == "train":
        run_train(args, cfg, rank, world, local)
    else:
        run_ours(args, cfg, rank, world, local)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
