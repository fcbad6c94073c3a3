#!/usr/bin/env python
"""Benchmark of the DSA hot path on GB300: DSA prefill tokens/s at T = S = 4096
(671B head shapes, bf16, top-2048), one JSON line on rank 0.

A step is one dsa_forward call (FP8 quantisation when configured, indexer,
top-k, q~ = q_nope W_UK, sparse latent attention, o_lat W_UV) over the whole
synthetic batch, inputs resident in HBM.  L2 is flushed (a 256 MiB write)
between timed steps, outside the timed events.  ``--impl reference`` times the
plain CPU oracle instead (a bounded sample of rows per step).

Under torchrun (N > 1) every rank runs the same workload on its own GPU (the
path shards by query rows / sequences with no exchange): weak scaling, value =
tokens of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DSA prefill tokens/s & decode queries/s on 1 GB300; % of tensor/HBM roofline"
CONFIG_NAMES = {0: "tiny-fp32-T256", 1: "prefill-bf16-T4096-S4096-top2048", 2: "prefill-bf16-T32768-S32768-top2048",
                3: "decode-bf16-64x1-S8192..65536-top2048", 4: "chunked-prefill-fp8idx-8x8192-S16384..65536-top2048"}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=1, help="workload 0..4 (1 = the headline prefill)")
    ap.add_argument("--cpu-rows", type=int, default=1024, help="rows of the oracle's bounded sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


def source_digest(paths):
    """sha256 over the given repository files, in order."""
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def ncu_traffic(stage: str, workload: str):
    """DRAM bytes per launch of the stage's kernel from the committed ncu
    capture (profiles/traffic.json), or None when there is no capture for this
    workload or the kernel's sources have changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        entry = json.load(f).get(stage)
    if not entry or entry.get("workload") != workload:
        return None
    srcs = entry["sources"]
    if not all(os.path.exists(os.path.join(ROOT, p)) for p in srcs) or source_digest(srcs) != entry["sha256"]:
        return None
    return float(entry["dram_bytes"])


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class NvmlClockSampler:
    """SM clock and clock-event reasons read through NVML (read-only queries)
    every 5 ms on a thread, so that a timed region of a few tens of
    milliseconds still gets samples.  Raises on construction if NVML cannot be
    loaded; ClockSampler (nvidia-smi) is the fallback."""
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}

    def __init__(self, uuid: str | None):
        import ctypes
        import threading
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        if uuid:
            rc = self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.dev))
        else:
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.dev))
        if rc != 0:
            raise RuntimeError("NVML device handle")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.samples = []
        self.stop_flag = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)
        mx = ctypes.c_uint()
        self.max_mhz = float(mx.value) if self.lib.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(mx)) == 0 else None

    def _run(self):
        ct = self.ct
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        while not self.stop_flag.is_set():
            if self.lib.nvmlDeviceGetClockInfo(self.dev, 1, ct.byref(clk)) == 0 and \
                    self.reasons_fn(self.dev, ct.byref(rs)) == 0:
                self.samples.append((float(clk.value), int(rs.value)))
            time.sleep(0.005)

    def start(self):
        self.thread.start()

    def stop(self):
        self.stop_flag.set()
        self.thread.join(timeout=2)
        self.lib.nvmlShutdown()
        if not self.samples:
            return None
        reasons = sorted({n for _, r in self.samples for bit, n in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples), "source": "NVML, 5 ms"}


def clock_sampler(uuid):
    try:
        return NvmlClockSampler(uuid)
    except Exception:
        return ClockSampler(uuid)


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.proc = None
        self.path = None
        self.uuid = uuid

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "200"]
            if self.uuid:
                cmd += ["-i", self.uuid]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def oracle_sample(wl, n_rows: int):
    """Run the oracle (indexer -> top-k -> sparse latent attention, absorbed
    form) on a fixed sample of rows; returns (seconds, rows, threads)."""
    import oracle
    import dsa_inputs as di
    from tests import helpers as H
    rows = di.sample_rows(wl, n_rows)
    t0 = time.perf_counter()
    H.oracle_rows(wl, rows)
    return time.perf_counter() - t0, len(rows), oracle.num_threads()


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def run_reference(args, world, rank):
    """The oracle on the host cores: each step a bounded sample of rows of the
    same workload; throughput in the same unit (tokens/s)."""
    if rank != 0:
        return
    import dsa_inputs as di
    wl = di.workload(args.config)
    for _ in range(args.warmup):
        oracle_sample(wl, max(1, args.cpu_rows // 8))
    secs, rows, threads = 0.0, 0, 1
    for _ in range(args.steps):
        s, n, threads = oracle_sample(wl, args.cpu_rows)
        secs += s
        rows += n
    value = rows / secs
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": CONFIG_NAMES[args.config], "sample_rows_per_step": args.cpu_rows},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"{args.cpu_rows} fixed query rows per step of the {CONFIG_NAMES[args.config]} "
                                       "workload, each row doing its full indexer, top-k and attention work"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    import torch

    import dsa_inputs as di
    import sparse_latent_attention_indexer_gb300 as dsa

    dev = torch.device("cuda", local)
    wl = di.workload(args.config)
    sh = wl.shape
    seqs = dsa.Seqs(wl.cu_q, wl.cu_k, wl.start_pos)
    host = wl.tensors
    t = {k: v.to(dev) for k, v in host.items()}
    ckv, kpe = t["kv_cache"][:, :sh.d_c], t["kv_cache"][:, sh.d_c:]
    M = wl.total_q
    out = torch.empty((M, sh.H, sh.d_v), dtype=t["q_nope"].dtype, device=dev)
    lse = torch.empty((M, sh.H), dtype=torch.float32, device=dev)
    idx = torch.empty((M, sh.k), dtype=torch.int32, device=dev)
    prob = dsa._problem(t["qI"], t["kI"], t["w"], t["q_nope"], t["q_pe"], ckv, kpe, t["W_UK"], t["W_UV"], sh.k,
                        sh.softmax_scale, sh.idx_fp8, out, lse, idx)
    ws = torch.empty(dsa.dsa_forward_workspace_size(prob, seqs), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        dsa.dsa_forward(t["qI"], t["kI"], t["w"], t["q_nope"], t["q_pe"], ckv, kpe, t["W_UK"], t["W_UV"], seqs, sh.k,
                        sh.softmax_scale, idx_fp8=sh.idx_fp8, out=out, lse=lse, idx_out=idx, workspace=ws)

    for _ in range(max(args.warmup, 0)):
        flush.zero_()
        step()
    torch.cuda.synchronize()

    nst = dsa._abi.DSA_STAGE_EVENTS
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nst)] for _ in range(args.steps)]
    clocks = clock_sampler(_gpu_uuid(local))
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    launches = 0
    for i in range(args.steps):
        flush.zero_()
        dsa.set_stage_events(ev[i])
        step()
        launches += dsa.last_launch_count()
    dsa.set_stage_events(None)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    step_ms = [ev[i][0].elapsed_time(ev[i][nst - 1]) for i in range(args.steps)]
    stage_ms = [statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps))
                for j in range(nst - 1)]
    ms = max_over_ranks(statistics.mean(step_ms), world)
    value = wl.total_q * world / (ms / 1e3)

    # roofline of the dominant stage: flops and compulsory HBM bytes per stage; the stage is
    # tensor-bound when its intensity is above the measured ridge point, else HBM-bound
    peaks, peak_src = load_peaks()
    pairs_sel, pairs_causal = wl.selected_pairs(), wl.causal_pairs()
    elt = 4 if sh.dtype == "f32" else 2
    ki_elt = 1 if sh.idx_fp8 else elt
    flops = {
        "indexer+topk": 2.0 * sh.H_I * sh.D_I * pairs_causal,
        "absorb_q": 2.0 * M * sh.H * sh.d_n * sh.d_c,
        "sparse_mla": 2.0 * sh.H * (2 * sh.d_c + sh.d_r) * pairs_sel,
        "absorb_v": 2.0 * M * sh.H * sh.d_c * sh.d_v,
    }
    hbm_bytes = {
        # k^I once, q^I, w, the fp32 scores written and read back, the selection written
        "indexer+topk": wl.total_k * sh.D_I * ki_elt + M * sh.H_I * (sh.D_I * ki_elt + 4) + 8 * pairs_causal
                        + 4 * M * sh.k,
        # W_UK, q_nope in, q~ out (the attention reads q_pe in place)
        "absorb_q": sh.H * sh.d_n * sh.d_c * elt + M * sh.H * sh.d_n * elt + M * sh.H * sh.d_c * elt,
        # each distinct selected latent row once, q~ and q_pe rows in, latent context out
        "sparse_mla": min(pairs_sel, wl.total_k) * (sh.d_c + sh.d_r) * elt + M * sh.H * (sh.d_c + sh.d_r) * elt
                      + M * sh.H * sh.d_c * elt + 4 * M * sh.k,
        "absorb_v": sh.H * sh.d_c * sh.d_v * elt + M * sh.H * (sh.d_c + sh.d_v) * elt,
    }
    names = ["quant", "indexer+topk", "absorb_q", "sparse_mla", "absorb_v"]
    stages = {n: {"ms": stage_ms[j]} for j, n in enumerate(names)}
    for n, f in flops.items():
        ok = stages[n]["ms"] > 0
        stages[n]["tflops"] = f / (stages[n]["ms"] * 1e9) if ok else None
        stages[n]["gbs"] = hbm_bytes[n] / (stages[n]["ms"] * 1e6) if ok else None
    dom = max(["sparse_mla", "indexer+topk", "absorb_q", "absorb_v"], key=lambda n: stages[n]["ms"])
    ridge = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if flops[dom] / hbm_bytes[dom] >= ridge:
        achieved, peak, unit, bound = stages[dom]["tflops"], peaks["bf16_tflops_sustained"], "TFLOP/s", "tensor"
        psrc = f"{peak_src} bf16 sustained (kernel timed inside a step)"
        alg = f"{flops[dom] / 1e9:.1f} GFLOP per launch"
    else:
        achieved, peak, unit, bound = stages[dom]["gbs"], peaks["hbm_gbs"], "GB/s", "hbm"
        psrc = f"{peak_src} HBM copy bandwidth"
        alg = f"{hbm_bytes[dom] / 1e6:.1f} MB per launch"
    roofline = {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak if achieved else None,
                "traffic": ncu_traffic(dom, CONFIG_NAMES[args.config]),
                "peak_source": psrc, "algorithmic": alg}

    e2e = None if args.no_e2e else measure_e2e(args, dsa, torch, dev, wl, host, t, seqs, out, lse, idx, ws)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        secs, rows, threads = oracle_sample(wl, args.cpu_rows)
        cpu = {"value": rows / secs, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{rows} fixed query rows of the same workload (first/last rows, rows around t = k-1, "
                         f"random rows), each doing its full indexer, top-k and attention work, {secs:.1f} s"}
    if rank != 0:
        return
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if sh.dtype == "bf16" else "f32", "data": "synthetic",
            "config": {"workload": CONFIG_NAMES[args.config], "tokens_per_step": M, "keys": wl.total_k,
                       "top_k": sh.k, "l2": "flushed (256 MiB write) before every timed step",
                       "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
            "roofline": roofline, "stages": stages, "gpu_launches": launches, "clocks": clk,
            "e2e": e2e, "cpu_baseline": cpu}
    print(json.dumps(line), flush=True)


def _gpu_uuid(local):
    try:
        import torch
        u = str(torch.cuda.get_device_properties(local).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


def measure_e2e(args, dsa, torch, dev, wl, host, t, seqs, out, lse, idx, ws):
    """The same step through the public API with HOST buffers: pinned host
    inputs copied in, dsa_forward, the output copied back, all inside the
    timed events."""
    sh = wl.shape
    pinned = {k: v.pin_memory() for k, v in host.items()}
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in pinned.values())
    d2h = out_host.numel() * out_host.element_size()
    ckv, kpe = t["kv_cache"][:, :sh.d_c], t["kv_cache"][:, sh.d_c:]
    times = []
    for i in range(args.warmup + args.steps):
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_ev.record()
        for k, v in pinned.items():
            t[k].copy_(v, non_blocking=True)
        dsa.dsa_forward(t["qI"], t["kI"], t["w"], t["q_nope"], t["q_pe"], ckv, kpe, t["W_UK"], t["W_UV"], seqs, sh.k,
                        sh.softmax_scale, idx_fp8=sh.idx_fp8, out=out, lse=lse, idx_out=idx, workspace=ws)
        out_host.copy_(out, non_blocking=True)
        e_ev.record()
        e_ev.synchronize()
        if i >= args.warmup:
            times.append(s_ev.elapsed_time(e_ev))
    ms = statistics.mean(times)
    return {"value": wl.total_q / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h}


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
