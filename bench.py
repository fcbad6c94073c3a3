#!/usr/bin/env python
"""Benchmark of the DSA hot path on GB300, one JSON line on rank 0.

Headline: DSA prefill tokens/s on the largest single-GPU prefill workload,
the chunked prefill with the FP8 indexer (8 sequences x 8192 new queries on
caches of 16K-65K keys, 671B head shapes, top-2048).  The same line carries
``decode`` (64 sequences x 1 query on caches of 8K-64K keys: decode
queries/s) and ``prefill_4k`` (T = S = 4096, bf16), each with its own stage
times, roofline, kernel timings and end-to-end figure.

A step is one dsa_forward call (FP8 quantisation when configured, indexer,
top-k, q~ = q_nope W_UK, sparse latent attention, o_lat W_UV) over the whole
synthetic batch, inputs resident in HBM.  L2 is flushed between timed steps,
outside the timed events: a 256 MiB write, then a 256 MiB read of another
buffer, so the written lines are written back before the step, not inside it.  ``--impl reference`` times the
plain CPU oracle instead (a bounded sample of rows per step).

Under torchrun (N > 1) every rank runs the same workload on its own GPU (the
path shards by query rows / sequences with no exchange): weak scaling, value =
queries of all ranks / the slowest rank's time.
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


UNITS = {0: "tokens/s", 1: "tokens/s", 2: "tokens/s", 3: "queries/s", 4: "tokens/s"}
EXTRA_KEYS = {3: "decode", 1: "prefill_4k", 2: "prefill_32k", 0: "tiny", 4: "chunked_prefill"}
# rows of the oracle's bounded sample: about 10 s on 16 host cores for the cpu_baseline leg, and a
# few seconds per step for the reference arm
CPU_ROWS = {0: 256, 1: 1024, 2: 320, 3: 64, 4: 384}
REF_ROWS = {0: 256, 1: 256, 2: 96, 3: 32, 4: 128}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=4,
                    help="headline workload 0..4 (4 = the chunked prefill with the FP8 indexer)")
    ap.add_argument("--extra", default="3,1",
                    help="comma-separated workloads measured in the same run (default: decode, 4K prefill)")
    ap.add_argument("--cpu-rows", type=int, default=None, help="rows of the oracle's bounded sample")
    ap.add_argument("--ref-rows", type=int, default=None, help="rows per step of the reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-next", action="store_true", help="skip the steps around the path and the FP8 latent cache")
    ap.add_argument("--rows", type=int, default=None,
                    help="keep only the first ROWS query rows of each workload (a small case of the same kernels, "
                         "for profiling); the sequences keep their whole caches")
    ap.add_argument("--seed", type=int, default=None,
                    help="tensor seed of the synthetic workloads (default: each workload's own)")
    ap.add_argument("--last-rows", type=int, default=None,
                    help="keep only the last LAST_ROWS query rows of the longest sequence (the heaviest rows), "
                         "for profiling")
    ap.add_argument("--fused-topk", type=int, choices=[0, 1], default=None,
                    help="1: the fused indexer + top-k kernel; 0: indexer then top-k; default: the library's")
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
        entries = json.load(f).get(stage) or []
    if isinstance(entries, dict):
        entries = [entries]
    entry = next((e for e in entries if e.get("workload") == workload), None)
    if entry is None:
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
    headline workload; throughput in the same unit (tokens/s)."""
    if rank != 0:
        return
    import dsa_inputs as di
    wl = di.workload(args.config, args.seed)
    n_rows = args.ref_rows if args.ref_rows is not None else REF_ROWS[args.config]
    for _ in range(args.warmup):
        oracle_sample(wl, max(1, n_rows // 8))
    secs, rows, threads = 0.0, 0, 1
    for _ in range(args.steps):
        s, n, threads = oracle_sample(wl, n_rows)
        secs += s
        rows += n
    value = rows / secs
    unit = UNITS[args.config]
    line = {"metric": METRIC, "value": value, "unit": unit, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": CONFIG_NAMES[args.config], "sample_rows_per_step": n_rows},
            "cpu_baseline": {"value": value, "unit": unit, "cores": threads, "kind": "oracle",
                             "sample": f"{n_rows} fixed query rows per step of the {CONFIG_NAMES[args.config]} "
                                       "workload, each row doing its full indexer, top-k and attention work"},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def sub_batch(wl, r0, r1):
    """Rows [r0, r1) of a batch as their own batch: (seqs arrays, first sequence,
    last sequence + 1), the sequences keeping their whole key caches."""
    cu_q = wl.cu_q
    bs = [b for b in range(wl.B) if cu_q[b] < r1 and cu_q[b + 1] > r0]
    sub_q, sub_k, sub_p = [0], [0], []
    for b in bs:
        lo, hi = max(cu_q[b], r0), min(cu_q[b + 1], r1)
        sub_q.append(sub_q[-1] + hi - lo)
        sub_k.append(sub_k[-1] + wl.S[b])
        sub_p.append(wl.start_pos[b] + lo - cu_q[b])
    return (sub_q, sub_k, sub_p), bs[0], bs[-1] + 1


def score_chunks(wl):
    """Row ranges of the forward's indexer launches (fp32 scores bounded at 1 GiB per chunk)."""
    ld = (max(max(wl.S), 1) + 3) // 4 * 4
    per = max(1, min(wl.total_q, (1 << 30) // (ld * 4)))
    return [(r0, min(wl.total_q, r0 + per)) for r0 in range(0, wl.total_q, per)]


def indexer_pairs_computed(wl, skip_dense=True):
    """(query, key) pairs the tensor-core indexer multiplies: for every group of
    4 consecutive queries of a sequence, every 128-key block up to the last
    query's position, for each query of the group; the forward skips groups
    whose queries all see at most k keys."""
    k = wl.shape.k
    total = 0
    for b in range(wl.B):
        T = wl.T[b]
        for t0 in range(0, T, 4):
            ntok = min(4, T - t0)
            last = wl.start_pos[b] + t0 + ntok - 1
            if skip_dense and last < k:
                continue
            total += (last // 128 + 1) * 128 * ntok
    return total


def stage_work(wl):
    """Algorithmic flops and compulsory HBM bytes of each stage of one step."""
    sh = wl.shape
    M = wl.total_q
    pairs_sel, pairs_causal = wl.selected_pairs(), wl.causal_pairs()
    elt = 4 if sh.dtype == "f32" else 2
    ki_elt = 1 if sh.idx_fp8 else elt
    # rows that need scores (the others select every causal key without them)
    scored = sum(1 for b in range(wl.B) for p in wl.row_positions(b) if p + 1 > sh.k)
    scored_pairs = sum(p + 1 for b in range(wl.B) for p in wl.row_positions(b) if p + 1 > sh.k)
    flops = {
        "indexer+topk": 2.0 * sh.H_I * sh.D_I * pairs_causal,
        "absorb_q": 2.0 * M * sh.H * sh.d_n * sh.d_c,
        "sparse_mla": 2.0 * sh.H * (2 * sh.d_c + sh.d_r) * pairs_sel,
        "absorb_v": 2.0 * M * sh.H * sh.d_c * sh.d_v,
    }
    hbm = {
        # k^I once, q^I and w of the scored rows, their fp32 scores written and read back, the selection
        "indexer+topk": wl.total_k * sh.D_I * ki_elt + scored * sh.H_I * (sh.D_I * ki_elt + 4) + 8 * scored_pairs
                        + 4 * M * sh.k,
        # W_UK, q_nope in, q~ out (the attention reads q_pe in place)
        "absorb_q": sh.H * sh.d_n * sh.d_c * elt + M * sh.H * sh.d_n * elt + M * sh.H * sh.d_c * elt,
        # each distinct selected latent row once, q~ and q_pe rows in, latent context out, the selection
        "sparse_mla": min(pairs_sel, wl.total_k) * (sh.d_c + sh.d_r) * elt + M * sh.H * (sh.d_c + sh.d_r) * elt
                      + M * sh.H * sh.d_c * elt + 4 * M * sh.k,
        "absorb_v": sh.H * sh.d_c * sh.d_v * elt + M * sh.H * (sh.d_c + sh.d_v) * elt,
    }
    return flops, hbm


def roofline_of(stage, ms, flops, hbm, peaks, peak_src, wl_name, fp8=False):
    """Tensor-bound when the stage's intensity is above the ridge point of the
    measured peaks, else HBM-bound.  The burst peak applies: every timed region
    here lasts well under a second."""
    tensor_peak = peaks["bf16_tflops"] * (2.0 if fp8 else 1.0)
    ridge = tensor_peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if flops / hbm >= ridge:
        achieved, peak, unit, bound = flops / (ms * 1e9), tensor_peak, "TFLOP/s", "tensor"
        psrc = (f"{peak_src} bf16 burst" + (" x 2 (nominal FP8 : bf16 ratio)" if fp8 else ""))
        alg = f"{flops / 1e9:.1f} GFLOP per launch"
    else:
        achieved, peak, unit, bound = hbm / (ms * 1e6), peaks["hbm_gbs"], "GB/s", "hbm"
        psrc = f"{peak_src} HBM copy bandwidth"
        alg = f"{hbm / 1e6:.1f} MB per launch"
    return {"kernel": stage, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": ncu_traffic(stage, wl_name), "peak_source": psrc,
            "algorithmic": alg}


def first_rows(wl, n):
    """The workload cut to its first n query rows: the sequences that hold them (the last one with
    fewer queries), each keeping its whole key cache."""
    if n is None or n >= wl.total_q:
        return wl
    import dsa_inputs as di
    T, S, P, cut = [], [], [], 0
    for b in range(wl.B):
        if cut >= n:
            break
        t = min(wl.T[b], n - cut)
        T.append(t)
        S.append(wl.S[b])
        P.append(wl.start_pos[b])
        cut += t
    nb, nk = len(T), wl.cu_k[len(T)]
    q_rows = [r for b in range(nb) for r in range(wl.cu_q[b], wl.cu_q[b] + T[b])]
    ten = {}
    for k, v in wl.tensors.items():
        if k in ("qI", "w", "q_nope", "q_pe"):
            ten[k] = v[q_rows]
        elif k in ("kI", "kv_cache"):
            ten[k] = v[:nk]
        else:
            ten[k] = v
    return di.Workload(wl.name + f"-first{n}", wl.shape, wl.seed, T, S, P, ten)


def last_rows(wl, n):
    """The workload cut to the last n query rows of its longest sequence (the longest causal
    prefixes: the heaviest rows), with that sequence's whole key cache."""
    if n is None:
        return wl
    import dsa_inputs as di
    b = max(range(wl.B), key=lambda i: wl.S[i])
    t = min(n, wl.T[b])
    q_rows = list(range(wl.cu_q[b + 1] - t, wl.cu_q[b + 1]))
    ten = {}
    for k, v in wl.tensors.items():
        if k in ("qI", "w", "q_nope", "q_pe"):
            ten[k] = v[q_rows]
        elif k in ("kI", "kv_cache"):
            ten[k] = v[wl.cu_k[b]:wl.cu_k[b + 1]]
        else:
            ten[k] = v
    return di.Workload(wl.name + f"-last{t}", wl.shape, wl.seed, [t], [wl.S[b]], [wl.start_pos[b] + wl.T[b] - t], ten)


class L2Flush:
    """Evicts L2 (129 MB) before a timed step: a 256 MiB write, then a 256 MiB
    read of a second buffer.  The read evicts the write's dirty lines, so their
    write-back happens here and not inside the step that follows."""

    def __init__(self, torch, dev):
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(64 << 20, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


L2_NOTE = "flushed before every timed step (a 256 MiB write, then a 256 MiB read of another buffer)"


def measure_workload(cfg, args, world, rank, local, with_cpu):
    """Times whole dsa_forward steps of workload `cfg`, then its indexer and
    top-k kernels on their own, then the end-to-end step from host buffers."""
    import torch

    import dsa_inputs as di
    import sparse_latent_attention_indexer_gb300 as dsa

    dev = torch.device("cuda", local)
    wl = last_rows(first_rows(di.workload(cfg, args.seed), args.rows), args.last_rows)
    sh = wl.shape
    name = CONFIG_NAMES[cfg] + (f" (first {args.rows} rows)" if args.rows else "")
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
    flush = L2Flush(torch, dev)

    def step():
        dsa.dsa_forward(t["qI"], t["kI"], t["w"], t["q_nope"], t["q_pe"], ckv, kpe, t["W_UK"], t["W_UV"], seqs, sh.k,
                        sh.softmax_scale, idx_fp8=sh.idx_fp8, out=out, lse=lse, idx_out=idx, workspace=ws)

    for _ in range(max(args.warmup, 0)):
        flush()
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
        flush()
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
    value = M * world / (ms / 1e3)

    peaks, peak_src = load_peaks()
    flops, hbm = stage_work(wl)
    names = ["quant", "indexer+topk", "absorb_q", "sparse_mla", "absorb_v"]
    stages = {n: {"ms": stage_ms[j]} for j, n in enumerate(names)}
    for n in flops:
        ok = stages[n]["ms"] > 0
        stages[n]["tflops"] = flops[n] / (stages[n]["ms"] * 1e9) if ok else None
        stages[n]["gbs"] = hbm[n] / (stages[n]["ms"] * 1e6) if ok else None
    dom = max(["sparse_mla", "indexer+topk", "absorb_q", "absorb_v"], key=lambda n: stages[n]["ms"])
    roofline = roofline_of(dom, stages[dom]["ms"], flops[dom], hbm[dom], peaks, peak_src, name,
                           fp8=(dom == "indexer+topk" and sh.idx_fp8))
    kernels = measure_indexer_topk(args, dsa, torch, wl, t, flush, peaks, peak_src)

    e2e = None if args.no_e2e else measure_e2e(args, dsa, torch, wl, host, t, seqs, out, lse, idx, ws, UNITS[cfg])
    cpu = None
    if with_cpu and rank == 0 and world == 1 and not args.no_cpu_baseline:
        n_rows = args.cpu_rows if args.cpu_rows is not None else CPU_ROWS[cfg]
        secs, rows, threads = oracle_sample(wl, n_rows)
        cpu = {"value": rows / secs, "unit": UNITS[cfg], "cores": threads, "kind": "oracle",
               "sample": f"{rows} fixed query rows of the same workload (first/last rows, rows around t = k-1, "
                         f"random rows), each doing its full indexer, top-k and attention work, {secs:.1f} s"}
    res = {"value": value, "unit": UNITS[cfg], "ms_per_step": ms,
           "dtype": "bf16" if sh.dtype == "bf16" else "f32",
           "config": {"workload": name, "queries_per_step": M, "keys": wl.total_k, "top_k": sh.k,
                      "indexer": "fp8 e4m3 + ue8m0 block scales" if sh.idx_fp8 else sh.dtype,
                      "l2": L2_NOTE,
                      "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                      **({"seed": args.seed} if args.seed is not None else {})},
           "roofline": roofline, "stages": stages, "kernels": kernels, "gpu_launches": launches, "clocks": clk,
           "e2e": e2e, "cpu_baseline": cpu}
    del t, out, lse, idx, ws, flush
    torch.cuda.empty_cache()
    return res


def measure_indexer_topk(args, dsa, torch, wl, t, flush, peaks, peak_src):
    """The indexer and the top-k kernels timed on their own (CUDA events around
    each launch, on the current stream), over the same row chunks the forward
    launches them on; the indexer's rate counts the pairs it multiplies."""
    sh = wl.shape
    if all(p + 1 <= sh.k for b in range(wl.B) for p in wl.row_positions(b)):
        return None  # every row selects all its causal keys: neither kernel runs
    q, k = t["qI"], t["kI"]
    qs = ks = None
    if sh.idx_fp8:
        q, qs = dsa.dsa_quant_e4m3_ue8m0(t["qI"])
        k, ks = dsa.dsa_quant_e4m3_ue8m0(t["kI"])
    chunks = score_chunks(wl)
    ld = (max(max(wl.S), 1) + 3) // 4 * 4
    per = chunks[0][1] - chunks[0][0]
    scores = torch.empty((per, ld), dtype=torch.float32, device=q.device)
    sel = torch.empty((per, sh.k), dtype=torch.int32, device=q.device)
    cu_k = wl.cu_k
    reps = max(1, min(3, args.steps))
    t_idx = t_topk = 0.0
    for rep in range(reps + 1):
        evs = []
        for r0, r1 in chunks:
            (sq, sk, sp), b0, b1 = sub_batch(wl, r0, r1)
            s = dsa.Seqs(sq, sk, sp)
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            flush()
            e[0].record()
            dsa.dsa_indexer_scores(q[r0:r1], k[cu_k[b0]:cu_k[b1]], t["w"][r0:r1], s,
                                   q_scale=None if qs is None else qs[r0 * sh.H_I:r1 * sh.H_I],
                                   k_scale=None if ks is None else ks[cu_k[b0]:cu_k[b1]], scores=scores[:r1 - r0])
            e[1].record()
            dsa.dsa_topk_select(scores[:r1 - r0], s, sh.k, idx=sel[:r1 - r0])
            e[2].record()
            evs.append(e)
        torch.cuda.synchronize()
        if rep == 0:
            continue  # warm-up
        t_idx += sum(e[0].elapsed_time(e[1]) for e in evs)
        t_topk += sum(e[1].elapsed_time(e[2]) for e in evs)
    t_idx /= reps
    t_topk /= reps
    pairs = indexer_pairs_computed(wl, skip_dense=False)
    flops = 2.0 * sh.H_I * sh.D_I * pairs
    fp8 = sh.idx_fp8
    tensor_peak = peaks["bf16_tflops"] * (2.0 if fp8 else 1.0)
    causal_scores = sum(p + 1 for b in range(wl.B) for p in wl.row_positions(b))
    decode = max(wl.T) == 1
    res = {"indexer": {"ms": t_idx, "pairs_computed": pairs, "tflops_computed": flops / (t_idx * 1e9),
                       "peak_tflops": tensor_peak,
                       "peak_source": f"{peak_src} bf16 burst" + (" x 2 (nominal FP8 : bf16 ratio)" if fp8 else ""),
                       "frac_of_tensor_peak": flops / (t_idx * 1e9) / tensor_peak},
           "topk": {"ms": t_topk, "score_bytes_read": 4 * causal_scores,
                    "gbs": 4 * causal_scores / (t_topk * 1e6)}}
    if decode:  # the decode indexer streams k^I once: HBM-bound
        kbytes = wl.total_k * sh.D_I * (1 if fp8 else 2)
        res["indexer"]["hbm_bytes"] = kbytes
        res["indexer"]["gbs"] = kbytes / (t_idx * 1e6)
        res["indexer"]["frac_of_hbm"] = kbytes / (t_idx * 1e6) / peaks["hbm_gbs"]
    res["note"] = ("timed outside the step, launch by launch over the forward's row chunks; dsa_indexer_scores "
                   "also writes -inf for the masked keys past the causal blocks, which the forward skips")
    return res


def run_ours(args, world, rank, local):
    if args.fused_topk is not None:
        import sparse_latent_attention_indexer_gb300 as dsa
        dsa.dsa_set_fused_topk(bool(args.fused_topk))
    extra = [int(x) for x in args.extra.split(",") if x.strip() != ""] if args.extra else []
    extra = [c for c in extra if c != args.config]
    main = measure_workload(args.config, args, world, rank, local, with_cpu=True)
    others = {}
    for c in extra:
        others[EXTRA_KEYS.get(c, f"config{c}")] = measure_workload(c, args, world, rank, local, with_cpu=False)
    nxt = None if args.no_next else measure_next(args, local)
    if rank != 0:
        return
    line = {"metric": METRIC, "value": main["value"], "unit": main["unit"], "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": main["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": main["dtype"], "data": "synthetic", "config": main["config"],
            "roofline": main["roofline"], "stages": main["stages"], "kernels": main["kernels"],
            "gpu_launches": main["gpu_launches"], "clocks": main["clocks"], "e2e": main["e2e"],
            "cpu_baseline": main["cpu_baseline"]}
    for key, r in others.items():
        r.pop("cpu_baseline", None)
        line[key] = r
    if nxt is not None:
        line["next"] = nxt
    print(json.dumps(line), flush=True)


def _time_ms(torch, fn, flush, steps, warmup):
    """Mean CUDA-event time of fn() on the current stream, L2 flushed before each call."""
    for _ in range(max(warmup, 1)):
        flush()
        fn()
    times = []
    for _ in range(steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    return statistics.mean(times)


def measure_next(args, local):
    """The steps on either side of the path and the FP8 latent cache, each timed
    on its own with CUDA events:
      * kv_prologue: the key side of 4096 new tokens (x [4096, 7168] bf16 times
        the stacked [768, 7168] weight, kv_norm, rotary k_pe, k_norm, the cache
        append with the FP8 indexer key);
      * output_proj: wo on the 4K prefill's attention output (4096 x 16384 ->
        7168);
      * prefill_4k_with_wo: the 4K prefill step with W_UV and wo chunk by chunk;
      * decode_fp8_latent: the decode workload with its latent cache in e4m3 +
        ue8m0 scales (656 instead of 1152 bytes per key)."""
    import math

    import torch

    import dsa_inputs as di
    import sparse_latent_attention_indexer_gb300 as dsa

    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    flush = L2Flush(torch, dev)
    g = torch.Generator().manual_seed(5)
    res = {}
    T, dim = 4096, 7168
    x = torch.randn(T, dim, generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn(768, dim, generator=g) / math.sqrt(dim)).to(torch.bfloat16).to(dev)
    ones512, ones128, zeros128 = (torch.ones(512, device=dev), torch.ones(128, device=dev),
                                  torch.zeros(128, device=dev))
    ang = torch.arange(T, dtype=torch.float64)[:, None] * (10000.0 ** (-torch.arange(32, dtype=torch.float64) / 32))
    cos_t, sin_t = torch.cos(ang).float().to(dev), torch.sin(ang).float().to(dev)
    seqs = dsa.Seqs([0, T], [0, T], [0])
    kv_cache = torch.empty(T, 576, dtype=torch.bfloat16, device=dev)
    k_codes = torch.empty(T, 128, dtype=torch.uint8, device=dev)
    k_scale = torch.empty(T, device=dev)
    wts = torch.empty(T, 64, device=dev)
    ws = torch.empty(dsa._abi.load().dsa_kv_prologue_workspace_size(dim, 512, 64, 128, 64, seqs.ref()),
                     dtype=torch.uint8, device=dev)
    ms = _time_ms(torch, lambda: dsa.dsa_kv_prologue(x, W, ones512, ones128, zeros128, cos_t, sin_t, seqs, kv_cache,
                                                     k_codes, w=wts, k_scale=k_scale, workspace=ws),
                  flush, args.steps, args.warmup)
    gemm_flop = 2.0 * T * dim * 768
    res["kv_prologue"] = {"tokens": T, "ms": ms, "tokens_per_s": T / (ms / 1e3),
                          "gemm_tflops": gemm_flop / (ms * 1e9),
                          "frac_of_tensor_peak": gemm_flop / (ms * 1e9) / peaks["bf16_tflops"],
                          "peak_source": f"{peak_src} bf16 burst",
                          "note": "tensor-core GEMM x . W_proj^T (45.1 GFLOP) plus the per-token norms, rotation "
                                  "and FP8 append, timed together"}
    del x, W, kv_cache, k_codes, k_scale, wts, ws
    out = torch.randn(T, 128 * 128, generator=g).to(torch.bfloat16).to(dev)
    wo = (torch.randn(dim, 128 * 128, generator=g) / 128.0).to(torch.bfloat16).to(dev)
    y = torch.empty(T, dim, dtype=torch.bfloat16, device=dev)
    ms = _time_ms(torch, lambda: dsa.dsa_output_proj(out, wo, y=y), flush, args.steps, args.warmup)
    flop = 2.0 * T * 16384 * dim
    res["output_proj"] = {"rows": T, "ms": ms, "tflops": flop / (ms * 1e9),
                          "frac_of_tensor_peak": flop / (ms * 1e9) / peaks["bf16_tflops"],
                          "peak_source": f"{peak_src} bf16 burst", "algorithmic": f"{flop / 1e9:.1f} GFLOP"}
    del out, y

    wl = di.workload(1)
    sh = wl.shape
    t = {k: v.to(dev) for k, v in wl.tensors.items()}
    ckv, kpe = t["kv_cache"][:, :sh.d_c], t["kv_cache"][:, sh.d_c:]
    s1 = dsa.Seqs(wl.cu_q, wl.cu_k, wl.start_pos)
    outs = {}

    def fwd(with_wo):
        outs["r"] = dsa.dsa_forward(t["qI"], t["kI"], t["w"], t["q_nope"], t["q_pe"], ckv, kpe, t["W_UK"], t["W_UV"],
                                    s1, sh.k, sh.softmax_scale, wo=wo if with_wo else None, want_out=not with_wo)
    ms0 = _time_ms(torch, lambda: fwd(False), flush, args.steps, args.warmup)
    ms1 = _time_ms(torch, lambda: fwd(True), flush, args.steps, args.warmup)
    res["prefill_4k_with_wo"] = {"ms": ms1, "tokens_per_s": wl.total_q / (ms1 / 1e3), "ms_without_wo": ms0,
                                 "wo_added_ms": ms1 - ms0,
                                 "note": "dsa_forward with the output projection: W_UV and wo in chunks of 2048 "
                                         "rows, the attention output of a chunk read back from L2 (not kept)"}
    del t, outs, wo
    torch.cuda.empty_cache()

    wl = di.workload(3)
    sh = wl.shape
    t = {k: v.to(dev) for k, v in wl.tensors.items()}
    ckv, kpe = t["kv_cache"][:, :sh.d_c], t["kv_cache"][:, sh.d_c:]
    codes, scales = dsa.dsa_quant_e4m3_ue8m0(ckv.contiguous())
    scales = scales.view(-1, sh.d_c // 128)
    s3 = dsa.Seqs(wl.cu_q, wl.cu_k, wl.start_pos)

    def dec(fp8):
        dsa.dsa_forward(t["qI"], t["kI"], t["w"], t["q_nope"], t["q_pe"], codes if fp8 else ckv, kpe, t["W_UK"],
                        t["W_UV"], s3, sh.k, sh.softmax_scale, kv_scale=scales if fp8 else None)
    ms_b = _time_ms(torch, lambda: dec(False), flush, args.steps, args.warmup)
    ms_8 = _time_ms(torch, lambda: dec(True), flush, args.steps, args.warmup)
    res["decode_fp8_latent"] = {"ms": ms_8, "queries_per_s": wl.total_q / (ms_8 / 1e3), "ms_bf16_latent": ms_b,
                                "latent_bytes_per_key": {"fp8": sh.d_c + 4 * (sh.d_c // 128) + 2 * sh.d_r,
                                                         "bf16": 2 * (sh.d_c + sh.d_r)}}
    del t, codes, scales
    torch.cuda.empty_cache()
    return res


def _gpu_uuid(local):
    try:
        import torch
        u = str(torch.cuda.get_device_properties(local).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


def measure_e2e(args, dsa, torch, wl, host, t, seqs, out, lse, idx, ws, unit):
    """The same step through the C-ABI call with HOST buffers (dsa_forward_host):
    every step copies that step's inputs from pinned host memory -- the new
    queries' tensors and the key-cache rows they append (each sequence's cache
    rows start_pos .. S-1; the rows before start_pos are the cache the earlier
    steps left resident) -- runs the forward and copies the output back, all
    inside the timed events.  Two pipeline slots, each with its own stream and
    device buffers, take alternate steps: the forwards run one after the other
    (each call waits for the previous step's forward through the call's
    compute events) while one step's copies overlap the other slot's kernels
    (the copy engines and the SMs work at the same time); the per-step time of
    one slot alone (copies and kernels back to back) is reported beside it."""
    sh = wl.shape
    cu_k = wl.cu_k
    new_rows = torch.cat([torch.arange(cu_k[b] + wl.start_pos[b], cu_k[b + 1]) for b in range(wl.B)])
    inputs = {"q_idx": host["qI"].pin_memory(), "w": host["w"].pin_memory(), "q_nope": host["q_nope"].pin_memory(),
              "q_pe": host["q_pe"].pin_memory(), "kv_new": host["kv_cache"][new_rows].contiguous().pin_memory(),
              "k_idx_new": host["kI"][new_rows].contiguous().pin_memory()}
    h2d = sum(v.numel() * v.element_size() for v in inputs.values())
    d2h = out.numel() * out.element_size()
    d_c = sh.d_c
    slots = []
    for si in range(2):
        if si == 0:
            dev, o, l, ix, w = t, out, lse, idx, ws
        else:
            dev = {k: t[k].clone() for k in ("qI", "kI", "w", "q_nope", "q_pe", "kv_cache")}
            dev["W_UK"], dev["W_UV"] = t["W_UK"], t["W_UV"]
            o, l, ix, w = torch.empty_like(out), torch.empty_like(lse), torch.empty_like(idx), torch.empty_like(ws)
        slots.append({"dev": dev, "out": o, "lse": l, "idx": ix, "ws": w, "stream": torch.cuda.Stream(),
                      "host": dict(inputs, out=torch.empty(out.shape, dtype=out.dtype).pin_memory())})

    done = [torch.cuda.Event(), torch.cuda.Event()]  # the forward of the slot's last step is enqueued
    copied = [torch.cuda.Event(), torch.cuda.Event()]  # the input copies of the slot's last step are enqueued

    def step(i, n_slots):
        sl = slots[i % n_slots]
        d = sl["dev"]
        # with two slots the forwards run one after the other (each waits for the previous step's),
        # while the copies of one step overlap the kernels of the other; the input copies also run
        # one after the other, so the first forward waits for one step's inputs, not two steps'
        chain = {} if n_slots == 1 else {"compute_done": done[i % 2], "compute_after": done[(i + 1) % 2] if i else None,
                                         "copy_done": copied[i % 2], "copy_after": copied[(i + 1) % 2] if i else None}
        dsa.dsa_forward_host(sl["host"], d["qI"], d["kI"], d["w"], d["q_nope"], d["q_pe"], d["kv_cache"][:, :d_c],
                             d["kv_cache"][:, d_c:], d["W_UK"], d["W_UV"], seqs, sh.k, sh.softmax_scale,
                             idx_fp8=sh.idx_fp8, out=sl["out"], lse=sl["lse"], idx_out=sl["idx"], workspace=sl["ws"],
                             stream=sl["stream"], **chain)

    def run(n_slots, steps, warmup):
        cur = torch.cuda.current_stream()
        for i in range(warmup):
            step(i, n_slots)
        torch.cuda.synchronize()
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_ev.record(cur)
        for sl in slots[:n_slots]:
            sl["stream"].wait_event(s_ev)
        for i in range(warmup, warmup + steps):
            step(i, n_slots)
        for sl in slots[:n_slots]:
            cur.wait_stream(sl["stream"])
        e_ev.record(cur)
        e_ev.synchronize()
        return s_ev.elapsed_time(e_ev) / steps

    steps = max(args.steps, 2)
    serial = run(1, steps, args.warmup)
    ms = run(2, steps, args.warmup)
    return {"value": wl.total_q / (ms / 1e3), "unit": unit, "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "serial_ms_per_step": serial, "serial_value": wl.total_q / (serial / 1e3),
            "call": "dsa_forward_host (pinned host buffers), two pipeline slots on their own streams, forwards and "
                    "input copies chained",
            "inputs": "the step's queries (q^I, w, q_nope, q_pe) and the cache rows they append "
                      "(latent + k_pe, k^I); the earlier cache rows stay resident"}


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
